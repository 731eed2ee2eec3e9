"""Seeded synthetic inputs for the ORPO head (shared by tests, the oracle and the bench).

This module holds none of the head's or the loss's arithmetic: it only draws
inputs.  All values are drawn on the CPU from numpy PCG64 streams in float32,
rounded to nearest-even bf16, and returned as raw bf16 bit patterns (uint16) so
that the CUDA path and the float64 oracle see exactly the same numbers.

Every array has its own stream keyed by (seed, array key, chunk index), so the
result does not depend on how many threads draw it.  Keys: lengths 0, mask 1,
targets 2, h 3, W 4, the random half of mixed h 5.

Workloads (sizes as stated for the five head shapes this library is measured
on; the pages' real data, chunk-segmenter / UltraFeedback pairs on Gemma e4b
and MiniCPM5, is not available, and these synthetic draws stand in for it):

  tiny     2 pairs x 64 rows (first 8 rows of each sequence are prompt rows,
           mask 0) -> M 256; d 256, V 4096; h ~ N(0,1); W ~ N(0, 4/d);
           uniform targets; no softcap; lambda 0.1.
  small    8 pairs, 16 response lengths ~ U{64..256} -> M drawn (~2.5k);
           d 2048, V 32000; same distributions; no softcap; lambda 0.1.
  e4b      16 pairs x 2 x 256 -> M 8192; d 2560, V 262144; softcap 30;
           peaked h_t = 0.5 N(0,1) + 3 W[y_t] / |W[y_t]|; lambda 0.1.
  largev   8 pairs x 2 x 1024 -> M 16384; d 4096, V 128256; h ~ N(0,1);
           targets Zipf(1.1) over ids (P(k) ~ (k+1)^-1.1); no softcap; lambda 0.2.
  ragged   64 pairs, 128 lengths ~ U{16..1024} packed, then pad rows
           (mask 0, seq_id -1) up to a multiple of 128; d 3840, V 262144;
           softcap 30; rows t < M/2 peaked as in e4b, the rest N(0,1); lambda 0.1.
  e4b_sharp  e4b's shapes and targets with a sharper peak, h_t = 0.5 N(0,1) +
           12 W[y_t] / |W[y_t]|: the target logit is about 24 (19.9 after the
           softcap) against N(0, 1.2) elsewhere, so p(target) ~ 0.999.  It
           stands in for the pages' real teacher-forced data, on which the
           backward skips were measured; e4b's own peak (3) leaves the softmax
           nearly flat at V = 262144 (p(target) ~ 1e-3).
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 22

K_LEN, K_MASK, K_TGT, K_H, K_W, K_H2 = 0, 1, 2, 3, 4, 5


@dataclass
class Workload:
    name: str
    h: np.ndarray          # uint16 bf16 bits [M, d]
    W: np.ndarray          # uint16 bf16 bits [V, d]
    targets: np.ndarray    # int32 [M]
    mask: np.ndarray       # uint8 [M]
    seq_id: np.ndarray     # int32 [M]
    n_pairs: int
    softcap: float
    lam: float
    meta: dict = field(default_factory=dict)

    @property
    def M(self):
        return self.h.shape[0]

    @property
    def d(self):
        return self.h.shape[1]

    @property
    def V(self):
        return self.W.shape[0]


def _rng(seed: int, key: int, chunk: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence(seed, spawn_key=(key, chunk))
    return np.random.Generator(np.random.PCG64(ss))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def normal_bf16(seed: int, key: int, shape, std: float) -> np.ndarray:
    """bf16 bits of std * N(0,1), drawn chunk by chunk on a thread pool."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)

    def work(c):
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        x = _rng(seed, key, c).standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = round_bf16(x)

    nchunks = (n + CHUNK - 1) // CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=min(_threads(), nchunks)) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


def _peaked_h(seed: int, W_bits: np.ndarray, targets: np.ndarray, rows: np.ndarray, d: int,
              key: int = K_H, peak: float = 3.0) -> np.ndarray:
    """bf16 bits of 0.5 N(0,1) + peak W[y] / |W[y]| for the given rows (input recipe only)."""
    noise = bf16_to_f32(normal_bf16(seed, key, (len(rows), d), 1.0)).astype(np.float64)
    Wy = bf16_to_f32(W_bits[targets[rows]]).astype(np.float64)
    nrm = np.linalg.norm(Wy, axis=1, keepdims=True)
    nrm[nrm == 0] = 1.0
    return round_bf16((0.5 * noise + peak * Wy / nrm).astype(np.float32))


def _layout(lengths: np.ndarray, prompt_rows: int = 0, pad_to: int = 1):
    """Packed rows for sequences of the given lengths; seq s = lengths[s] rows."""
    M0 = int(lengths.sum())
    M = ((M0 + pad_to - 1) // pad_to) * pad_to
    seq_id = np.full(M, -1, dtype=np.int32)
    mask = np.zeros(M, dtype=np.uint8)
    r = 0
    for s, L in enumerate(lengths):
        seq_id[r:r + L] = s
        mask[r + prompt_rows:r + L] = 1
        r += L
    return seq_id, mask


def _uniform_targets(seed, M, V):
    return _rng(seed, K_TGT).integers(0, V, size=M, dtype=np.int64).astype(np.int32)


def _zipf_targets(seed, M, V, a=1.1):
    w = np.arange(1, V + 1, dtype=np.float64) ** (-a)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = _rng(seed, K_TGT).random(M)
    return np.minimum(np.searchsorted(cdf, u, side="right"), V - 1).astype(np.int32)


NAMES = ("tiny", "small", "e4b", "largev", "ragged", "e4b_sharp")


def make(name: str, seed: int = 0, M: int | None = None, d: int | None = None,
         V: int | None = None) -> Workload:
    """Build one workload.  M / d / V overrides shrink a recipe for tests (the
    structure is kept: pair count scales with M where the recipe has fixed lengths)."""
    if name == "tiny":
        d = d or 256
        V = V or 4096
        P = 2
        L = 64 if M is None else max(9, M // (2 * P))
        lengths = np.full(2 * P, L)
        seq_id, mask = _layout(lengths, prompt_rows=8)
        Mx = len(seq_id)
        tg = _uniform_targets(seed, Mx, V)
        W = normal_bf16(seed, K_W, (V, d), (4.0 / d) ** 0.5)
        h = normal_bf16(seed, K_H, (Mx, d), 1.0)
        return Workload(name, h, W, tg, mask, seq_id, P, 0.0, 0.1)
    if name == "small":
        d = d or 2048
        V = V or 32000
        P = 8
        lo, hi = (64, 256) if M is None else (max(1, M // 32), max(2, M // 8))
        lengths = _rng(seed, K_LEN).integers(lo, hi + 1, size=2 * P)
        seq_id, mask = _layout(lengths)
        Mx = len(seq_id)
        tg = _uniform_targets(seed, Mx, V)
        W = normal_bf16(seed, K_W, (V, d), (4.0 / d) ** 0.5)
        h = normal_bf16(seed, K_H, (Mx, d), 1.0)
        return Workload(name, h, W, tg, mask, seq_id, P, 0.0, 0.1)
    if name in ("e4b", "e4b_sharp"):
        d = d or 2560
        V = V or 262144
        L = 256
        P = 16 if M is None else max(1, M // (2 * L))
        lengths = np.full(2 * P, L)
        seq_id, mask = _layout(lengths)
        Mx = len(seq_id)
        tg = _uniform_targets(seed, Mx, V)
        W = normal_bf16(seed, K_W, (V, d), (4.0 / d) ** 0.5)
        h = _peaked_h(seed, W, tg, np.arange(Mx), d, peak=3.0 if name == "e4b" else 12.0)
        return Workload(name, h, W, tg, mask, seq_id, P, 30.0, 0.1)
    if name == "largev":
        d = d or 4096
        V = V or 128256
        L = 1024
        P = 8 if M is None else max(1, M // (2 * L))
        lengths = np.full(2 * P, L)
        seq_id, mask = _layout(lengths)
        Mx = len(seq_id)
        tg = _zipf_targets(seed, Mx, V)
        W = normal_bf16(seed, K_W, (V, d), (4.0 / d) ** 0.5)
        h = normal_bf16(seed, K_H, (Mx, d), 1.0)
        return Workload(name, h, W, tg, mask, seq_id, P, 0.0, 0.2)
    if name == "ragged":
        d = d or 3840
        V = V or 262144
        P = 64 if M is None else max(1, M // 1040)
        lengths = _rng(seed, K_LEN).integers(16, 1024 + 1, size=2 * P)
        seq_id, mask = _layout(lengths, pad_to=128)
        Mx = len(seq_id)
        tg = _uniform_targets(seed, Mx, V)
        W = normal_bf16(seed, K_W, (V, d), (4.0 / d) ** 0.5)
        half = Mx // 2
        h = np.empty((Mx, d), dtype=np.uint16)
        h[:half] = _peaked_h(seed, W, tg, np.arange(half), d)
        h[half:] = normal_bf16(seed, K_H2, (Mx - half, d), 1.0)
        return Workload(name, h, W, tg, mask, seq_id, P, 30.0, 0.1)
    raise KeyError(name)


def synthetic_logp(seed: int, seq_id: np.ndarray, mask: np.ndarray, scale: float = 2.0,
                   offset: float = -3.0) -> np.ndarray:
    """Plausible per-token log-probs (strictly negative) for testing the loss on its own."""
    r = _rng(seed, 9)
    x = offset - scale * np.abs(r.standard_normal(len(seq_id)))
    return np.minimum(x, -1e-3).astype(np.float32)


def quantize_affine(W_bits: np.ndarray, bits: int, group: int):
    """Affine group quantisation of bf16 weights (input preparation for the quantised head).

    Per row and group of `group` consecutive columns: bias = min, scale = (max - min) / (2^bits - 1),
    both rounded to bf16; q = clip(round((w - bias) / scale), 0, 2^bits - 1).  Returns
    (wq uint8 [V, d * bits / 8], scales bf16 bits [V, d / group], biases bf16 bits [V, d / group]);
    4-bit values are packed two per byte, even column in the low nibble.
    """
    W = bf16_to_f32(W_bits).astype(np.float64)
    V, d = W.shape
    g = W.reshape(V, d // group, group)
    lo, hi = g.min(axis=2), g.max(axis=2)
    levels = (1 << bits) - 1
    scale = np.where(hi > lo, (hi - lo) / levels, 1.0)
    s_bits = round_bf16(scale.astype(np.float32))
    b_bits = round_bf16(lo.astype(np.float32))
    s = bf16_to_f32(s_bits).astype(np.float64)[:, :, None]
    b = bf16_to_f32(b_bits).astype(np.float64)[:, :, None]
    q = np.clip(np.rint((g - b) / s), 0, levels).astype(np.uint8).reshape(V, d)
    if bits == 4:
        wq = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    else:
        wq = q
    return np.ascontiguousarray(wq), s_bits, b_bits
