"""orpo_loss parity against the float64 oracle on synthetic per-token logp."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import LOSS_RTOL, dev, gpu_loss

pytestmark = pytest.mark.gpu


def run(logp, seq, mask, P, lam):
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).astype(dt)).to(dev())
    return gpu_loss(t(logp, np.float32), t(seq, np.int32), t(mask, np.uint8), P, lam)


def compare(logp, seq, mask, P, lam):
    out, ell, g, st = run(logp, seq, mask, P, lam)
    assert st == 0
    ref = oracle.orpo_loss(logp.astype(np.float32).astype(np.float64), seq, mask, P, lam)
    for a, b in zip(out, ref.metrics()):
        assert abs(a - b) <= LOSS_RTOL * max(abs(b), 1e-6), (out, ref.metrics())
    assert np.allclose(ell, ref.ell, rtol=1e-6, atol=1e-7)
    assert np.allclose(g, ref.g, rtol=1e-5, atol=1e-12)
    assert np.all(g[(mask == 0) | (seq < 0)] == 0)


@pytest.mark.parametrize("name", ["tiny", "small", "e4b", "largev", "ragged"])
def test_workload_layouts(name):
    w = workloads.make(name, d=8, V=16)
    logp = workloads.synthetic_logp(3, w.seq_id, w.mask)
    compare(logp, w.seq_id, w.mask, w.n_pairs, w.lam)


def test_padding_anywhere_and_many_pairs():
    rng = np.random.default_rng(5)
    P = 300
    lengths = rng.integers(1, 40, size=2 * P)
    seq = np.repeat(np.arange(2 * P), lengths).astype(np.int32)
    # sprinkle padding rows (-1) at random places
    pads = rng.integers(0, len(seq), size=500)
    seq = np.insert(seq, np.sort(pads), -1).astype(np.int32)
    mask = (rng.random(len(seq)) > 0.2).astype(np.uint8)
    mask[seq < 0] = 0
    # guarantee each sequence keeps a response row
    for s in range(2 * P):
        mask[np.where(seq == s)[0][-1]] = 1
    logp = workloads.synthetic_logp(7, seq, mask, scale=1.0, offset=-0.5)
    compare(logp, seq, mask, P, 0.25)


def test_lambda_zero_and_big_lambda():
    w = workloads.make("small", d=8, V=16)
    logp = workloads.synthetic_logp(1, w.seq_id, w.mask)
    compare(logp, w.seq_id, w.mask, w.n_pairs, 0.0)
    compare(logp, w.seq_id, w.mask, w.n_pairs, 5.0)


def test_near_zero_mean_logp_is_stable():
    seq = np.array([0] * 4 + [1] * 4, dtype=np.int32)
    mask = np.ones(8, dtype=np.uint8)
    logp = np.array([-1e-6] * 4 + [-2.0] * 4, dtype=np.float32)
    compare(logp, seq, mask, 1, 0.1)


def test_errors_are_flagged():
    seq = np.array([0, 0, 1, 1], dtype=np.int32)
    logp = np.full(4, -1.0, dtype=np.float32)
    _, _, _, st = run(logp, seq, np.array([1, 1, 0, 0], np.uint8), 1, 0.1)
    assert st & (1 << 6)                       # empty rejected response
    _, _, _, st = run(logp, np.array([0, 1, 0, 1], np.int32), np.ones(4, np.uint8), 1, 0.1)
    assert st & (1 << 5)                       # ids decrease
    _, _, _, st = run(logp, np.array([0, 0, 1, 2], np.int32), np.ones(4, np.uint8), 1, 0.1)
    assert st & (1 << 5)                       # id beyond 2P
    _, _, _, st = run(np.array([0, 0, -1, -1], np.float32), seq, np.ones(4, np.uint8), 1, 0.1)
    assert st & (1 << 7)                       # l_w = 0: log1mexp is -inf


def test_bitwise_reproducible():
    w = workloads.make("ragged", d=8, V=16)
    logp = workloads.synthetic_logp(2, w.seq_id, w.mask)
    a = run(logp, w.seq_id, w.mask, w.n_pairs, w.lam)
    b = run(logp, w.seq_id, w.mask, w.n_pairs, w.lam)
    assert all(np.array_equal(x, y) for x, y in zip(a[:3], b[:3]))


def test_largest_pair_count():
    # ORPO_MAX_PAIRS pairs: the loss kernel's largest shared-memory layout
    import orpo_preference_loss_gb300 as orpo
    P = orpo.MAX_PAIRS
    rng = np.random.default_rng(11)
    lengths = rng.integers(1, 9, size=2 * P)
    seq = np.repeat(np.arange(2 * P), lengths).astype(np.int32)
    mask = np.ones(len(seq), dtype=np.uint8)
    logp = workloads.synthetic_logp(13, seq, mask, scale=1.0, offset=-0.5)
    compare(logp, seq, mask, P, 0.1)
    # and a small batch right after it on the same device still runs (the opt-in covers every size)
    seq2 = np.repeat(np.arange(4), 3).astype(np.int32)
    compare(workloads.synthetic_logp(14, seq2, np.ones(12, np.uint8)), seq2, np.ones(12, np.uint8), 2, 0.1)
