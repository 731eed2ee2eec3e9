"""Plain float64 oracle for the flash-CCE ORPO head (CPU, numpy).

TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU
baseline call this module; the CUDA library never does.  Every quantity is the
plain definition written out in float64 on the exact values of the bf16 inputs
(no rounding to bf16 or fp32 anywhere), with the vocabulary processed in row
chunks so that a bounded ``[chunk, V]`` block is the largest array held.

Sources (mlx-bun "Training — design (ORPO, flash-CCE head, prefix sharing,
segmented backward)" page, and the "Steel flash-CCE — handoff" page):

* ``head_forward``  — §5.1 "The head: from token-chunking to the flash-CCE
  kernel": per-token ``logp_t = z~[t, y_t] - logsumexp_v z~[t, v]`` with
  ``z = h W^T`` and the Gemma final-logit softcap ``z~ = c tanh(z / c)``
  (implementation spec of the fused linear-CE head, forward bullet).
* ``orpo_loss``     — §1 "The objective": ``L = NLL(chosen) + lambda * L_OR``,
  ``L_OR = -log sigmoid(log_odds)``,
  ``log_odds = (l_w - l_r) - (log1mexp(l_w) - log1mexp(l_r))`` with ``l`` the
  length-normalised (mean) response log-probability; batch reduction
  ``nll = mean(-l_w)``, ``or = mean(softplus(-log_odds))`` (file-by-file
  ``loss.ts`` bullet); metrics loss / nll / or / accuracy (``l_w > l_r``) /
  margin (mean chosen-minus-rejected log-odds, "Small sets over-fit fast").
  NLL scope is the ``response`` reading (``NLL = -l_w``).
* ``pref_loss``     — the sibling objectives on the same logp engine ("Training
  — design" §8.3 SimPO; the xtrain post-training page, Stage P1, for DPO's
  summed sequence log-prob with cached reference log-probs; IPO and hinge are
  named there without formulas and take their standard forms).
* ``dequant_affine`` — the quantised head's weights (§5.1 tier 4: the head is
  4/8-bit affine group-quantised with scales and biases; here dequantised to
  bf16 before the contraction, see the function).
* ``head_backward`` — implementation spec, backward bullet: recompute the
  logits, ``dZ = g * (onehot_y - softmax(z~)) * sech^2(z / c)``, then
  ``dh = dZ W`` and (the head-weight gradient that the pages leave to the
  head-LoRA follow-on) ``dW = dZ^T h``.  Optionally with the coefficient
  filter of the backward skips ("Steel flash-CCE — handoff" §E; "Training —
  design" §5.1): tiles of the coefficient that lie wholly below eps are dropped.
* ``head_block_max`` — the forward's per-(row group, vocabulary tile) maxima of
  the softcapped logits that the block skip reads (handoff §E, blockMax).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, library routines, invariants and central finite differences).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

LN2 = math.log(2.0)


class OracleError(ValueError):
    """Raised where the GPU library reports a data error through its status word."""

    def __init__(self, kind: str, msg: str):
        super().__init__(f"{kind}: {msg}")
        self.kind = kind


# --------------------------------------------------------------------------
# inputs
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of bf16 bit patterns (uint16): bf16 is the top half of fp32."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    f32 = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return f32.astype(np.float64)


# --------------------------------------------------------------------------
# scalar pieces
# --------------------------------------------------------------------------

def log1mexp(x):
    """log(1 - exp(x)) for x < 0, two-branch form (Maechler 2012).

    The ORPO objective (§1) needs log(1 - e^l) for the mean log-prob l; the pages
    flag the x -> 0^- end as the NaN hazard and ask for a clamp or a two-branch
    form.  Branch point -ln 2: log(-expm1(x)) above it, log1p(-exp(x)) below.
    x = 0 gives -inf (the GPU path reports that as a non-finite loss).
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(divide="ignore"):
        out = np.where(x > -LN2,
                       np.log(-np.expm1(np.minimum(x, 0.0))),
                       np.log1p(-np.exp(np.minimum(x, 0.0))))
    if np.any(x > 0):
        raise OracleError("arg", "log1mexp is defined for x <= 0 only")
    return out if out.ndim else float(out)


def softplus(x):
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def softcap_value(z: np.ndarray, c: float) -> np.ndarray:
    """z~ = c * tanh(z / c) when c > 0, else z (softcap off)."""
    return c * np.tanh(z / c) if c > 0 else z


def softcap_slope(z: np.ndarray, c: float) -> np.ndarray:
    """d z~ / d z = 1 - tanh^2(z / c) = sech^2(z / c) when c > 0, else 1."""
    if c > 0:
        t = np.tanh(z / c)
        return 1.0 - t * t
    return np.ones_like(z)


PROMPT = 2  # mask value of a prompt row that only the full-scope NLL supervises


def _response_rows(mask) -> np.ndarray:
    """Response rows: nonzero mask other than the prompt marker."""
    m = np.asarray(mask)
    return (m != 0) & (m != PROMPT)


def _row_chunk(V: int, budget_elems: int = 1 << 23) -> int:
    return max(1, budget_elems // max(1, V))


# --------------------------------------------------------------------------
# head forward: logp and lse
# --------------------------------------------------------------------------

def head_forward(h: np.ndarray, W: np.ndarray, targets: np.ndarray, mask: np.ndarray,
                 softcap: float = 0.0):
    """Per-token response log-prob and log-sum-exp.

    h [M, d], W [V, d] float64; targets [M] int; mask [M] (0 = prompt/pad row).
    Returns (logp [M], lse [M]).  lse is defined for every row; logp is 0 on
    mask = 0 rows, whose targets are never read.  A target outside [0, V) on a
    mask = 1 row raises OracleError("target").
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    M, V = h.shape[0], W.shape[0]
    targets = np.asarray(targets).astype(np.int64)
    mask = np.asarray(mask).astype(bool)
    logp = np.zeros(M, dtype=np.float64)
    lse = np.zeros(M, dtype=np.float64)
    bad = mask & ((targets < 0) | (targets >= V))
    if np.any(bad):
        raise OracleError("target", f"target out of range on row {int(np.argmax(bad))}")
    step = _row_chunk(V)
    for r0 in range(0, M, step):
        r1 = min(M, r0 + step)
        z = softcap_value(h[r0:r1] @ W.T, softcap)          # [rows, V]
        zmax = z.max(axis=1)
        lse[r0:r1] = zmax + np.log(np.exp(z - zmax[:, None]).sum(axis=1))
        rows = np.arange(r1 - r0)
        m = mask[r0:r1]
        tgt = z[rows[m], targets[r0:r1][m]]
        logp[r0:r1][m] = tgt - lse[r0:r1][m]
    return logp, lse


# --------------------------------------------------------------------------
# ORPO loss over sequences / pairs
# --------------------------------------------------------------------------

@dataclass
class LossResult:
    loss: float
    nll: float
    orr: float          # mean L_OR
    accuracy: float
    margin: float
    ell: np.ndarray     # [2P] mean response log-prob per sequence
    log_odds: np.ndarray  # [P]
    g: np.ndarray       # [M] dL/dlogp_t
    n: np.ndarray       # [2P] response-token count per sequence

    def metrics(self) -> np.ndarray:
        return np.array([self.loss, self.nll, self.orr, self.accuracy, self.margin])


def orpo_loss(logp: np.ndarray, seq_id: np.ndarray, mask: np.ndarray, n_pairs: int,
              lam: float, scope: str = "response") -> LossResult:
    """ORPO objective and its gradient with respect to every per-token logp.

    Sequence 2p is the chosen response of pair p and 2p+1 the rejected one.
    Rows with seq_id = -1 are padding.  mask: 0 = not supervised, 2 = prompt
    row (only the full-scope NLL sees it), any other nonzero value = response
    row.  l_s is the mean of logp over the response rows of sequence s.  Per pair:
        x_p  = (l_w - l_r) - (log1mexp(l_w) - log1mexp(l_r))
        L    = (1/P) sum_p [ NLL_p + lam * softplus(-x_p) ]
    with NLL_p = -l_w (scope "response"), or, for scope "full" ("Training —
    design" §1, combineFullNll), the token mean of -logp over the chosen
    sequence's prompt and response rows: -((P-1) pm + M l_w) / ((P-1) + M).
    Gradient (closed form; d x / d l_w = 1 / (1 - e^{l_w})):
        OR part: G_w = -(lam/P) sigmoid(-x) / (1 - e^{l_w}),
                 G_r =  (lam/P) sigmoid(-x) / (1 - e^{l_r}),  spread as G_s / n_s
                 over the response rows of s;
        NLL part: -1/(P n_w) on the chosen response rows (response scope), or
                 -1/(P N_w) on every chosen prompt and response row (full scope).
    """
    if scope not in ("response", "full"):
        raise OracleError("arg", "scope is 'response' or 'full'")
    logp = np.asarray(logp, dtype=np.float64)
    seq_id = np.asarray(seq_id).astype(np.int64)
    P = int(n_pairs)
    if P < 1:
        raise OracleError("arg", "n_pairs must be >= 1")
    S = 2 * P
    if np.any((seq_id < -1) | (seq_id >= S)):
        raise OracleError("seqid", "sequence id out of range")
    valid = seq_id >= 0
    ids = seq_id[valid]
    if np.any(np.diff(ids) < 0):
        raise OracleError("seqid", "sequence ids are not non-decreasing")
    use = valid & _response_rows(mask)
    sup = valid & (np.asarray(mask) != 0)          # response + prompt rows (full-scope NLL)
    n = np.bincount(seq_id[use], minlength=S).astype(np.float64)
    if np.any(n == 0):
        raise OracleError("empty", f"sequence {int(np.argmin(n))} has no response token")
    tot = np.bincount(seq_id[use], weights=logp[use], minlength=S)
    ell = tot / n
    lw, lr = ell[0::2], ell[1::2]
    if np.any(ell > 0):
        raise OracleError("nonfinite", "a mean log-prob is positive")
    N = np.bincount(seq_id[sup], minlength=S).astype(np.float64)
    tot_full = np.bincount(seq_id[sup], weights=logp[sup], minlength=S)
    nll_p = -lw if scope == "response" else -(tot_full[0::2] / N[0::2])
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        x = (lw - lr) - (log1mexp(lw) - log1mexp(lr))
        lor = softplus(-x)
        nll = float(np.mean(nll_p))
        orr = float(np.mean(lor))
        loss = nll + lam * orr
        acc = float(np.mean(lw > lr))
        margin = float(np.mean(x))
        sig = sigmoid(-x)
        # 1 / (1 - e^l) = -1 / expm1(l)
        inv_w = -1.0 / np.expm1(lw)
        inv_r = -1.0 / np.expm1(lr)
        Gw = (-lam * sig * inv_w) / P
        Gr = (lam * sig * inv_r) / P
    # l = 0 (a response whose every target has probability 1) makes log1mexp
    # -inf; the value and gradient are then reported as non-finite, not clamped.
    if not (np.isfinite(loss) and np.all(np.isfinite(x)) and np.all(np.isfinite(Gw))
            and np.all(np.isfinite(Gr))):
        raise OracleError("nonfinite", "loss, log-odds or gradient is not finite")
    G = np.empty(S)
    G[0::2], G[1::2] = Gw, Gr
    g = np.zeros_like(logp)
    g[use] = G[seq_id[use]] / n[seq_id[use]]
    chosen = (seq_id % 2 == 0)
    if scope == "response":
        rows = use & chosen
        g[rows] += -1.0 / (P * n[seq_id[rows]])
    else:
        rows = sup & chosen
        g[rows] += -1.0 / (P * N[seq_id[rows]])
    return LossResult(loss=loss, nll=nll, orr=orr, accuracy=acc, margin=margin,
                      ell=ell, log_odds=x, g=g, n=n)


# --------------------------------------------------------------------------
# head backward: dh and dW
# --------------------------------------------------------------------------

TILE_ROWS, TILE_COLS = 128, 256   # tile of the backward skips (rows x vocabulary columns)
GROUP_ROWS = 32                    # row group of the forward's block maxima


def _tile_keep(coef: np.ndarray, active: np.ndarray, eps: float, tile=(TILE_ROWS, TILE_COLS)) -> np.ndarray:
    """Element mask of the tiles that the coefficient filter keeps.

    "Steel flash-CCE — handoff" §E (coefficient filter) and "Training — design"
    §5.1 (the Apple-CCE backward skips, default eps 1e-5): a block of the
    coefficient whose entries all lie below eps is skipped.  The block here is a
    tile of ``tile`` rows x columns aligned to row 0 and vocabulary column 0 of
    the whole [M, V] coefficient, and the coefficient is the part of dZ that
    does not depend on the batch scale, (onehot - p) sech^2, taken over the rows
    whose cotangent g is nonzero (the other rows' dZ is identically 0).  A tile
    is kept when one such entry has magnitude >= eps.  ``coef`` holds a row
    chunk that starts on a tile boundary.
    """
    tr, tc = tile
    R, V = coef.shape
    a = np.where(active[:, None], np.abs(coef), 0.0)
    nr, nc = -(-R // tr), -(-V // tc)
    padded = np.zeros((nr * tr, nc * tc))
    padded[:R, :V] = a
    keep = padded.reshape(nr, tr, nc, tc).max(axis=(1, 3)) >= eps
    return np.repeat(np.repeat(keep, tr, axis=0), tc, axis=1)[:R, :V]


def head_block_max(h: np.ndarray, W: np.ndarray, mask: np.ndarray, softcap: float = 0.0,
                   group=(GROUP_ROWS, TILE_COLS)) -> np.ndarray:
    """Block maxima of the softcapped logits, in base-2 units (z~ log2 e).

    "Steel flash-CCE — handoff" §E (blockMax vocabulary-block skip: the
    backward skips cold (token block, vocabulary block) programs using the
    forward's blockMax).  Entry [q, j] is the largest z~[t, v] log2(e) over the
    rows t of row group q (``group[0]`` rows from row 0) with mask != 0 and the
    columns v of vocabulary tile j (``group[1]`` columns); -inf where the group
    has no such row.  Shape [ceil(M / group[0]), ceil(V / group[1])].
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    M, V = h.shape[0], W.shape[0]
    gr, gc = group
    nq, nj = -(-M // gr), -(-V // gc)
    mask = np.asarray(mask).astype(bool)
    out = np.full((nq, nj), -np.inf)
    step = max(gr, _row_chunk(V) // gr * gr)
    for r0 in range(0, M, step):
        r1 = min(M, r0 + step)
        z = softcap_value(h[r0:r1] @ W.T, softcap) / LN2
        z[~mask[r0:r1]] = -np.inf
        R = r1 - r0
        padded = np.full((-(-R // gr) * gr, nj * gc), -np.inf)
        padded[:R, :V] = z
        out[r0 // gr:r0 // gr + padded.shape[0] // gr] = padded.reshape(-1, gr, nj, gc).max(axis=(1, 3))
    return out


def head_backward(h: np.ndarray, W: np.ndarray, targets: np.ndarray, mask: np.ndarray,
                  lse: np.ndarray, g: np.ndarray, softcap: float = 0.0, filter_eps: float = 0.0,
                  tile=(TILE_ROWS, TILE_COLS), vocab=None):
    """dh = dZ W and dW = dZ^T h with dZ = g (onehot_y - softmax(z~)) sech^2(z/c).

    softmax is rebuilt from the given lse: p = exp(z~ - lse).  Rows with
    mask = 0 carry no gradient (their g is treated as 0 and their target is not
    read).  With ``filter_eps`` > 0 the coefficient filter of the backward
    skips applies: every ``tile`` of dZ whose coefficient entries all lie below
    filter_eps is dropped (see ``_tile_keep``).  Returns (dh [M, d], dW [V, d])
    in float64.  ``vocab = (c0, c1)`` restricts the sums to vocabulary columns
    [c0, c1) (c0 on a tile boundary; lse still covers the whole vocabulary):
    dh is then their share of the gradient and dW holds rows c0 .. c1-1 only.
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    M, d = h.shape
    targets = np.asarray(targets).astype(np.int64)
    mask = np.asarray(mask).astype(bool)
    if vocab is not None:
        c0, c1 = vocab
        if c0 % tile[1] != 0:
            raise OracleError("arg", "a vocabulary slice starts on a tile boundary")
        W = W[c0:c1]
        inside = (targets >= c0) & (targets < c1)
        targets = np.where(inside, targets - c0, 0)
        onehot_rows = mask & inside
    else:
        onehot_rows = mask
    V = W.shape[0]
    lse = np.asarray(lse, dtype=np.float64)
    g = np.where(mask, np.asarray(g, dtype=np.float64), 0.0)
    dh = np.zeros((M, d))
    dW = np.zeros((V, d))
    step = _row_chunk(V)
    if filter_eps > 0:
        step = max(tile[0], step // tile[0] * tile[0])  # chunks start on tile boundaries
    for r0 in range(0, M, step):
        r1 = min(M, r0 + step)
        gr = g[r0:r1]
        if not np.any(gr != 0.0):
            continue
        z = h[r0:r1] @ W.T
        zt = softcap_value(z, softcap)
        p = np.exp(zt - lse[r0:r1, None])
        onehot = np.zeros_like(p)
        rows = np.arange(r1 - r0)
        m = onehot_rows[r0:r1]
        onehot[rows[m], targets[r0:r1][m]] = 1.0
        coef = (onehot - p) * softcap_slope(z, softcap)
        if filter_eps > 0:
            coef = np.where(_tile_keep(coef, gr != 0.0, filter_eps, tile), coef, 0.0)
        dZ = gr[:, None] * coef
        dh[r0:r1] = dZ @ W
        dW += dZ.T @ h[r0:r1]
    return dh, dW


def full_chain(h, W, targets, mask, seq_id, n_pairs, lam, softcap=0.0, scope="response"):
    """Forward, loss and backward in sequence, as one training step of the head."""
    logp, lse = head_forward(h, W, targets, mask, softcap)
    res = orpo_loss(logp, seq_id, mask, n_pairs, lam, scope)
    dh, dW = head_backward(h, W, targets, mask, lse, res.g, softcap)
    return logp, lse, res, dh, dW


# --------------------------------------------------------------------------
# sibling preference objectives on the same per-token logp
# --------------------------------------------------------------------------

PREF_KINDS = ("orpo", "simpo", "dpo", "ipo", "hinge")


def pref_loss(kind: str, logp, seq_id, mask, n_pairs: int, beta: float, gamma: float = 0.0, ref=None):
    """Preference objective `kind` over pairs, value and gradient w.r.t. each logp.

    orpo  : the ORPO objective above with lambda = beta (gamma unused).
    simpo : mean response log-prob l; per pair softplus(-beta((l_w - l_r) - gamma))
            ("Training — design" §8.3); no NLL term.
    dpo   : per-sequence SUM s of logp over response rows, cached reference sums
            r (ref[2P]); D = (s_w - r_w) - (s_r - r_r); per pair
            -log sigmoid(beta * D) (xtrain post-training page, Stage P1).
    ipo   : (D - 1/(2 beta))^2 on the same D (the standard IPO loss; the pages
            only name it).
    hinge : max(0, 1 - beta * D) (SLiC-style hinge on the same D; named only).
    The batch value is the mean over pairs.  Returns a LossResult whose `ell`
    holds the per-sequence mean (orpo, simpo) or sum (dpo, ipo, hinge), `nll`
    is mean(-ell_w), `orr` the mean preference term, `accuracy` the fraction of
    pairs whose chosen statistic (ell_w, or s_w - r_w) beats the rejected one,
    and `margin` the mean of the argument the preference term is applied to.
    """
    if kind == "orpo":
        return orpo_loss(logp, seq_id, mask, n_pairs, beta)
    if kind not in PREF_KINDS:
        raise OracleError("arg", f"unknown kind {kind}")
    logp = np.asarray(logp, dtype=np.float64)
    seq_id = np.asarray(seq_id).astype(np.int64)
    P = int(n_pairs)
    S = 2 * P
    if P < 1:
        raise OracleError("arg", "n_pairs must be >= 1")
    if np.any((seq_id < -1) | (seq_id >= S)) or np.any(np.diff(seq_id[seq_id >= 0]) < 0):
        raise OracleError("seqid", "bad sequence ids")
    use = (seq_id >= 0) & _response_rows(mask)
    n = np.bincount(seq_id[use], minlength=S).astype(np.float64)
    if np.any(n == 0):
        raise OracleError("empty", "a sequence has no response token")
    tot = np.bincount(seq_id[use], weights=logp[use], minlength=S)
    mean_kind = kind == "simpo"
    ell = tot / n if mean_kind else tot
    w, r = ell[0::2], ell[1::2]
    if mean_kind:
        u = beta * ((w - r) - gamma)
        term = softplus(-u)
        dterm_dw = -beta * sigmoid(-u)             # d term / d l_w ; d / d l_r is the negative
        chosen_better = w > r
        margin = u
    else:
        if ref is None:
            raise OracleError("arg", "reference log-probs are required")
        ref = np.asarray(ref, dtype=np.float64)
        D = (w - ref[0::2]) - (r - ref[1::2])
        chosen_better = D > 0
        if kind == "dpo":
            term = softplus(-beta * D)
            dterm_dw = -beta * sigmoid(-beta * D)
            margin = beta * D
        elif kind == "ipo":
            if beta <= 0:
                raise OracleError("arg", "ipo needs beta > 0")
            c = D - 1.0 / (2.0 * beta)
            term = c * c
            dterm_dw = 2.0 * c
            margin = D
        else:  # hinge
            a = 1.0 - beta * D
            term = np.maximum(a, 0.0)
            dterm_dw = np.where(a > 0, -beta, 0.0)
            margin = beta * D
    G = np.empty(S)
    G[0::2] = dterm_dw / P
    G[1::2] = -dterm_dw / P
    g = np.zeros_like(logp)
    scale = n[seq_id[use]] if mean_kind else 1.0
    g[use] = G[seq_id[use]] / scale
    loss = float(np.mean(term))
    if not np.isfinite(loss):
        raise OracleError("nonfinite", "loss is not finite")
    return LossResult(loss=loss, nll=float(np.mean(-w)), orr=loss, accuracy=float(np.mean(chosen_better)),
                      margin=float(np.mean(margin)), ell=ell, log_odds=margin, g=g, n=n)


# --------------------------------------------------------------------------
# quantized head: affine group dequantisation
# --------------------------------------------------------------------------

def _round_bf16(x32: np.ndarray) -> np.ndarray:
    """fp32 -> nearest-even bf16, returned as float64 values."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return (r.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def dequant_affine(wq: np.ndarray, scales_bits: np.ndarray, biases_bits: np.ndarray, bits: int, group: int,
                   d: int) -> np.ndarray:
    """Weights of an affine group-quantised head ("Training — design" §5.1 tier 4: 4/8-bit affine
    dequant with per-group scales and biases).

    wq: uint8 [V, d * bits / 8]; for 4 bits element j of a row is the low nibble of byte j/2 when j
    is even and the high nibble when j is odd; for 8 bits it is byte j.  scales, biases: bf16 bit
    patterns [V, d / group].  The head's weight is W[v, j] = bf16(scale * q + bias), the product and
    sum taken in fp32 (the product of a bf16 scale and q < 256 is exact) and rounded once to bf16,
    nearest even.  Returns W as float64 [V, d].
    """
    wq = np.asarray(wq, dtype=np.uint8)
    V = wq.shape[0]
    if bits == 4:
        q = np.empty((V, d), dtype=np.uint8)
        q[:, 0::2] = wq & 0x0F
        q[:, 1::2] = wq >> 4
    elif bits == 8:
        q = wq[:, :d]
    else:
        raise OracleError("arg", "bits must be 4 or 8")
    s = bf16_bits_to_f64(scales_bits).astype(np.float32)
    b = bf16_bits_to_f64(biases_bits).astype(np.float32)
    s_full = np.repeat(s, group, axis=1)[:, :d]
    b_full = np.repeat(b, group, axis=1)[:, :d]
    w32 = s_full * q.astype(np.float32) + b_full
    return _round_bf16(w32)
