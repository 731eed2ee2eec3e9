"""Pins for the float64 oracle: each check ties it to something other than itself.

closed forms (tests/golden/orpo_closed_form.txt), library routines
(torch cross_entropy / logsigmoid in float64, mpmath at 50 digits), invariants
(uniform logits, logit shift, softmax row sums) and central finite differences.
"""

import math
import os

import mpmath
import numpy as np
import pytest
import torch

import oracle
from oracle import OracleError

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- log1mexp

def test_log1mexp_closed_values():
    mpmath.mp.dps = 50
    assert oracle.log1mexp(-math.log(2.0)) == pytest.approx(-math.log(2.0), rel=1e-15)
    # log(1 - e^-1e-10) = log(1e-10 - 5e-21 + ...) = -23.02585092994045... (mpmath below)
    v = oracle.log1mexp(-1e-10)
    ref = float(mpmath.log(1 - mpmath.exp(mpmath.mpf("-1e-10"))))
    assert v == pytest.approx(ref, rel=1e-14)
    assert abs(v - (-23.025850929990457)) < 1e-12
    v50 = oracle.log1mexp(-50.0)
    assert v50 == pytest.approx(-1.9287498479639178e-22, rel=1e-12)


def test_log1mexp_matches_mpmath_and_is_stable():
    mpmath.mp.dps = 400   # enough digits for 1 - e^x down to x = -800
    xs = -np.concatenate([np.logspace(-300, -1, 60), np.linspace(0.05, 5, 60),
                          np.linspace(5, 800, 40)])
    vals = oracle.log1mexp(xs)
    assert np.all(np.isfinite(vals))
    for x, v in zip(xs, vals):
        ref = float(mpmath.log(-mpmath.expm1(mpmath.mpf(float(x)))))
        assert v == pytest.approx(ref, rel=1e-13, abs=1e-300)
    order = np.argsort(xs)
    # 1 - e^x shrinks as x rises toward 0, so log1mexp is non-increasing in x
    assert np.all(np.diff(vals[order]) <= 0), "log1mexp must be non-increasing"


# ---------------------------------------------------------------- ORPO loss closed forms

def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "orpo_closed_form.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows


def _ev(expr):
    mpmath.mp.dps = 50
    return float(eval(expr, {"ln": lambda v: mpmath.log(mpmath.mpf(v)), "__builtins__": {}}))


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_orpo_closed_form(row):
    name, lw, lr, lam, x, lor, L, gw, gr = row
    lw, lr, lam = _ev(lw), _ev(lr), _ev(lam)
    # two-token sequences with the given mean, so a sum-instead-of-mean slip shows
    logp = np.array([lw + 0.25, lw - 0.25, lr - 0.5, lr + 0.5])
    seq = np.array([0, 0, 1, 1])
    mask = np.ones(4, dtype=np.uint8)
    res = oracle.orpo_loss(logp, seq, mask, 1, lam)
    assert res.log_odds[0] == pytest.approx(_ev(x), abs=1e-13)
    assert res.orr == pytest.approx(_ev(lor), rel=1e-13)
    assert res.loss == pytest.approx(_ev(L), rel=1e-13)
    assert res.nll == pytest.approx(-lw, rel=1e-14)
    # per-token gradient = per-sequence gradient / n_s (n_s = 2 here)
    assert res.g[0] == pytest.approx(_ev(gw) / 2, rel=1e-12, abs=1e-15)
    assert res.g[2] == pytest.approx(_ev(gr) / 2, rel=1e-12, abs=1e-15)


def test_orpo_two_pairs_mean_over_pairs_and_library_logsigmoid():
    # pair 0 = golden "half_quarter", pair 1 = golden "swapped": loss is their mean
    lw = np.array([math.log(0.5), math.log(0.25)])
    lr = np.array([math.log(0.25), math.log(0.5)])
    logp = np.array([lw[0], lr[0], lr[0], lw[1], lr[1]])
    seq = np.array([0, 1, 1, 2, 3])
    res = oracle.orpo_loss(logp, seq, np.ones(5), 2, 0.1)
    x = np.array([math.log(3), -math.log(3)])
    lor_lib = -torch.nn.functional.logsigmoid(torch.tensor(x, dtype=torch.float64)).numpy()
    assert res.orr == pytest.approx(lor_lib.mean(), rel=1e-14)
    assert res.loss == pytest.approx(np.mean(-lw) + 0.1 * lor_lib.mean(), rel=1e-14)
    assert res.accuracy == 0.5
    assert res.margin == pytest.approx(0.0, abs=1e-14)
    # per-sequence ell uses the mean over its own rows
    assert res.ell[1] == pytest.approx(lr[0])
    assert list(res.n) == [1, 2, 1, 1]


def test_orpo_gradient_matches_finite_differences():
    rng = np.random.default_rng(3)
    M = 23
    seq = np.array([0] * 4 + [1] * 6 + [-1] + [2] * 3 + [3] * 5 + [-1] * 2 + [4, 5])
    mask = np.ones(M, dtype=np.uint8)
    mask[[0, 4, 11]] = 0
    logp = -0.2 - 3 * np.abs(rng.standard_normal(M))
    lam = 0.37
    res = oracle.orpo_loss(logp, seq, mask, 3, lam)
    eps = 1e-6
    for t in range(M):
        lp, lm = logp.copy(), logp.copy()
        lp[t] += eps
        lm[t] -= eps
        fd = (oracle.orpo_loss(lp, seq, mask, 3, lam).loss
              - oracle.orpo_loss(lm, seq, mask, 3, lam).loss) / (2 * eps)
        assert res.g[t] == pytest.approx(fd, rel=1e-6, abs=1e-9), t
        if mask[t] == 0 or seq[t] < 0:
            assert res.g[t] == 0.0


def test_orpo_errors():
    with pytest.raises(OracleError) as e:
        oracle.orpo_loss(np.array([-1.0, -1.0]), np.array([0, 0]), np.ones(2), 1, 0.1)
    assert e.value.kind == "empty"
    with pytest.raises(OracleError) as e:
        oracle.orpo_loss(np.array([-1.0, -1.0]), np.array([1, 0]), np.ones(2), 1, 0.1)
    assert e.value.kind == "seqid"
    with pytest.raises(OracleError) as e:
        oracle.orpo_loss(np.array([-1.0, -1.0]), np.array([0, 2]), np.ones(2), 1, 0.1)
    assert e.value.kind == "seqid"
    with pytest.raises(OracleError) as e:
        oracle.orpo_loss(np.array([0.0, -1.0]), np.array([0, 1]), np.ones(2), 1, 0.1)
    assert e.value.kind == "nonfinite"


# ---------------------------------------------------------------- head forward

@pytest.mark.parametrize("softcap", [0.0, 30.0])
def test_uniform_logits_give_minus_log_v(softcap):
    M, d, V = 5, 8, 37
    h = _rand(0, M, d)
    W = np.zeros((V, d))
    y = np.arange(M) % V
    logp, lse = oracle.head_forward(h, W, y, np.ones(M), softcap)
    assert np.all(logp == -math.log(V)) or np.allclose(logp, -math.log(V), atol=1e-15)
    assert np.allclose(lse, math.log(V), atol=1e-15)
    logp2, _ = oracle.head_forward(np.zeros((M, d)), _rand(1, V, d), y, np.ones(M), softcap)
    assert np.allclose(logp2, -math.log(V), atol=1e-15)


@pytest.mark.parametrize("softcap", [0.0, 3.0])
def test_forward_matches_torch_cross_entropy(softcap):
    M, d, V = 17, 12, 53
    h, W = _rand(4, M, d, scale=2.0), _rand(5, V, d)
    y = np.random.default_rng(6).integers(0, V, M)
    mask = np.ones(M, dtype=np.uint8)
    mask[[2, 9]] = 0
    logp, lse = oracle.head_forward(h, W, y, mask, softcap)
    z = torch.tensor(h) @ torch.tensor(W).T
    if softcap > 0:
        z = softcap * torch.tanh(z / softcap)
    ce = torch.nn.functional.cross_entropy(z, torch.tensor(y), reduction="none").numpy()
    assert np.allclose(logp[mask == 1], -ce[mask == 1], rtol=1e-13, atol=1e-12)
    assert np.all(logp[mask == 0] == 0)
    assert np.allclose(lse, torch.logsumexp(z, dim=1).numpy(), rtol=1e-14, atol=1e-12)


def test_forward_logit_shift_invariance():
    # an extra constant feature shifts every logit of a row by the same amount
    M, d, V = 9, 6, 31
    h, W = _rand(7, M, d), _rand(8, V, d)
    y = np.arange(M) * 3 % V
    c = 11.5
    h2 = np.concatenate([h, np.ones((M, 1))], axis=1)
    W2 = np.concatenate([W, np.full((V, 1), c)], axis=1)
    lp1, ls1 = oracle.head_forward(h, W, y, np.ones(M))
    lp2, ls2 = oracle.head_forward(h2, W2, y, np.ones(M))
    assert np.allclose(lp1, lp2, atol=1e-13)
    assert np.allclose(ls2 - ls1, c, atol=1e-12)


def test_softcap_large_cap_reduces_to_off():
    M, d, V = 6, 10, 40
    h, W = _rand(9, M, d), _rand(10, V, d)
    y = np.arange(M)
    a, _ = oracle.head_forward(h, W, y, np.ones(M), 0.0)
    b, _ = oracle.head_forward(h, W, y, np.ones(M), 1e6)
    assert np.allclose(a, b, atol=1e-9)
    z = np.linspace(-40, 40, 81)
    eps = 1e-6
    fd = (oracle.softcap_value(z + eps, 30.0) - oracle.softcap_value(z - eps, 30.0)) / (2 * eps)
    assert np.allclose(oracle.softcap_slope(z, 30.0), fd, rtol=1e-8, atol=1e-10)


def test_forward_target_errors_only_on_response_rows():
    h, W = _rand(1, 3, 4), _rand(2, 5, 4)
    y = np.array([1, 99, 2])
    with pytest.raises(OracleError) as e:
        oracle.head_forward(h, W, y, np.ones(3))
    assert e.value.kind == "target"
    logp, _ = oracle.head_forward(h, W, y, np.array([1, 0, 1]))
    assert logp[1] == 0.0


# ---------------------------------------------------------------- backward

def _tiny_problem(softcap, seed=11):
    rng = np.random.default_rng(seed)
    M, d, V, P = 12, 8, 16, 2
    seq = np.array([0, 0, 0, 1, 1, 1, 1, 1, 2, 2, 3, 3])
    mask = np.ones(M, dtype=np.uint8)
    mask[[0, 3]] = 0
    h = rng.standard_normal((M, d)) * 1.5
    W = rng.standard_normal((V, d)) * 0.9
    y = rng.integers(0, V, M)
    return h, W, y, mask, seq, P, 0.3, softcap


def _loss_of(h, W, y, mask, seq, P, lam, softcap):
    logp, _ = oracle.head_forward(h, W, y, mask, softcap)
    return oracle.orpo_loss(logp, seq, mask, P, lam).loss


@pytest.mark.parametrize("softcap", [0.0, 2.5])
def test_backward_matches_central_finite_differences(softcap):
    h, W, y, mask, seq, P, lam, c = _tiny_problem(softcap)
    _, _, res, dh, dW = oracle.full_chain(h, W, y, mask, seq, P, lam, c)
    eps = 1e-6
    fd_h = np.zeros_like(h)
    for i in range(h.shape[0]):
        for j in range(h.shape[1]):
            hp, hm = h.copy(), h.copy()
            hp[i, j] += eps
            hm[i, j] -= eps
            fd_h[i, j] = (_loss_of(hp, W, y, mask, seq, P, lam, c)
                          - _loss_of(hm, W, y, mask, seq, P, lam, c)) / (2 * eps)
    fd_W = np.zeros_like(W)
    for i in range(W.shape[0]):
        for j in range(W.shape[1]):
            Wp, Wm = W.copy(), W.copy()
            Wp[i, j] += eps
            Wm[i, j] -= eps
            fd_W[i, j] = (_loss_of(h, Wp, y, mask, seq, P, lam, c)
                          - _loss_of(h, Wm, y, mask, seq, P, lam, c)) / (2 * eps)
    assert np.allclose(dh, fd_h, rtol=1e-6, atol=1e-9)
    assert np.allclose(dW, fd_W, rtol=1e-6, atol=1e-9)
    assert np.all(dh[mask == 0] == 0)


def test_backward_row_sum_invariant():
    h, W, y, mask, seq, P, lam, _ = _tiny_problem(0.0, seed=5)
    _, _, res, dh, dW = oracle.full_chain(h, W, y, mask, seq, P, lam, 0.0)
    # without softcap every row of dZ sums to 0, so the columns of dW sum to 0
    assert np.allclose(dW.sum(axis=0), 0.0, atol=1e-13)


def test_backward_lambda_zero_is_chosen_cross_entropy():
    h, W, y, mask, seq, P, _, _ = _tiny_problem(0.0, seed=6)
    logp, lse, res, dh, dW = oracle.full_chain(h, W, y, mask, seq, P, 0.0, 0.0)
    # loss = mean over pairs of the mean CE of the chosen response (torch, float64)
    z = torch.tensor(h) @ torch.tensor(W).T
    ce = torch.nn.functional.cross_entropy(z, torch.tensor(y), reduction="none").numpy()
    want = np.mean([ce[(seq == 2 * p) & (mask == 1)].mean() for p in range(P)])
    assert res.loss == pytest.approx(want, rel=1e-13)
    rejected = (seq % 2 == 1)
    assert np.all(res.g[rejected] == 0) and np.all(dh[rejected] == 0)
    # and the chosen rows' dh equals autograd of that CE (torch, float64)
    ht = torch.tensor(h, requires_grad=True)
    zt = ht @ torch.tensor(W).T
    cet = torch.nn.functional.cross_entropy(zt, torch.tensor(y), reduction="none")
    tot = sum(cet[torch.tensor((seq == 2 * p) & (mask == 1))].mean() for p in range(P)) / P
    tot.backward()
    assert np.allclose(dh, ht.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_backward_masked_rows_ignore_targets():
    h, W, y, mask, seq, P, lam, c = _tiny_problem(2.5, seed=8)
    out1 = oracle.full_chain(h, W, y, mask, seq, P, lam, c)
    y2 = y.copy()
    y2[mask == 0] = 10 ** 6   # never read on prompt rows
    out2 = oracle.full_chain(h, W, y2, mask, seq, P, lam, c)
    assert np.array_equal(out1[3], out2[3]) and np.array_equal(out1[4], out2[4])
