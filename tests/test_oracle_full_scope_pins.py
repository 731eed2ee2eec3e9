"""Pins for the full-scope NLL (sft_scope = full) of the oracle.

"Training — design" §1: the NLL runs over the chosen sequence's prompt and
response positions, combined as -((P-1) pm + M l_w) / ((P-1) + M); the odds
ratio keeps response-only means.  Mask value 2 marks a supervised prompt row."""

import math

import numpy as np
import pytest
import torch

import oracle


def test_closed_form_full_scope():
    # chosen: prompt rows logp ln(1/2) x2, response ln(1/4) x2 ; rejected: response ln(1/8) x2
    logp = np.log(np.array([0.5, 0.5, 0.25, 0.25, 0.125, 0.125]))
    seq = np.array([0, 0, 0, 0, 1, 1])
    mask = np.array([2, 2, 1, 1, 1, 1])
    res = oracle.orpo_loss(logp, seq, mask, 1, 0.0, scope="full")
    assert res.loss == pytest.approx(1.5 * math.log(2.0), rel=1e-15)
    resp = oracle.orpo_loss(logp, seq, mask, 1, 0.0, scope="response")
    assert resp.loss == pytest.approx(2.0 * math.log(2.0), rel=1e-15)
    # the odds ratio ignores prompt rows in both scopes
    assert res.log_odds[0] == resp.log_odds[0]
    assert res.ell[0] == pytest.approx(math.log(0.25))


def test_matches_the_pages_combine_formula():
    rng = np.random.default_rng(2)
    Pm, Mr = 7, 5                                   # P - 1 prompt positions, M response positions
    logp = -np.abs(rng.standard_normal(Pm + Mr + 3)) - 0.1
    seq = np.array([0] * (Pm + Mr) + [1] * 3)
    mask = np.array([2] * Pm + [1] * Mr + [1] * 3)
    res = oracle.orpo_loss(logp, seq, mask, 1, 0.0, scope="full")
    pm = logp[:Pm].mean()
    lw = logp[Pm:Pm + Mr].mean()
    combine = -((Pm) * pm + Mr * lw) / (Pm + Mr)
    assert res.nll == pytest.approx(combine, rel=1e-14)


def test_lambda_zero_is_torch_mean_cross_entropy_over_prompt_and_response():
    rng = np.random.default_rng(4)
    M, d, V = 14, 6, 20
    h, W = rng.standard_normal((M, d)), rng.standard_normal((V, d))
    y = rng.integers(0, V, M)
    seq = np.array([0] * 8 + [1] * 6)
    mask = np.array([0, 2, 2, 2, 1, 1, 1, 1, 2, 1, 1, 1, 1, 1])
    logp, lse, res, dh, dW = oracle.full_chain(h, W, y, mask, seq, 1, 0.0, scope="full")
    z = torch.tensor(h) @ torch.tensor(W).T
    rows = torch.tensor((seq == 0) & (mask != 0))
    ce = torch.nn.functional.cross_entropy(z[rows], torch.tensor(y)[rows], reduction="mean")
    assert res.loss == pytest.approx(ce.item(), rel=1e-13)
    # rejected prompt rows carry no gradient in either scope
    assert np.all(res.g[(seq == 1) & (mask == 2)] == 0)


@pytest.mark.parametrize("lam", [0.0, 0.4])
def test_full_scope_gradient_matches_finite_differences(lam):
    rng = np.random.default_rng(9)
    seq = np.array([0] * 6 + [1] * 5 + [-1] + [2] * 4 + [3] * 3)
    mask = np.array([2, 2, 1, 1, 0, 1, 2, 1, 1, 1, 1, 0, 2, 1, 1, 1, 1, 1, 1])
    logp = -0.2 - 2 * np.abs(rng.standard_normal(len(seq)))
    res = oracle.orpo_loss(logp, seq, mask, 2, lam, scope="full")
    eps = 1e-6
    for t in range(len(seq)):
        lp, lm = logp.copy(), logp.copy()
        lp[t] += eps
        lm[t] -= eps
        fd = (oracle.orpo_loss(lp, seq, mask, 2, lam, scope="full").loss
              - oracle.orpo_loss(lm, seq, mask, 2, lam, scope="full").loss) / (2 * eps)
        assert res.g[t] == pytest.approx(fd, rel=1e-6, abs=1e-9), t


def test_full_scope_chain_matches_finite_differences():
    rng = np.random.default_rng(21)
    M, d, V = 10, 5, 12
    h, W = rng.standard_normal((M, d)), rng.standard_normal((V, d)) * 0.8
    y = rng.integers(0, V, M)
    seq = np.array([0] * 5 + [1] * 5)
    mask = np.array([2, 2, 1, 1, 1, 2, 1, 1, 1, 1])
    _, _, res, dh, dW = oracle.full_chain(h, W, y, mask, seq, 1, 0.3, 2.0, scope="full")

    def loss(hh, WW):
        lp, _ = oracle.head_forward(hh, WW, y, mask, 2.0)
        return oracle.orpo_loss(lp, seq, mask, 1, 0.3, scope="full").loss

    eps = 1e-6
    for (i, j) in [(0, 0), (1, 3), (4, 2), (5, 4), (9, 1)]:
        hp, hm = h.copy(), h.copy()
        hp[i, j] += eps
        hm[i, j] -= eps
        assert dh[i, j] == pytest.approx((loss(hp, W) - loss(hm, W)) / (2 * eps), rel=1e-6, abs=1e-9)
    for (i, j) in [(0, 0), (3, 1), (y[0], 2), (y[5], 4), (11, 3)]:
        Wp, Wm = W.copy(), W.copy()
        Wp[i, j] += eps
        Wm[i, j] -= eps
        assert dW[i, j] == pytest.approx((loss(h, Wp) - loss(h, Wm)) / (2 * eps), rel=1e-6, abs=1e-9)
