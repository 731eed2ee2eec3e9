"""Pins for the sibling preference objectives of the float64 oracle.

DPO: the xtrain post-training page's own degenerate gates (policy equal to the
reference gives Delta = 0 and L = log 2; beta -> 0 gives a vanishing gradient).
Every kind: a hand-derived closed form on two-token sequences (so a sum/mean
mix-up shows), torch logsigmoid where the value is a log-sigmoid, and central
finite differences of the batch value w.r.t. every token logp."""

import math

import numpy as np
import pytest
import torch

import oracle

SEQ = np.array([0, 0, 1, 1])
MASK = np.ones(4, dtype=np.uint8)


def two_token(w_each, r_each):
    return np.array([w_each, w_each, r_each, r_each], dtype=np.float64)


def test_dpo_policy_equal_reference_gives_log2():
    logp = two_token(-1.3, -2.1)
    ref = np.array([2 * -1.3, 2 * -2.1])       # reference sums equal the policy sums
    res = oracle.pref_loss("dpo", logp, SEQ, MASK, 1, 0.7, ref=ref)
    assert res.loss == pytest.approx(math.log(2.0), rel=1e-15)
    assert res.margin == 0.0
    # gradient at Delta = 0: -beta/2 on each chosen token (sum, not mean), +beta/2 on rejected
    assert np.allclose(res.g, [-0.35, -0.35, 0.35, 0.35], rtol=1e-14)


def test_dpo_beta_to_zero_kills_the_gradient():
    logp = two_token(-0.4, -3.0)
    ref = np.array([-2.0, -1.0])
    res = oracle.pref_loss("dpo", logp, SEQ, MASK, 1, 1e-12, ref=ref)
    assert np.max(np.abs(res.g)) < 1e-12
    assert res.loss == pytest.approx(math.log(2.0), rel=1e-9)


def test_dpo_closed_form_and_library_logsigmoid():
    # s_w = -2, r_w = -3 -> +1 ; s_l = -6, r_l = -5 -> -1 ; D = 2 ; beta = 0.5 -> L = softplus(-1)
    logp = two_token(-1.0, -3.0)
    res = oracle.pref_loss("dpo", logp, SEQ, MASK, 1, 0.5, ref=np.array([-3.0, -5.0]))
    lib = -torch.nn.functional.logsigmoid(torch.tensor(1.0, dtype=torch.float64)).item()
    assert res.loss == pytest.approx(lib, rel=1e-15)
    assert res.loss == pytest.approx(math.log(1 + math.exp(-1.0)), rel=1e-15)
    assert res.accuracy == 1.0 and res.margin == pytest.approx(1.0)
    assert list(res.ell) == [-2.0, -6.0]               # per-sequence SUM


def test_simpo_closed_form():
    # l_w = -1, l_r = -2, beta = 2, gamma = 0.5: u = 2((−1 − −2) − 0.5) = 1 -> softplus(-1)
    logp = np.array([-0.5, -1.5, -1.0, -3.0])
    res = oracle.pref_loss("simpo", logp, SEQ, MASK, 1, 2.0, 0.5)
    assert res.loss == pytest.approx(math.log(1 + math.exp(-1.0)), rel=1e-15)
    assert list(res.ell) == [-1.0, -2.0]              # per-sequence MEAN
    s = 1 / (1 + math.e)                                # sigmoid(-1)
    assert np.allclose(res.g, [-2 * s / 2, -2 * s / 2, 2 * s / 2, 2 * s / 2], rtol=1e-14)


def test_ipo_closed_forms():
    beta = 0.25                                        # 1/(2 beta) = 2
    ref = np.array([0.0, 0.0])
    at_target = oracle.pref_loss("ipo", two_token(-1.0, -2.0), SEQ, MASK, 1, beta, ref=ref)  # D = -2 + 4 = 2
    assert at_target.loss == 0.0 and np.all(at_target.g == 0)
    zero = oracle.pref_loss("ipo", two_token(-1.0, -1.0), SEQ, MASK, 1, beta, ref=ref)        # D = 0 -> 4
    assert zero.loss == pytest.approx(4.0)
    assert np.allclose(zero.g, [-4.0, -4.0, 4.0, 4.0])  # 2 (D - 2) = -4 on chosen tokens


def test_hinge_closed_forms():
    ref = np.array([0.0, 0.0])
    flat = oracle.pref_loss("hinge", two_token(-1.0, -1.0), SEQ, MASK, 1, 0.5, ref=ref)      # D = 0 -> 1
    assert flat.loss == 1.0 and np.allclose(flat.g, [-0.5, -0.5, 0.5, 0.5])
    done = oracle.pref_loss("hinge", two_token(-1.0, -2.0), SEQ, MASK, 1, 0.5, ref=ref)      # beta D = 1
    assert done.loss == 0.0 and np.all(done.g == 0)


@pytest.mark.parametrize("kind", oracle.PREF_KINDS)
def test_gradient_matches_finite_differences(kind):
    rng = np.random.default_rng(11)
    seq = np.array([0] * 3 + [1] * 5 + [-1] + [2] * 4 + [3] * 2 + [4, 5, 5])
    mask = np.ones(len(seq), dtype=np.uint8)
    mask[[0, 9]] = 0
    logp = -0.3 - 2 * np.abs(rng.standard_normal(len(seq)))
    ref = -1.0 - 2 * np.abs(rng.standard_normal(6))
    beta, gamma = 0.8, 0.3
    res = oracle.pref_loss(kind, logp, seq, mask, 3, beta, gamma, ref=ref)
    eps = 1e-6
    for t in range(len(seq)):
        lp, lm = logp.copy(), logp.copy()
        lp[t] += eps
        lm[t] -= eps
        fd = (oracle.pref_loss(kind, lp, seq, mask, 3, beta, gamma, ref=ref).loss
              - oracle.pref_loss(kind, lm, seq, mask, 3, beta, gamma, ref=ref).loss) / (2 * eps)
        assert res.g[t] == pytest.approx(fd, rel=1e-6, abs=1e-9), (kind, t)
