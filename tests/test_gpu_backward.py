"""Backward parity (dh, dW) and the whole forward -> loss -> backward chain
against the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import (GRAD_RELFRO, LOGP_ATOL, LOSS_RTOL, dev, f64, gpu_backward, gpu_forward, gpu_loss,
                         relfro, to_dev)

pytestmark = pytest.mark.gpu


def oracle_chain(w, softcap=None):
    c = w.softcap if softcap is None else softcap
    return oracle.full_chain(f64(w.h), f64(w.W), w.targets, w.mask, w.seq_id, w.n_pairs, w.lam, c)


def check_backward_given(w, lse, g, softcap, **kw):
    """Backward alone: both sides get the same lse and g (from the oracle)."""
    t = to_dev(w)
    dh, dW, st = gpu_backward(t, lse, g, w.M, w.V, w.d, softcap, **kw)
    assert st == 0
    rdh, rdW = oracle.head_backward(f64(w.h), f64(w.W), w.targets, w.mask, lse.astype(np.float32), g.astype(
        np.float32), softcap)
    return dh, dW, rdh, rdW


@pytest.mark.parametrize("name,softcap", [("tiny", None), ("tiny", 30.0), ("small", None)])
def test_backward_with_oracle_lse_and_g(name, softcap):
    w = workloads.make(name)
    c = w.softcap if softcap is None else softcap
    logp, lse, res, _, _ = oracle_chain(w, c)
    dh, dW, rdh, rdW = check_backward_given(w, lse, res.g, c)
    assert relfro(dh, rdh) < GRAD_RELFRO
    assert relfro(dW, rdW) < GRAD_RELFRO
    assert np.all(dh[w.mask == 0] == 0)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_full_chain(name):
    w = workloads.make(name)
    logp_r, lse_r, res, dh_r, dW_r = oracle_chain(w)
    t = to_dev(w)
    logp, lse, st = gpu_forward(t, w.M, w.V, w.d, w.softcap)
    assert st == 0
    assert np.max(np.abs(logp - logp_r)) < LOGP_ATOL and np.max(np.abs(lse - lse_r)) < LOGP_ATOL
    lt = torch.from_numpy(logp).to(dev())
    out, ell, g, st = gpu_loss(lt, t["seq_id"], t["mask"], w.n_pairs, w.lam)
    assert st == 0
    assert abs(out[0] - res.loss) <= LOSS_RTOL * abs(res.loss)
    dh, dW, st = gpu_backward(t, lse, g, w.M, w.V, w.d, w.softcap)
    assert st == 0
    assert relfro(dh, dh_r) < GRAD_RELFRO
    assert relfro(dW, dW_r) < GRAD_RELFRO


@pytest.mark.parametrize("M,V,d", [(1, 256, 64), (127, 1000, 72), (129, 4160, 136), (300, 513, 256)])
def test_ragged_shapes(M, V, d):
    w = workloads.make("tiny", M=M + 64, d=d, V=V)
    w.h, w.targets, w.mask, w.seq_id = w.h[:M], w.targets[:M], w.mask[:M], w.seq_id[:M]
    w.mask[0] = 1
    assert w.M == M
    rng = np.random.default_rng(M + V + d)
    g = (rng.standard_normal(M) * 0.01).astype(np.float32)
    for c in (0.0, 30.0):
        _, lse = oracle.head_forward(f64(w.h), f64(w.W), w.targets, w.mask, c)
        dh, dW, rdh, rdW = check_backward_given(w, lse, g, c)
        assert relfro(dh, rdh) < GRAD_RELFRO and relfro(dW, rdW) < GRAD_RELFRO


def test_accumulate_dw():
    w = workloads.make("tiny")
    logp, lse, res, dh_r, dW_r = oracle_chain(w)
    base = np.random.default_rng(1).standard_normal(dW_r.shape).astype(np.float32) * 1e-3
    dh, dW, rdh, rdW = check_backward_given(w, lse, res.g, w.softcap, dW_init=base, accumulate=True)
    assert relfro(dW - base, rdW) < GRAD_RELFRO
    assert relfro(dh, rdh) < GRAD_RELFRO


def test_backward_is_bitwise_reproducible():
    w = workloads.make("small")
    _, lse, res, _, _ = oracle_chain(w)
    t = to_dev(w)
    a = gpu_backward(t, lse, res.g, w.M, w.V, w.d, w.softcap)
    b = gpu_backward(t, lse, res.g, w.M, w.V, w.d, w.softcap)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_zero_rows_give_zero_gradient():
    w = workloads.make("tiny")
    _, lse, _, _, _ = oracle_chain(w)
    g = np.zeros(w.M, dtype=np.float32)
    t = to_dev(w)
    dh, dW, st = gpu_backward(t, lse, g, w.M, w.V, w.d, w.softcap)
    assert st == 0 and np.all(dh == 0) and np.all(dW == 0)


def test_full_scope_chain():
    """sft_scope = full: prompt rows (mask 2) go through the head and the NLL."""
    w = workloads.make("tiny")
    mask = w.mask.copy()
    mask[mask == 0] = 2          # the recipe's 8 prompt rows per sequence become supervised prompt rows
    w.mask = mask
    logp_r, lse_r, res, dh_r, dW_r = oracle.full_chain(f64(w.h), f64(w.W), w.targets, mask, w.seq_id, w.n_pairs,
                                                       w.lam, w.softcap, scope="full")
    t = to_dev(w)
    logp, lse, st = gpu_forward(t, w.M, w.V, w.d, w.softcap)
    assert st == 0 and np.max(np.abs(logp - logp_r)) < LOGP_ATOL
    import orpo_preference_loss_gb300 as orpo
    out = torch.empty(5, device=dev())
    ell = torch.empty(2 * w.n_pairs, device=dev())
    g = torch.empty(w.M, device=dev())
    stt = torch.zeros(1, dtype=torch.int32, device=dev())
    orpo.orpo_pref_loss("orpo_full", torch.from_numpy(logp).to(dev()), t["seq_id"], t["mask"], w.n_pairs, w.lam,
                        0.0, None, out, ell, g, stt)
    torch.cuda.synchronize()
    assert int(stt.item()) == 0
    assert abs(float(out[0]) - res.loss) <= LOSS_RTOL * abs(res.loss)
    dh, dW, st = gpu_backward(t, lse, g.cpu().numpy(), w.M, w.V, w.d, w.softcap)
    assert st == 0
    assert relfro(dh, dh_r) < GRAD_RELFRO and relfro(dW, dW_r) < GRAD_RELFRO
    assert np.abs(dh[mask == 2]).sum() > 0      # prompt rows of chosen sequences carry gradient now
