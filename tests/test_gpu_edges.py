"""Degenerate and boundary cases of the head on the GPU, each against the oracle."""

import numpy as np
import pytest
import torch

import oracle
import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import (GRAD_RELFRO, LOGP_ATOL, dev, f64, gpu_backward, gpu_forward, relfro, status_tensor,
                         to_dev, workspace)

pytestmark = pytest.mark.gpu


def rows(w, M):
    w.h, w.targets, w.mask, w.seq_id = w.h[:M], w.targets[:M], w.mask[:M], w.seq_id[:M]
    w.mask = w.mask.copy()
    w.mask[:] = 1
    return w


@pytest.mark.parametrize("softcap", [0.0, 30.0])
def test_single_word_vocabulary(softcap):
    # V = 1: every row's only logit is its target, so logp = 0 and the gradient vanishes
    w = rows(workloads.make("tiny", M=200, d=64, V=1), 150)
    logp, lse, st = gpu_forward(to_dev(w), w.M, w.V, w.d, softcap)
    assert st == 0 and np.all(np.abs(logp) < 1e-6)
    _, rs = oracle.head_forward(f64(w.h), f64(w.W), w.targets, w.mask, softcap)
    assert np.max(np.abs(lse - rs)) < LOGP_ATOL
    g = np.full(w.M, 0.01, dtype=np.float32)
    dh, dW, st = gpu_backward(to_dev(w), lse, g, w.M, w.V, w.d, softcap)
    assert st == 0 and np.max(np.abs(dh)) < 1e-6 and np.max(np.abs(dW)) < 1e-6


def test_minimum_hidden_size_and_single_row():
    w = rows(workloads.make("tiny", M=100, d=8, V=300), 1)
    logp, lse, st = gpu_forward(to_dev(w), w.M, w.V, w.d, 0.0)
    rl, rs = oracle.head_forward(f64(w.h), f64(w.W), w.targets, w.mask, 0.0)
    assert st == 0 and abs(logp[0] - rl[0]) < LOGP_ATOL and abs(lse[0] - rs[0]) < LOGP_ATOL
    g = np.array([0.7], dtype=np.float32)
    dh, dW, st = gpu_backward(to_dev(w), rs, g, w.M, w.V, w.d, 0.0)
    rdh, rdW = oracle.head_backward(f64(w.h), f64(w.W), w.targets, w.mask, rs, g, 0.0)
    assert st == 0 and relfro(dh, rdh) < GRAD_RELFRO and relfro(dW, rdW) < GRAD_RELFRO


def test_empty_batch_backward_zeroes_or_keeps_dw():
    V, d = 512, 64
    W = torch.randn(V, d, device=dev()).to(torch.bfloat16)
    empty_i = torch.empty(0, dtype=torch.int32, device=dev())
    empty_u = torch.empty(0, dtype=torch.uint8, device=dev())
    empty_f = torch.empty(0, dtype=torch.float32, device=dev())
    h = torch.empty((0, d), dtype=torch.bfloat16, device=dev())
    dh = torch.empty((0, d), dtype=torch.float32, device=dev())
    dW = torch.full((V, d), 3.0, device=dev())
    st = status_tensor()
    ws = torch.empty(16, dtype=torch.uint8, device=dev())
    orpo.orpo_head_bwd(h, W, empty_i, empty_u, empty_f, empty_f, 0.0, dh, dW, True, ws, st)
    torch.cuda.synchronize()
    assert torch.all(dW == 3.0)                # accumulate: nothing added
    orpo.orpo_head_bwd(h, W, empty_i, empty_u, empty_f, empty_f, 0.0, dh, dW, False, ws, st)
    torch.cuda.synchronize()
    assert torch.all(dW == 0.0) and int(st.item()) == 0


@pytest.mark.parametrize("softcap", [0.5, 1e6])
def test_extreme_softcaps(softcap):
    w = workloads.make("small", M=600, d=128, V=3000)
    logp, lse, st = gpu_forward(to_dev(w), w.M, w.V, w.d, softcap)
    rl, rs = oracle.head_forward(f64(w.h), f64(w.W), w.targets, w.mask, softcap)
    assert st == 0 and np.max(np.abs(logp - rl)) < LOGP_ATOL and np.max(np.abs(lse - rs)) < LOGP_ATOL
    g = np.random.default_rng(1).standard_normal(w.M).astype(np.float32) * 1e-2
    dh, dW, st = gpu_backward(to_dev(w), rs, g, w.M, w.V, w.d, softcap)
    rdh, rdW = oracle.head_backward(f64(w.h), f64(w.W), w.targets, w.mask, rs.astype(np.float32), g, softcap)
    assert st == 0 and relfro(dh, rdh) < GRAD_RELFRO and relfro(dW, rdW) < GRAD_RELFRO


def test_lambda_zero_chain_is_chosen_cross_entropy():
    w = workloads.make("small", M=700, d=256, V=5000)
    w.lam = 0.0
    logp_r, lse_r, res, dh_r, dW_r = oracle.full_chain(f64(w.h), f64(w.W), w.targets, w.mask, w.seq_id,
                                                       w.n_pairs, 0.0, 0.0)
    head = orpo.OrpoHead(w.M, w.V, w.d, w.n_pairs, device=dev())
    t = to_dev(w)
    out = head.step(t["h"], t["W"], t["targets"], t["mask"], t["seq_id"], 0.0, 0.0)
    torch.cuda.synchronize()
    assert int(head.status.item()) == 0
    assert abs(float(out[0]) - res.loss) <= 1e-4 * abs(res.loss)
    g = head.g.cpu().numpy()
    assert np.all(g[w.seq_id % 2 == 1] == 0)        # rejected responses get no gradient at lambda = 0
    assert relfro(head.dh.cpu().numpy(), dh_r) < GRAD_RELFRO and relfro(head.dW.cpu().numpy(), dW_r) < GRAD_RELFRO
