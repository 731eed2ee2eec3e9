"""Backward skips on the GPU ("Steel flash-CCE — handoff" §E; "Training — design" §5.1):
the forward's block maxima against the oracle, the coefficient filter against the
oracle's filtered gradient, the block skip (which must leave the filtered result
unchanged, bit for bit), the limits of eps, and multi-block runs checked on sampled
row and vocabulary tiles."""

import numpy as np
import pytest
import torch

import oracle
import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import GRAD_RELFRO, LOGP_ATOL, dev, f64, gpu_backward, gpu_forward, relfro, status_tensor, \
    to_dev, workspace

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634


def fwd_bmax(t, M, V, d, softcap):
    logp = torch.full((M,), float("nan"), dtype=torch.float32, device=dev())
    lse = torch.full((M,), float("nan"), dtype=torch.float32, device=dev())
    bm = torch.full(orpo.block_max_shape(M, V), float("nan"), dtype=torch.float32, device=dev())
    st = status_tensor()
    orpo.orpo_head_fwd_bmax(t["h"], t["W"], t["targets"], t["mask"], softcap, logp, lse, bm, workspace(M, V, d), st)
    torch.cuda.synchronize()
    return logp.cpu().numpy(), lse.cpu().numpy(), bm, int(st.item())


def bwd_skip(t, lse_np, g_np, bm, eps, M, V, d, softcap, dW_init=None, accumulate=False, with_dW=True):
    lse = torch.from_numpy(np.asarray(lse_np, dtype=np.float32)).to(dev())
    g = torch.from_numpy(np.asarray(g_np, dtype=np.float32)).to(dev())
    dh = torch.full((M, d), float("nan"), dtype=torch.float32, device=dev())
    dW = None
    if with_dW:
        dW = (torch.full((V, d), float("nan"), dtype=torch.float32, device=dev()) if dW_init is None
              else torch.from_numpy(np.asarray(dW_init, dtype=np.float32)).to(dev()))
    st = status_tensor()
    orpo.orpo_head_bwd_skip(t["h"], t["W"], t["targets"], t["mask"], lse, g, bm, eps, softcap, dh, dW, accumulate,
                            workspace(M, V, d), st)
    torch.cuda.synchronize()
    return dh.cpu().numpy(), (dW.cpu().numpy() if with_dW else None), int(st.item())


def orpo_g(w, logp):
    return oracle.orpo_loss(logp, w.seq_id, w.mask, w.n_pairs, w.lam).g


@pytest.mark.parametrize("name,M,V,d,softcap", [("tiny", 300, 1000, 72, 0.0), ("e4b_sharp", 384, 4196, 128, 30.0),
                                                ("tiny", 97, 300, 64, 30.0)])
def test_block_max_matches_oracle(name, M, V, d, softcap):
    w = workloads.make(name, M=M, d=d, V=V)
    if w.M > 64:
        w.mask[32:64] = 0                      # a whole 32-row group unsupervised: -inf
    t = to_dev(w)
    logp, lse, bm, st = fwd_bmax(t, w.M, w.V, w.d, softcap)
    assert st == 0
    ref = oracle.head_block_max(f64(w.h), f64(w.W), w.mask, softcap)
    got = bm.cpu().numpy()
    assert got.shape == ref.shape
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    assert np.max(np.abs(got[fin] - ref[fin])) < LOGP_ATOL * LOG2E
    # the same logp / lse as the plain forward, bit for bit
    logp0, lse0, st0 = gpu_forward(t, w.M, w.V, w.d, softcap)
    assert st0 == 0 and np.array_equal(logp, logp0) and np.array_equal(lse, lse0)


# Inputs where the filter matters and the gradient stays well conditioned in fp32: with the sharp
# recipe uncapped, 1 - p(target) falls to ~2e-5 and the fp32 logits' rounding alone moves the target
# coefficient g (1 - p) by several percent, filter or not.
@pytest.mark.parametrize("name,M,V,d,softcap,eps", [("e4b_sharp", 512, 65536, 256, 30.0, 1e-5),
                                                    ("e4b", 512, 65536, 256, 0.0, 3e-3),
                                                    ("e4b", 512, 65536, 256, 1000.0, 3e-3)])  # hybrid softcap form
def test_skip_matches_filtered_oracle(name, M, V, d, softcap, eps):
    w = workloads.make(name, M=M, d=d, V=V)
    h, W = f64(w.h), f64(w.W)
    logp_r, lse_r = oracle.head_forward(h, W, w.targets, w.mask, softcap)
    g = orpo_g(w, logp_r)
    t = to_dev(w)
    _, lse, bm, st = fwd_bmax(t, w.M, w.V, w.d, softcap)
    assert st == 0 and np.max(np.abs(lse - lse_r)) < LOGP_ATOL
    lse32, g32 = lse_r.astype(np.float32), g.astype(np.float32)
    dh, dW, st = bwd_skip(t, lse32, g32, bm, eps, w.M, w.V, w.d, softcap)
    assert st == 0
    rdh, rdW = oracle.head_backward(h, W, w.targets, w.mask, lse32, g32, softcap, filter_eps=eps)
    edh, edW = oracle.head_backward(h, W, w.targets, w.mask, lse32, g32, softcap)
    assert relfro(dh, rdh) < GRAD_RELFRO and relfro(dW, rdW) < GRAD_RELFRO
    # the inputs make the filter matter: the filtered gradient is far from the exact one, so
    # matching it means the kept and dropped tiles were chosen as the oracle chose them
    assert relfro(rdh, edh) > 3 * GRAD_RELFRO
    # the block skip changes no bit of the filtered result
    dh1, dW1, st1 = bwd_skip(t, lse32, g32, None, eps, w.M, w.V, w.d, softcap)
    assert st1 == 0 and np.array_equal(dh, dh1) and np.array_equal(dW, dW1)


def test_zero_eps_is_the_dense_backward():
    w = workloads.make("tiny")
    t = to_dev(w)
    logp, lse, bm, st = fwd_bmax(t, w.M, w.V, w.d, 30.0)
    g = orpo_g(w, logp.astype(np.float64))
    dh0, dW0, st0 = gpu_backward(t, lse, g, w.M, w.V, w.d, 30.0)
    dh1, dW1, st1 = bwd_skip(t, lse, g, bm, 0.0, w.M, w.V, w.d, 30.0)
    assert st0 == 0 and st1 == 0
    assert np.array_equal(dh0, dh1) and np.array_equal(dW0, dW1)


@pytest.mark.parametrize("use_bmax", [False, True])
def test_eps_above_every_coefficient_drops_everything(use_bmax):
    # |onehot - p| sech^2 <= 1 < 2: every tile is empty, and the first writes still store zeros
    w = workloads.make("small")
    t = to_dev(w)
    logp, lse, bm, st = fwd_bmax(t, w.M, w.V, w.d, 0.0)
    g = orpo_g(w, logp.astype(np.float64))
    dh, dW, st = bwd_skip(t, lse, g, bm if use_bmax else None, 2.0, w.M, w.V, w.d, 0.0)
    assert st == 0 and not dh.any() and not dW.any()
    init = np.random.default_rng(1).standard_normal((w.V, w.d)).astype(np.float32)
    _, dW2, st = bwd_skip(t, lse, g, bm if use_bmax else None, 2.0, w.M, w.V, w.d, 0.0, dW_init=init,
                          accumulate=True)
    assert st == 0 and np.array_equal(dW2, init)


def test_accumulate_and_frozen_head_with_skips():
    w = workloads.make("e4b_sharp", M=512, d=256, V=65536)   # about half the tiles dropped
    t = to_dev(w)
    logp, lse, bm, st = fwd_bmax(t, w.M, w.V, w.d, 30.0)
    g = orpo_g(w, logp.astype(np.float64))
    dh, dW, st = bwd_skip(t, lse, g, bm, 1e-5, w.M, w.V, w.d, 30.0)
    init = np.random.default_rng(2).standard_normal((w.V, w.d)).astype(np.float32)
    dh2, dW2, st2 = bwd_skip(t, lse, g, bm, 1e-5, w.M, w.V, w.d, 30.0, dW_init=init, accumulate=True)
    dh3, _, st3 = bwd_skip(t, lse, g, bm, 1e-5, w.M, w.V, w.d, 30.0, with_dW=False)
    assert st == st2 == st3 == 0
    assert np.array_equal(dh, dh2) and np.array_equal(dh, dh3)
    np.testing.assert_allclose(dW2, init + dW, rtol=1e-6, atol=1e-6)


def test_multiblock_skip_on_sampled_tiles():
    # 2 row blocks x 5 vocabulary blocks (blocks of 8448 x 13312: 66 row tiles, 52 vocabulary
    # tiles); sampled row tiles and vocabulary tiles against the oracle, whose filter tiles line up
    # with the library's
    w = workloads.make("e4b_sharp", M=16384 + 512, d=256, V=65536)   # about half the tiles dropped
    assert w.M == 16896
    t = to_dev(w)
    _, lse, bm, st = fwd_bmax(t, w.M, w.V, w.d, 30.0)
    assert st == 0
    rng = np.random.default_rng(4)
    g = (rng.standard_normal(w.M) * 1e-3 * (w.mask != 0)).astype(np.float32)
    eps = 1e-5
    dh, dW, st = bwd_skip(t, lse, g, bm, eps, w.M, w.V, w.d, 30.0)
    assert st == 0
    dh1, dW1, st1 = bwd_skip(t, lse, g, None, eps, w.M, w.V, w.d, 30.0)
    assert st1 == 0 and np.array_equal(dh, dh1) and np.array_equal(dW, dW1)
    h, W = f64(w.h), f64(w.W)
    for mt in (0, 65, 66, 127, w.M // 128 - 1):       # first / last tile of each row block
        r = slice(128 * mt, min(w.M, 128 * mt + 128))
        rdh, _ = oracle.head_backward(h[r], W, w.targets[r], w.mask[r], lse[r], g[r], 30.0, filter_eps=eps)
        assert relfro(dh[r], rdh) < GRAD_RELFRO
    for vt in (0, 51, 52, 255):                       # across vocabulary blocks, the last one included
        c0 = 256 * vt
        _, rdW = oracle.head_backward(h, W, w.targets, w.mask, lse, g, 30.0, filter_eps=eps, vocab=(c0, c0 + 256))
        if np.linalg.norm(rdW) == 0:
            assert not dW[c0:c0 + 256].any()
        else:
            assert relfro(dW[c0:c0 + 256], rdW) < GRAD_RELFRO


def test_plan_rounds_beyond_one_slot_area():
    # 8 row blocks x 32 vocabulary blocks = 256 blocks; at 17.25 KiB a slot, the 4 MiB skip area holds
    # 237, so the plan runs in two rounds and slots are reused
    M, d, V = 131072, 64, 262144
    w = workloads.make("e4b_sharp", M=M, d=d, V=V)
    assert w.M == M
    t = to_dev(w)
    _, lse, bm, st = fwd_bmax(t, w.M, w.V, w.d, 30.0)
    assert st == 0
    g = (np.random.default_rng(8).standard_normal(w.M) * 1e-3 * (w.mask != 0)).astype(np.float32)
    eps = 1e-5
    dh, dW, st = bwd_skip(t, lse, g, bm, eps, w.M, w.V, w.d, 30.0)
    dh1, dW1, st1 = bwd_skip(t, lse, g, None, eps, w.M, w.V, w.d, 30.0)
    assert st == 0 and st1 == 0 and np.array_equal(dh, dh1) and np.array_equal(dW, dW1)
    h, W = f64(w.h), f64(w.W)
    for mt in (0, 900, w.M // 128 - 1):               # row tiles in the first and the second round
        r = slice(128 * mt, 128 * mt + 128)
        rdh, _ = oracle.head_backward(h[r], W, w.targets[r], w.mask[r], lse[r], g[r], 30.0, filter_eps=eps)
        assert relfro(dh[r], rdh) < GRAD_RELFRO
    for vt in (0, 1023):
        c0 = 256 * vt
        _, rdW = oracle.head_backward(h, W, w.targets, w.mask, lse, g, 30.0, filter_eps=eps, vocab=(c0, c0 + 256))
        assert relfro(dW[c0:c0 + 256], rdW) < GRAD_RELFRO


def test_quantised_head_with_skips():
    # the pages' own configuration: a 4-bit head with the skips on; checked against the oracle on the
    # dequantised weights
    w = workloads.make("e4b_sharp", M=512, d=256, V=65536)
    bits, group, softcap, eps = 4, 64, 30.0, 1e-5
    wq, s, b = workloads.quantize_affine(w.W, bits, group)
    Wd = oracle.dequant_affine(wq, s, b, bits, group, w.d)
    t = to_dev(w)
    q = (torch.from_numpy(wq).to(dev()), torch.from_numpy(s.view(np.int16)).to(dev()).view(torch.bfloat16),
         torch.from_numpy(b.view(np.int16)).to(dev()).view(torch.bfloat16))
    M, V, d = w.M, w.V, w.d
    ws = torch.empty(orpo.orpo_head_q_workspace_bytes(M, V, d), dtype=torch.uint8, device=dev())
    st = status_tensor()
    logp = torch.empty(M, device=dev())
    lse = torch.empty(M, device=dev())
    bm = torch.full(orpo.block_max_shape(M, V), float("nan"), device=dev())
    orpo.orpo_head_fwd_q_bmax(t["h"], *q, bits, group, t["targets"], t["mask"], softcap, logp, lse, bm, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    h = f64(w.h)
    logp_r, lse_r = oracle.head_forward(h, Wd, w.targets, w.mask, softcap)
    assert np.max(np.abs(lse.cpu().numpy() - lse_r)) < LOGP_ATOL
    ref_bm = oracle.head_block_max(h, Wd, w.mask, softcap)
    got_bm = bm.cpu().numpy()
    fin = np.isfinite(ref_bm)
    assert np.array_equal(np.isneginf(got_bm), np.isneginf(ref_bm))
    assert np.max(np.abs(got_bm[fin] - ref_bm[fin])) < LOGP_ATOL * LOG2E
    g = orpo_g(w, logp_r).astype(np.float32)
    lse32 = lse_r.astype(np.float32)
    grads = []
    for use_bm in (True, False):
        dh = torch.empty((M, d), device=dev())
        dW = torch.empty((V, d), device=dev())
        orpo.orpo_head_bwd_q_skip(t["h"], *q, bits, group, t["targets"], t["mask"], torch.from_numpy(lse32).to(dev()),
                                  torch.from_numpy(g).to(dev()), bm if use_bm else None, eps, softcap, dh, dW, False,
                                  ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        grads.append((dh.cpu().numpy(), dW.cpu().numpy()))
    rdh, rdW = oracle.head_backward(h, Wd, w.targets, w.mask, lse32, g, softcap, filter_eps=eps)
    assert relfro(grads[0][0], rdh) < GRAD_RELFRO and relfro(grads[0][1], rdW) < GRAD_RELFRO
    assert np.array_equal(grads[0][0], grads[1][0]) and np.array_equal(grads[0][1], grads[1][1])


def test_quantised_skips_are_the_bf16_skips_on_the_dequantised_weights():
    # several dequantised blocks (2 forward W blocks of 131072 rows, 32 backward vocabulary blocks):
    # the quantised path computes the same tiles in the same order as the bf16 path fed the
    # dequantised weights, so the block maxima and the skipped backward agree bit for bit
    w = workloads.make("e4b_sharp", M=16384, d=1024, V=262144)
    bits, group, softcap, eps = 4, 64, 30.0, 1e-5
    wq, s, b = workloads.quantize_affine(w.W, bits, group)
    Wd = oracle.dequant_affine(wq, s, b, bits, group, w.d)
    M, V, d = w.M, w.V, w.d
    t = to_dev(w)
    t["W"] = torch.from_numpy(workloads.round_bf16(Wd.astype(np.float32)).view(np.int16)).to(dev()).view(torch.bfloat16)
    q = (torch.from_numpy(wq).to(dev()), torch.from_numpy(s.view(np.int16)).to(dev()).view(torch.bfloat16),
         torch.from_numpy(b.view(np.int16)).to(dev()).view(torch.bfloat16))
    assert orpo.orpo_head_q_workspace_bytes(M, V, d) < V * d * 2 + orpo.orpo_head_workspace_bytes(M, V, d)
    wsq = torch.empty(orpo.orpo_head_q_workspace_bytes(M, V, d), dtype=torch.uint8, device=dev())
    st = status_tensor()
    lse_q = torch.empty(M, device=dev())
    logp_q = torch.empty(M, device=dev())
    bm_q = torch.full(orpo.block_max_shape(M, V), float("nan"), device=dev())
    orpo.orpo_head_fwd_q_bmax(t["h"], *q, bits, group, t["targets"], t["mask"], softcap, logp_q, lse_q, bm_q, wsq, st)
    logp_b, lse_b, bm_b, st_b = fwd_bmax(t, M, V, d, softcap)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and st_b == 0
    assert np.array_equal(bm_q.cpu().numpy(), bm_b.cpu().numpy())
    assert np.max(np.abs(lse_q.cpu().numpy() - lse_b)) < 1e-4     # only the split merge order differs
    g = orpo_g(w, logp_b.astype(np.float64)).astype(np.float32)
    lse_t = torch.from_numpy(lse_b).to(dev())
    g_t = torch.from_numpy(g).to(dev())
    dh_q = torch.empty((M, d), device=dev())
    dW_q = torch.empty((V, d), device=dev())
    orpo.orpo_head_bwd_q_skip(t["h"], *q, bits, group, t["targets"], t["mask"], lse_t, g_t, bm_q, eps, softcap, dh_q,
                              dW_q, False, wsq, st)
    dh_b, dW_b, st_b = bwd_skip(t, lse_b, g, bm_b, eps, M, V, d, softcap)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and st_b == 0
    assert np.array_equal(dh_q.cpu().numpy(), dh_b) and np.array_equal(dW_q.cpu().numpy(), dW_b)
