"""The quantised head (4/8-bit affine groups) against the oracle on the
dequantised weights, and bitwise against the bf16 path fed the same weights."""

import numpy as np
import pytest
import torch

import oracle
import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import GRAD_RELFRO, LOGP_ATOL, dev, f64, gpu_backward, gpu_forward, relfro, status_tensor, to_dev

pytestmark = pytest.mark.gpu


def quant_dev(w, bits, group):
    wq, s, b = workloads.quantize_affine(w.W, bits, group)
    Wd = oracle.dequant_affine(wq, s, b, bits, group, w.d)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    return (t(wq), t(s.view(np.int16)).view(torch.bfloat16), t(b.view(np.int16)).view(torch.bfloat16)), Wd


def run_q(t, q, bits, group, w, softcap, g=None, lse_in=None, with_dw=True):
    M, V, d = w.M, w.V, w.d
    ws = torch.empty(orpo.orpo_head_q_workspace_bytes(M, V, d), dtype=torch.uint8, device=dev())
    st = status_tensor()
    logp = torch.empty(M, device=dev())
    lse = torch.empty(M, device=dev())
    orpo.orpo_head_fwd_q(t["h"], *q, bits, group, t["targets"], t["mask"], softcap, logp, lse, ws, st)
    out = {"logp": logp, "lse": lse}
    if g is not None:
        dh = torch.empty((M, d), device=dev())
        dW = torch.empty((V, d), device=dev()) if with_dw else None
        lse_t = torch.from_numpy(np.asarray(lse_in, dtype=np.float32)).to(dev())
        orpo.orpo_head_bwd_q(t["h"], *q, bits, group, t["targets"], t["mask"], lse_t,
                             torch.from_numpy(np.asarray(g, dtype=np.float32)).to(dev()), softcap, dh, dW, False, ws,
                             st)
        out["dh"], out["dW"] = dh, dW
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out.items()}, int(st.item())


@pytest.mark.parametrize("name,bits,group", [("tiny", 4, 64), ("tiny", 8, 32), ("small", 4, 128)])
def test_quantised_head_matches_oracle(name, bits, group):
    w = workloads.make(name)
    q, Wd = quant_dev(w, bits, group)
    logp_r, lse_r, res, dh_r, dW_r = oracle.full_chain(f64(w.h), Wd, w.targets, w.mask, w.seq_id, w.n_pairs, w.lam,
                                                       w.softcap)
    out, st = run_q(to_dev(w), q, bits, group, w, w.softcap, g=res.g, lse_in=lse_r)
    assert st == 0
    assert np.max(np.abs(out["logp"] - logp_r)) < LOGP_ATOL and np.max(np.abs(out["lse"] - lse_r)) < LOGP_ATOL
    assert relfro(out["dh"], dh_r) < GRAD_RELFRO and relfro(out["dW"], dW_r) < GRAD_RELFRO


def test_quantised_backward_is_the_bf16_backward_on_the_dequantised_weights():
    w = workloads.make("small", M=900, d=256, V=5000)
    q, Wd = quant_dev(w, 4, 64)
    _, lse_r, res, _, _ = oracle.full_chain(f64(w.h), Wd, w.targets, w.mask, w.seq_id, w.n_pairs, w.lam, 0.0)
    t = to_dev(w)
    out, st = run_q(t, q, 4, 64, w, 0.0, g=res.g, lse_in=lse_r)
    w2 = workloads.make("small", M=900, d=256, V=5000)
    w2.W = workloads.round_bf16(Wd.astype(np.float32))          # exact: Wd already holds bf16 values
    dh, dW, st2 = gpu_backward(to_dev(w2), lse_r, res.g, w.M, w.V, w.d, 0.0)
    assert st == 0 and st2 == 0
    assert np.array_equal(out["dh"], dh) and np.array_equal(out["dW"], dW)
    # frozen head: dW skipped, dh unchanged
    out2, st3 = run_q(t, q, 4, 64, w, 0.0, g=res.g, lse_in=lse_r, with_dw=False)
    assert st3 == 0 and out2["dW"] is None and np.array_equal(out2["dh"], dh)


def test_blocks_dequantised_by_the_spare_warps_are_the_bf16_path_bit_for_bit():
    """At M >= 8192 every vocabulary block after the first is dequantised by the spare warps of the
    previous block's kernels while it is multiplied; the backward must still equal the bf16 backward
    fed the dequantised weights bit for bit (same blocks, same tiles), the forward the oracle."""
    w = workloads.make("small", M=8200, d=256, V=70000)
    assert w.M >= 8192
    q, Wd = quant_dev(w, 4, 64)
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, w.M - 1], rng.choice(w.M, 40, replace=False)]))
    logp_r, lse_r = oracle.head_forward(f64(w.h[rows]), Wd, w.targets[rows], w.mask[rows], 0.0)
    g = (rng.standard_normal(w.M) * 1e-3).astype(np.float32)
    w2 = workloads.make("small", M=8200, d=256, V=70000)
    w2.W = workloads.round_bf16(Wd.astype(np.float32))          # exact: Wd already holds bf16 values
    t2 = to_dev(w2)
    _, lse_in, st0 = gpu_forward(t2, w.M, w.V, w.d, 0.0)          # any lse serves a bitwise comparison
    t = to_dev(w)
    out, st = run_q(t, q, 4, 64, w, 0.0, g=g, lse_in=lse_in)
    assert st0 == 0 and st == 0
    assert np.max(np.abs(out["logp"][rows] - logp_r)) < LOGP_ATOL and np.max(np.abs(out["lse"][rows] - lse_r)) < LOGP_ATOL
    dh, dW, st2 = gpu_backward(t2, lse_in, g, w.M, w.V, w.d, 0.0)
    assert st2 == 0
    assert np.array_equal(out["dh"], dh) and np.array_equal(out["dW"], dW)


def test_quantised_head_with_split_dh_matches_oracle():
    """M 512 (the pages' batch size), d 256: the dh GEMM splits each tile's K range (65536 columns)
    over several SMs, here on the dequantised weights, with one dequantisation launch per block."""
    w = workloads.make("e4b", M=512, d=256, V=65536)
    q, Wd = quant_dev(w, 4, 64)
    logp_r, lse_r, res, dh_r, dW_r = oracle.full_chain(f64(w.h), Wd, w.targets, w.mask, w.seq_id, w.n_pairs, w.lam,
                                                       w.softcap)
    out, st = run_q(to_dev(w), q, 4, 64, w, w.softcap, g=res.g, lse_in=lse_r)
    assert st == 0
    assert np.max(np.abs(out["logp"] - logp_r)) < LOGP_ATOL and np.max(np.abs(out["lse"] - lse_r)) < LOGP_ATOL
    assert relfro(out["dh"], dh_r) < GRAD_RELFRO and relfro(out["dW"], dW_r) < GRAD_RELFRO
    out2, st2 = run_q(to_dev(w), q, 4, 64, w, w.softcap, g=res.g, lse_in=lse_r, with_dw=False)
    assert st2 == 0 and np.array_equal(out2["dh"], out["dh"])


def test_quantised_e4b_full_size_several_blocks():
    w = workloads.make("e4b")
    q, Wd = quant_dev(w, 4, 64)
    t = to_dev(w)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, w.M - 1], rng.choice(w.M, 30, replace=False)]))
    logp_r, lse_r = oracle.head_forward(f64(w.h[rows]), Wd, w.targets[rows], w.mask[rows], w.softcap)
    g = np.zeros(w.M, dtype=np.float32)
    g[rows] = (rng.standard_normal(len(rows)) * 1e-3).astype(np.float32)
    lse_in = np.zeros(w.M, dtype=np.float32)
    lse_in[rows] = lse_r
    out, st = run_q(t, q, 4, 64, w, w.softcap, g=g, lse_in=lse_in)
    assert st == 0
    assert np.max(np.abs(out["logp"][rows] - logp_r)) < LOGP_ATOL
    assert np.max(np.abs(out["lse"][rows] - lse_r)) < LOGP_ATOL
    rdh_rows, rdW = oracle.head_backward(f64(w.h[rows]), Wd, w.targets[rows], w.mask[rows], lse_in[rows], g[rows],
                                         w.softcap)
    rdh = np.zeros((w.M, w.d))
    rdh[rows] = rdh_rows
    assert relfro(out["dh"], rdh) < GRAD_RELFRO and relfro(out["dW"], rdW) < GRAD_RELFRO
