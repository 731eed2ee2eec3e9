"""Split K of the dh GEMM (few rows, long vocabulary blocks) against the oracle.

With M 1024 the dh class has 8 row tiles of 128 rows (4 cluster units), each
contracting over a vocabulary block of about 87k columns, so the kernel cuts every
tile's K range into parts that run on different SMs; the part that finishes last
sums all parts in part order.  V 262151 makes three vocabulary blocks of equal
width (87552 columns, the last 87047): the first split and stored, the others
split and reduce-added onto it.  d 136 leaves most of each 256-column tile
outside the output.
"""

import numpy as np
import pytest
import torch

import oracle
import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import (GRAD_RELFRO, LOGP_ATOL, LOSS_RTOL, dev, f64, gpu_backward, relfro, status_tensor, to_dev,
                         workspace)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def case():
    w = workloads.make("e4b", M=1024, d=136, V=262151)
    logp, lse, res, dh, dW = oracle.full_chain(f64(w.h), f64(w.W), w.targets, w.mask, w.seq_id, w.n_pairs, w.lam,
                                               w.softcap)
    return w, to_dev(w), lse, res, dh, dW


def test_chain_with_split_dh_matches_oracle(case):
    w, t, lse_r, res, dh_r, dW_r = case
    M, P = w.M, w.n_pairs
    logp = torch.empty(M, dtype=torch.float32, device=dev())
    lse = torch.empty(M, dtype=torch.float32, device=dev())
    out = torch.empty(5, dtype=torch.float32, device=dev())
    ell = torch.empty(2 * P, dtype=torch.float32, device=dev())
    g = torch.empty(M, dtype=torch.float32, device=dev())
    dh = torch.full((M, w.d), float("nan"), dtype=torch.float32, device=dev())
    dW = torch.full((w.V, w.d), float("nan"), dtype=torch.float32, device=dev())
    ws = workspace(M, w.V, w.d)
    st = status_tensor()
    orpo.orpo_head_fwd(t["h"], t["W"], t["targets"], t["mask"], w.softcap, logp, lse, ws, st)
    orpo.orpo_loss(logp, t["seq_id"], t["mask"], P, w.lam, out, ell, g, st)
    orpo.orpo_head_bwd(t["h"], t["W"], t["targets"], t["mask"], lse, g, w.softcap, dh, dW, False, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.max(np.abs(lse.cpu().numpy() - lse_r)) < LOGP_ATOL
    assert abs(float(out[0].item()) - res.loss) <= LOSS_RTOL * abs(res.loss)
    dh, dW = dh.cpu().numpy(), dW.cpu().numpy()
    assert relfro(dh, dh_r) < GRAD_RELFRO and relfro(dW, dW_r) < GRAD_RELFRO
    row_err = np.linalg.norm(dh - dh_r, axis=1) / np.linalg.norm(dh_r, axis=1)
    assert np.max(row_err) < 2e-2


def test_split_dh_is_bitwise_reproducible_and_frozen_head_agrees(case):
    w, t, lse_r, res, _, _ = case
    a = gpu_backward(t, lse_r, res.g, w.M, w.V, w.d, w.softcap)
    b = gpu_backward(t, lse_r, res.g, w.M, w.V, w.d, w.softcap)
    assert a[2] == 0 and b[2] == 0
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # frozen head (no dW class in the launch): the same dh, bit for bit
    dh = torch.full((w.M, w.d), float("nan"), dtype=torch.float32, device=dev())
    st = status_tensor()
    orpo.orpo_head_bwd(t["h"], t["W"], t["targets"], t["mask"],
                       torch.from_numpy(np.asarray(lse_r, dtype=np.float32)).to(dev()),
                       torch.from_numpy(np.asarray(res.g, dtype=np.float32)).to(dev()), w.softcap, dh, None, False,
                       workspace(w.M, w.V, w.d), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and np.array_equal(dh.cpu().numpy(), a[0])
