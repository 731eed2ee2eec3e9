"""Dense-cotangent backward across several row and vocabulary blocks.

The whole chain (forward, ORPO loss, backward) runs on the GPU through the C
ABI, on a batch with two row blocks (M 19968 > 16384 rows per block: two of
9984) and four vocabulary blocks with a ragged last one (V 50257: three of 12800
columns and one of 11857).  The cotangent is the ORPO loss gradient itself, so
every response row carries a nonzero g and every bf16 dZ block is dense: each dh
tile is the reduce-add of four vocabulary blocks and each dW tile of two row
blocks.  The float64 oracle
runs the same chain on the same bf16 inputs ("Training — design" §2: the parity
ladder against a plain reference, with a non-uniform cotangent).

Checked: dh and dW to the 1e-2 relative Frobenius bar; every row of dh to 2e-2
of its own norm (a row computed in the wrong block, or a block added twice,
fails here even when the global norm hides it); dW's largest entry error to
1e-2 of its largest entry.
"""

import numpy as np
import pytest
import torch

import oracle
import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import GRAD_RELFRO, LOGP_ATOL, LOSS_RTOL, dev, f64, relfro, status_tensor, to_dev, workspace

pytestmark = pytest.mark.gpu

M_ROWS, D, V = 20000, 136, 50257


@pytest.fixture(scope="module", params=[30.0, 0.0], ids=["softcap30", "nocap"])
def chain(request):
    softcap = request.param
    w = workloads.make("e4b", M=M_ROWS, d=D, V=V)  # 39 pairs x 2 x 256 rows = 19968, peaked h
    M, P = w.M, w.n_pairs
    t = to_dev(w)
    logp = torch.empty(M, dtype=torch.float32, device=dev())
    lse = torch.empty(M, dtype=torch.float32, device=dev())
    out = torch.empty(5, dtype=torch.float32, device=dev())
    ell = torch.empty(2 * P, dtype=torch.float32, device=dev())
    g = torch.empty(M, dtype=torch.float32, device=dev())
    dh = torch.full((M, D), float("nan"), dtype=torch.float32, device=dev())
    dW = torch.full((V, D), float("nan"), dtype=torch.float32, device=dev())
    ws = workspace(M, V, D)
    st = status_tensor()
    orpo.orpo_head_fwd(t["h"], t["W"], t["targets"], t["mask"], softcap, logp, lse, ws, st)
    orpo.orpo_loss(logp, t["seq_id"], t["mask"], P, w.lam, out, ell, g, st)
    orpo.orpo_head_bwd(t["h"], t["W"], t["targets"], t["mask"], lse, g, softcap, dh, dW, False, ws, st)
    torch.cuda.synchronize()
    gpu = dict(status=int(st.item()), logp=logp.cpu().numpy(), lse=lse.cpu().numpy(), loss=float(out[0].item()),
               g=g.cpu().numpy(), dh=dh.cpu().numpy(), dW=dW.cpu().numpy())
    del t, ws, dh, dW
    torch.cuda.empty_cache()
    ref = oracle.full_chain(f64(w.h), f64(w.W), w.targets, w.mask, w.seq_id, P, w.lam, softcap)
    return w, gpu, ref


def test_shape_spans_several_blocks(chain):
    w, _, _ = chain
    assert w.M > 16384 and w.M <= 2 * 16384          # two row blocks
    assert 3 * 12800 < V < 4 * 12800                  # four vocabulary blocks, the last ragged
    assert np.all(w.mask == 1)                        # every row a response row: g dense


def test_forward_and_loss(chain):
    w, gpu, (logp, lse, res, _, _) = chain
    assert gpu["status"] == 0
    assert np.max(np.abs(gpu["lse"] - lse)) < LOGP_ATOL
    assert np.max(np.abs(gpu["logp"] - logp)) < LOGP_ATOL
    assert abs(gpu["loss"] - res.loss) <= LOSS_RTOL * abs(res.loss)
    assert np.count_nonzero(gpu["g"]) == w.M


def test_dense_dh_every_row(chain):
    _, gpu, (_, _, _, dh, _) = chain
    assert relfro(gpu["dh"], dh) < GRAD_RELFRO
    row_err = np.linalg.norm(gpu["dh"] - dh, axis=1) / np.linalg.norm(dh, axis=1)
    assert np.max(row_err) < 2e-2, int(np.argmax(row_err))


def test_dense_dW_every_block(chain):
    _, gpu, (_, _, _, _, dW) = chain
    assert relfro(gpu["dW"], dW) < GRAD_RELFRO
    assert np.max(np.abs(gpu["dW"] - dW)) <= 1e-2 * np.max(np.abs(dW))
    for v0 in range(0, V, 12800):  # each vocabulary block on its own
        blk = slice(v0, min(V, v0 + 12800))
        assert relfro(gpu["dW"][blk], dW[blk]) < GRAD_RELFRO, v0
