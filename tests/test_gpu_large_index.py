"""Row indices past 2^24 and element offsets past 2^31: M = 2^24 + 333 rows of d = 136, so h and dh
hold more than 2^31 elements, with a ragged V = 300 and the softcap on.  Forward, loss and backward
run over every row; the oracle checks seeded sample rows (the last rows among them), the whole loss
and gradient g, and all of dh and dW for a cotangent supported on sampled rows.  Inputs are drawn on
the device from a seeded generator and the sampled rows copied back for the oracle.  A vocabulary
of 2^20 + 37 columns checks the other extreme: the most forward splits and a ragged last tile."""

import numpy as np
import pytest
import torch

import oracle
import orpo_preference_loss_gb300 as orpo
from gpu_helpers import GRAD_RELFRO, LOGP_ATOL, LOSS_RTOL, dev, relfro

pytestmark = pytest.mark.gpu

M, D, V, P = (1 << 24) + 333, 136, 300, 2048
SOFTCAP, LAM = 30.0, 0.1


def bits(x):
    return x.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module")
def big():
    g = torch.Generator(device=dev()).manual_seed(2024)
    h = torch.empty((M, D), dtype=torch.bfloat16, device=dev())
    for r0 in range(0, M, 1 << 22):  # bounded fp32 temporaries
        r1 = min(M, r0 + (1 << 22))
        h[r0:r1] = torch.randn((r1 - r0, D), generator=g, device=dev()).to(torch.bfloat16)
    W = (torch.randn((V, D), generator=g, device=dev()) * (2.0 / D ** 0.5)).to(torch.bfloat16)
    targets = torch.randint(0, V, (M,), generator=g, device=dev(), dtype=torch.int32)
    mask = torch.ones(M, dtype=torch.uint8, device=dev())
    mask[::977] = 0                                   # unsupervised rows inside the sequences
    seq_id = (torch.arange(M, device=dev(), dtype=torch.int64) * (2 * P) // M).to(torch.int32)
    ws = torch.empty(orpo.orpo_head_workspace_bytes(M, V, D), dtype=torch.uint8, device=dev())
    rng = np.random.default_rng(5)
    edge = [0, (1 << 24) - 1, 1 << 24, (1 << 31) // D - 1, (1 << 31) // D, M - 129, M - 2, M - 1]
    rows = np.unique(np.concatenate([edge, rng.choice(M, 24, replace=False)]))
    yield dict(h=h, W=W, targets=targets, mask=mask, seq_id=seq_id, ws=ws, rows=rows,
               W64=oracle.bf16_bits_to_f64(bits(W)))
    torch.cuda.empty_cache()


def test_forward_and_loss_past_32_bit_offsets(big):
    b = big
    logp = torch.full((M,), float("nan"), device=dev())
    lse = torch.full((M,), float("nan"), device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    orpo.orpo_head_fwd(b["h"], b["W"], b["targets"], b["mask"], SOFTCAP, logp, lse, b["ws"], st)
    out = torch.empty(5, device=dev())
    ell = torch.empty(2 * P, device=dev())
    gl = torch.full((M,), float("nan"), device=dev())
    orpo.orpo_loss(logp, b["seq_id"], b["mask"], P, LAM, out, ell, gl, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, orpo.orpo_status_string(int(st.item()))
    assert bool(torch.isfinite(lse).all())
    assert bool((logp[b["mask"] == 0] == 0).all())

    rows = b["rows"]
    rt = torch.from_numpy(rows).to(dev())
    tg, mk = b["targets"][rt].cpu().numpy(), b["mask"][rt].cpu().numpy()
    rl, rs = oracle.head_forward(oracle.bf16_bits_to_f64(bits(b["h"][rt])), b["W64"], tg, mk, SOFTCAP)
    assert np.max(np.abs(lse[rt].cpu().numpy() - rs)) < LOGP_ATOL
    assert np.max(np.abs(logp[rt].cpu().numpy() - rl)) < LOGP_ATOL

    # the loss over all 2^24 rows, on the GPU's own logp
    lp, sq, mm = logp.cpu().numpy(), b["seq_id"].cpu().numpy(), b["mask"].cpu().numpy()
    res = oracle.orpo_loss(lp, sq, mm, P, LAM)
    o = out.cpu().numpy()
    assert abs(o[0] - res.loss) <= LOSS_RTOL * abs(res.loss)
    gg = gl.cpu().numpy()
    assert np.max(np.abs(gg - res.g)) <= 1e-5 * np.max(np.abs(res.g))


def test_backward_past_32_bit_offsets(big):
    b = big
    rows = b["rows"]
    mk_rows = b["mask"][torch.from_numpy(rows).to(dev())].cpu().numpy()
    rows = rows[mk_rows == 1]
    rt = torch.from_numpy(rows).to(dev())
    h_rows = oracle.bf16_bits_to_f64(bits(b["h"][rt]))
    tg = b["targets"][rt].cpu().numpy()
    ones = np.ones(len(rows), dtype=np.uint8)
    _, lse_rows = oracle.head_forward(h_rows, b["W64"], tg, ones, SOFTCAP)
    gv = (np.random.default_rng(9).standard_normal(len(rows)) * 1e-3).astype(np.float32)
    lse = torch.zeros(M, device=dev())
    g = torch.zeros(M, device=dev())
    lse[rt] = torch.from_numpy(lse_rows.astype(np.float32)).to(dev())
    g[rt] = torch.from_numpy(gv).to(dev())
    dh = torch.full((M, D), float("nan"), device=dev())
    dW = torch.full((V, D), float("nan"), device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    orpo.orpo_head_bwd(b["h"], b["W"], b["targets"], b["mask"], lse, g, SOFTCAP, dh, dW, False, b["ws"], st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, orpo.orpo_status_string(int(st.item()))

    rdh, rdW = oracle.head_backward(h_rows, b["W64"], tg, ones, lse_rows.astype(np.float32), gv, SOFTCAP)
    assert relfro(dh[rt].cpu().numpy(), rdh) < GRAD_RELFRO
    assert relfro(dW.cpu().numpy(), rdW) < GRAD_RELFRO
    # every other row of dh, the last ones included, is exactly zero (and was written)
    nz = torch.nonzero(dh.abs().amax(dim=1) != 0).flatten().cpu().numpy()
    assert set(nz.tolist()) <= set(rows.tolist())
    assert bool(torch.isfinite(dh).all())


def test_vocabulary_past_2_20_with_a_ragged_tail():
    # V = 2^20 + 37 at small M: the forward runs its most splits with many tiles each, and the
    # backward's vocabulary blocks end in a 37-column tile; every row is checked, and dh and dW
    # exactly for a cotangent on a few rows
    Mv, Dv, Vv, cap = 256, 64, (1 << 20) + 37, 30.0
    g = torch.Generator(device=dev()).manual_seed(7)
    h = torch.randn((Mv, Dv), generator=g, device=dev()).to(torch.bfloat16)
    W = (torch.randn((Vv, Dv), generator=g, device=dev()) * (2.0 / Dv ** 0.5)).to(torch.bfloat16)
    tg = torch.randint(0, Vv, (Mv,), generator=g, device=dev(), dtype=torch.int32)
    tg[:4] = torch.tensor([Vv - 1, Vv - 37, Vv - 38, 0], dtype=torch.int32)  # targets in and next to the tail
    mk = torch.ones(Mv, dtype=torch.uint8, device=dev())
    ws = torch.empty(orpo.orpo_head_workspace_bytes(Mv, Vv, Dv), dtype=torch.uint8, device=dev())
    logp = torch.empty(Mv, device=dev())
    lse = torch.empty(Mv, device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    orpo.orpo_head_fwd(h, W, tg, mk, cap, logp, lse, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    h64, W64 = oracle.bf16_bits_to_f64(bits(h)), oracle.bf16_bits_to_f64(bits(W))
    tgn, mkn = tg.cpu().numpy(), mk.cpu().numpy()
    rl, rs = oracle.head_forward(h64, W64, tgn, mkn, cap)
    assert np.max(np.abs(lse.cpu().numpy() - rs)) < LOGP_ATOL
    assert np.max(np.abs(logp.cpu().numpy() - rl)) < LOGP_ATOL

    rows = np.array([0, 1, 2, 3, 100, 255])
    gv = np.zeros(Mv, dtype=np.float32)
    gv[rows] = (np.random.default_rng(3).standard_normal(len(rows)) * 1e-3).astype(np.float32)
    dh = torch.full((Mv, Dv), float("nan"), device=dev())
    dW = torch.full((Vv, Dv), float("nan"), device=dev())
    orpo.orpo_head_bwd(h, W, tg, mk, lse, torch.from_numpy(gv).to(dev()), cap, dh, dW, False, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    lse_n = lse.cpu().numpy()
    rdh, rdW = oracle.head_backward(h64[rows], W64, tgn[rows], mkn[rows], lse_n[rows], gv[rows], cap)
    assert relfro(dh.cpu().numpy()[rows], rdh) < GRAD_RELFRO
    assert relfro(dW.cpu().numpy(), rdW) < GRAD_RELFRO
    other = np.ones(Mv, dtype=bool)
    other[rows] = False
    assert np.all(dh.cpu().numpy()[other] == 0)
