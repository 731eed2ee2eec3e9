"""Forward parity (logp, lse) against the float64 oracle, element by element."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import LOGP_ATOL, f64, gpu_forward, status_tensor, to_dev, workspace

pytestmark = pytest.mark.gpu


def check(w, softcap=None):
    softcap = w.softcap if softcap is None else softcap
    t = to_dev(w)
    logp, lse, st = gpu_forward(t, w.M, w.V, w.d, softcap)
    assert st == 0
    rl, rs = oracle.head_forward(f64(w.h), f64(w.W), w.targets, w.mask, softcap)
    assert np.all(np.isfinite(logp)) and np.all(np.isfinite(lse))
    assert np.max(np.abs(lse - rs)) < LOGP_ATOL
    assert np.max(np.abs(logp - rl)) < LOGP_ATOL
    assert np.all(logp[w.mask == 0] == 0)


def test_tiny():
    check(workloads.make("tiny"))


def test_tiny_with_softcap():
    check(workloads.make("tiny"), softcap=3.0)


def test_small():
    check(workloads.make("small"))


@pytest.mark.parametrize("M,V,d", [(1, 256, 64), (127, 1000, 72), (129, 4096 + 64, 136), (300, 513, 256),
                                   (640, 2304, 520)])
def test_ragged_shapes(M, V, d):
    w = workloads.make("tiny", M=M + 64, d=d, V=V)
    # trim to exactly M rows (keeps the recipe's prompt mask where present)
    w.h, w.targets, w.mask, w.seq_id = w.h[:M], w.targets[:M], w.mask[:M], w.seq_id[:M]
    w.mask[0] = 1
    assert w.M == M
    check(w)
    check(w, softcap=30.0)


def test_peaked_e4b_rows_reduced():
    # the e4b recipe (peaked h, softcap 30) at a reduced vocabulary and row count
    check(workloads.make("e4b", M=512, d=256, V=8192))


def test_target_out_of_range_is_flagged():
    w = workloads.make("tiny", M=128, d=64, V=512)
    w.targets = w.targets.copy()
    w.targets[10] = w.V + 5
    w.mask[10] = 1
    w.targets[11] = -7
    w.mask[11] = 0            # prompt row: never read, no error from it alone
    t = to_dev(w)
    logp, lse, st = gpu_forward(t, w.M, w.V, w.d, 0.0)
    assert st & (1 << 4)
    assert logp[10] == 0.0


def test_deterministic():
    w = workloads.make("tiny")
    t = to_dev(w)
    a = gpu_forward(t, w.M, w.V, w.d, 0.0)
    b = gpu_forward(t, w.M, w.V, w.d, 0.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_rows_agree_whatever_the_batch_around_them():
    # The same 128 rows alone (one row tile: many vocabulary splits), at the front of an 8192-row
    # batch (64 row tiles in pairs: few splits) and at its ragged end: the split count, the pairing,
    # the unit order and the rows' tile position all change, and only the fp32 merge order differs.
    w = workloads.make("e4b", M=8192, d=256, V=65536 + 320)
    t = to_dev(w)
    sub = slice(0, 128)

    def rows_of(idx):
        u = {k: (v if k == "W" else v[idx].contiguous()) for k, v in t.items()}
        M = u["targets"].shape[0]
        return gpu_forward(u, M, w.V, w.d, w.softcap)

    perm = torch.cat([torch.arange(128, 8192 - 5, device=t["h"].device), torch.arange(0, 128, device=t["h"].device),
                      torch.arange(8192 - 5, 8192, device=t["h"].device)])
    alone = rows_of(torch.arange(0, 128, device=t["h"].device))
    front = rows_of(torch.arange(0, 8192, device=t["h"].device))
    back = rows_of(perm)          # the 128 rows sit at 8059..8186, across a tile boundary
    assert alone[2] == front[2] == back[2] == 0
    pos = slice(8192 - 5 - 128, 8192 - 5)
    for got in ((front[0][sub], front[1][sub]), (back[0][pos], back[1][pos])):
        assert np.max(np.abs(got[0] - alone[0])) < 1e-4
        assert np.max(np.abs(got[1] - alone[1])) < 1e-4
    rl, rs = oracle.head_forward(f64(w.h[sub]), f64(w.W), w.targets[sub], w.mask[sub], w.softcap)
    assert np.max(np.abs(alone[1] - rs)) < LOGP_ATOL
    assert np.max(np.abs(alone[0] - rl)) < LOGP_ATOL
