"""Parity at the full workload sizes (e4b, large-vocab, ragged), in the launch
configuration the benchmark times.

Forward: every row is computed on the GPU; a seeded sample of rows (including
the first, the last and ragged-tail rows) is compared with the oracle.
Backward: the cotangent g is nonzero on a seeded sample of rows only, so the
oracle computes ALL of dh and dW exactly from those rows; the GPU runs its full
backward over every row and vocabulary block.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import GRAD_RELFRO, LOGP_ATOL, f64, gpu_backward, gpu_forward, relfro, to_dev

pytestmark = pytest.mark.gpu

NAMES = ["e4b", "largev", "ragged"]


@pytest.fixture(scope="module", params=NAMES)
def full(request):
    w = workloads.make(request.param)
    t = to_dev(w)
    W64 = f64(w.W)
    rng = np.random.default_rng(123)
    resp = np.where(w.mask == 1)[0]
    rows = np.unique(np.concatenate([[0, w.M - 1, resp[-1]], rng.choice(w.M, 45, replace=False),
                                     rng.choice(resp, 16, replace=False)]))
    yield w, t, W64, rows
    del t
    torch.cuda.empty_cache()


def test_forward_sampled_rows(full):
    w, t, W64, rows = full
    logp, lse, st = gpu_forward(t, w.M, w.V, w.d, w.softcap)
    assert st == 0
    assert np.all(np.isfinite(lse))
    rl, rs = oracle.head_forward(f64(w.h[rows]), W64, w.targets[rows], w.mask[rows], w.softcap)
    assert np.max(np.abs(lse[rows] - rs)) < LOGP_ATOL
    assert np.max(np.abs(logp[rows] - rl)) < LOGP_ATOL
    assert np.all(logp[w.mask == 0] == 0)


def test_backward_restricted_support(full):
    w, t, W64, rows = full
    rows = rows[w.mask[rows] == 1][:48]
    rng = np.random.default_rng(7)
    g = np.zeros(w.M, dtype=np.float32)
    g[rows] = (rng.standard_normal(len(rows)) * 1e-3).astype(np.float32)
    h_rows = f64(w.h[rows])
    _, lse_rows = oracle.head_forward(h_rows, W64, w.targets[rows], w.mask[rows], w.softcap)
    lse = np.zeros(w.M, dtype=np.float32)
    lse[rows] = lse_rows.astype(np.float32)
    dh, dW, st = gpu_backward(t, lse, g, w.M, w.V, w.d, w.softcap)
    assert st == 0
    rdh_rows, rdW = oracle.head_backward(h_rows, W64, w.targets[rows], w.mask[rows], lse[rows], g[rows],
                                         w.softcap)
    rdh = np.zeros((w.M, w.d))
    rdh[rows] = rdh_rows
    assert relfro(dh, rdh) < GRAD_RELFRO
    assert relfro(dW, rdW) < GRAD_RELFRO
    other = np.ones(w.M, dtype=bool)
    other[rows] = False
    assert np.all(dh[other] == 0)


@pytest.mark.parametrize("d", [1600, 1544])
def test_multiblock_ragged_vocab_and_hidden(d):
    """M 20000 (two row blocks of 10240 rows), V 50257 (four vocabulary blocks of 12800 columns, the
    last ragged); d 1544 is not a multiple of 64, so the MN-major operands take the 2-D-box path."""
    w = workloads.make("small", M=20000, d=d, V=50257)
    t = to_dev(w)
    W64 = f64(w.W)
    rng = np.random.default_rng(31)
    rows = np.unique(np.concatenate([[0, w.M - 1, 10239, 10240], rng.choice(w.M, 36, replace=False)]))
    logp, lse, st = gpu_forward(t, w.M, w.V, w.d, 0.0)
    assert st == 0
    rl, rs = oracle.head_forward(f64(w.h[rows]), W64, w.targets[rows], w.mask[rows], 0.0)
    assert np.max(np.abs(lse[rows] - rs)) < LOGP_ATOL and np.max(np.abs(logp[rows] - rl)) < LOGP_ATOL
    g = np.zeros(w.M, dtype=np.float32)
    g[rows] = (rng.standard_normal(len(rows)) * 1e-3).astype(np.float32)
    lse_in = np.zeros(w.M, dtype=np.float32)
    lse_in[rows] = rs.astype(np.float32)
    dh, dW, st = gpu_backward(t, lse_in, g, w.M, w.V, w.d, 0.0)
    assert st == 0
    rdh_rows, rdW = oracle.head_backward(f64(w.h[rows]), W64, w.targets[rows], w.mask[rows], lse_in[rows], g[rows],
                                         0.0)
    rdh = np.zeros((w.M, w.d))
    rdh[rows] = rdh_rows
    assert relfro(dh, rdh) < GRAD_RELFRO and relfro(dW, rdW) < GRAD_RELFRO
