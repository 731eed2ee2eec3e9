"""orpo_head_fwd_static: the forward for callers that cannot allocate device
memory (for example a plugin hook that receives only its input and output
buffers, or a service that forbids cudaMalloc after start-up).  Its split
partials live in a fixed array inside the library instead of a caller
workspace.  Checked through the C ABI against orpo_head_fwd, twice in a row
(the array keeps the previous call's contents between calls).

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""

import numpy as np
import pytest
import torch

import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import LOGP_ATOL, dev, status_tensor, to_dev, workspace

pytestmark = pytest.mark.gpu


def _run_static(t, M):
    logp = torch.full((M,), float("nan"), dtype=torch.float32, device=dev())
    lse = torch.full((M,), float("nan"), dtype=torch.float32, device=dev())
    st = status_tensor()
    return logp, lse, st


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("e4b", dict(M=2048, d=512, V=32768))])
def test_static_forward_matches_workspace_forward_twice(name, kw):
    w = workloads.make(name, **kw)
    t = to_dev(w)
    ref_logp = torch.empty(w.M, dtype=torch.float32, device=dev())
    ref_lse = torch.empty(w.M, dtype=torch.float32, device=dev())
    ref_st = status_tensor()
    orpo.orpo_head_fwd(t["h"], t["W"], t["targets"], t["mask"], w.softcap, ref_logp, ref_lse,
                       workspace(w.M, w.V, w.d), ref_st)
    for _ in range(2):
        logp, lse, st = _run_static(t, w.M)
        orpo.orpo_head_fwd_static(t["h"], t["W"], t["targets"], t["mask"], w.softcap, logp, lse, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and int(ref_st.item()) == 0
        assert np.max(np.abs(logp.cpu().numpy() - ref_logp.cpu().numpy())) < LOGP_ATOL
        assert np.max(np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy())) < LOGP_ATOL


@pytest.mark.parametrize("M,V", [(65536, 50257), (60000, 8192)])
def test_static_forward_at_its_row_limit_matches_oracle(M, V):
    """At these sizes the fixed array holds fewer vocabulary splits than the workspace forward picks
    (8 against 18 and 32), so the split count is capped; M = 65536 is the largest M accepted.  Sampled
    rows, the last ones included, are compared with the float64 oracle, and every row with the
    workspace forward."""
    import oracle
    from gpu_helpers import f64

    w = workloads.make("tiny", M=M, d=64, V=V)
    assert w.M == M
    t = to_dev(w)
    ref_logp = torch.empty(M, dtype=torch.float32, device=dev())
    ref_lse = torch.empty(M, dtype=torch.float32, device=dev())
    ref_st = status_tensor()
    orpo.orpo_head_fwd(t["h"], t["W"], t["targets"], t["mask"], w.softcap, ref_logp, ref_lse,
                       workspace(M, V, w.d), ref_st)
    logp, lse, st = _run_static(t, M)
    orpo.orpo_head_fwd_static(t["h"], t["W"], t["targets"], t["mask"], w.softcap, logp, lse, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(ref_st.item()) == 0
    logp, lse = logp.cpu().numpy(), lse.cpu().numpy()
    assert np.max(np.abs(logp - ref_logp.cpu().numpy())) < LOGP_ATOL
    assert np.max(np.abs(lse - ref_lse.cpu().numpy())) < LOGP_ATOL
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.arange(4), np.arange(M - 130, M), rng.choice(M, 120, replace=False)]))
    rl, rs = oracle.head_forward(f64(w.h[rows]), f64(w.W), w.targets[rows], w.mask[rows], w.softcap)
    assert np.max(np.abs(lse[rows] - rs)) < LOGP_ATOL
    assert np.max(np.abs(logp[rows] - rl)) < LOGP_ATOL


def test_static_forward_rejects_rows_beyond_its_fixed_scratch():
    lib = orpo.load()
    M = orpo.FWD_STATIC_MAX_ROWS + 1
    fake = torch.empty(16, dtype=torch.uint8, device=dev())
    p = fake.data_ptr()
    rc = lib.orpo_head_fwd_static(p, p, p, p, M, 1024, 64, 0.0, p, p, p, None)
    assert rc == 8  # ORPO_ERR_TOO_LARGE, nothing launched
    assert "ORPO_FWD_STATIC_MAX_ROWS" in orpo.orpo_status_string(rc)
