"""Failure detection on the GPU without a fault: a bounded on-chip wait that
runs out reports ORPO_STATUS_TIMEOUT through the status word, the kernel
returns, and the context keeps working; data errors are reported, not trapped."""

import time

import numpy as np
import pytest
import torch

import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import LOGP_ATOL, gpu_forward, status_tensor, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    st = status_tensor()
    t0 = time.perf_counter()
    orpo.orpo_debug_wait_timeout(st, 50_000_000)      # 50 ms on a barrier nothing completes
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) & orpo.STATUS_BITS["timeout"]
    assert 0.04 < dt < 5.0
    # the context is intact: a normal forward still runs and is correct
    w = workloads.make("tiny")
    a = gpu_forward(to_dev(w), w.M, w.V, w.d, 0.0)
    assert a[2] == 0 and np.all(np.isfinite(a[1]))


def test_nan_hidden_state_is_reported_not_trapped():
    w = workloads.make("tiny")
    w.h = w.h.copy()
    w.h[5, :] = 0x7FC0          # bf16 NaN in one row
    logp, lse, st = gpu_forward(to_dev(w), w.M, w.V, w.d, 0.0)
    assert st & orpo.STATUS_BITS["nonfinite"]
    ok = np.ones(w.M, dtype=bool)
    ok[5] = False
    assert np.all(np.isfinite(lse[ok]))
