"""orpo_pref_loss (ORPO, SimPO, DPO, IPO, hinge) against the float64 oracle on
synthetic per-token logp and reference sums, at every workload's row layout."""

import numpy as np
import pytest
import torch

import oracle
import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import LOSS_RTOL, dev, status_tensor

pytestmark = pytest.mark.gpu


def run(kind, logp, seq, mask, P, beta, gamma, ref):
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).astype(dt)).to(dev())
    out = torch.full((5,), float("nan"), device=dev())
    ell = torch.empty(2 * P, device=dev())
    g = torch.full((len(seq),), float("nan"), device=dev())
    st = status_tensor()
    orpo.orpo_pref_loss(kind, t(logp, np.float32), t(seq, np.int32), t(mask, np.uint8), P, beta, gamma,
                        None if ref is None else t(ref, np.float32), out, ell, g, st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ell.cpu().numpy(), g.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("kind", ["orpo", "simpo", "dpo", "ipo", "hinge"])
@pytest.mark.parametrize("name", ["tiny", "small", "ragged"])
def test_matches_oracle(kind, name):
    w = workloads.make(name, d=8, V=16)
    logp = workloads.synthetic_logp(5, w.seq_id, w.mask, scale=0.5, offset=-1.0)
    rng = np.random.default_rng(3)
    # reference sums near the policy's own sums, so the log-ratio D is O(1)
    sums = np.bincount(w.seq_id[(w.seq_id >= 0) & (w.mask == 1)],
                       weights=logp[(w.seq_id >= 0) & (w.mask == 1)].astype(np.float64), minlength=2 * w.n_pairs)
    ref = (sums + rng.standard_normal(2 * w.n_pairs)).astype(np.float32)
    beta, gamma = (0.1, 0.0) if kind == "orpo" else (0.5, 0.2)
    use_ref = ref if kind in ("dpo", "ipo", "hinge") else None
    out, ell, g, st = run(kind, logp, w.seq_id, w.mask, w.n_pairs, beta, gamma, use_ref)
    assert st == 0
    r = oracle.pref_loss(kind, logp.astype(np.float64), w.seq_id, w.mask, w.n_pairs, beta, gamma,
                         ref=None if use_ref is None else use_ref.astype(np.float64))
    want = np.array([r.loss, r.nll, r.orr if kind != "orpo" else r.orr, r.accuracy, r.margin])
    for a, b in zip(out, want):
        assert abs(a - b) <= LOSS_RTOL * max(abs(b), 1e-6), (kind, out, want)
    assert np.allclose(ell, r.ell, rtol=1e-6, atol=1e-6)
    assert np.allclose(g, r.g, rtol=1e-5, atol=1e-12)


def test_dpo_policy_equal_reference_gives_log2_on_gpu():
    seq = np.repeat(np.arange(8), 5).astype(np.int32)
    mask = np.ones(len(seq), dtype=np.uint8)
    logp = workloads.synthetic_logp(1, seq, mask)
    ref = np.bincount(seq, weights=logp.astype(np.float64)).astype(np.float32)
    out, _, g, st = run("dpo", logp, seq, mask, 4, 0.3, 0.0, ref)
    assert st == 0 and abs(out[0] - np.log(2.0)) < 1e-6 and abs(out[4]) < 1e-5


@pytest.mark.parametrize("name", ["tiny", "small", "ragged"])
def test_orpo_full_scope_matches_oracle(name):
    w = workloads.make(name, d=8, V=16)
    mask = w.mask.copy()
    rng = np.random.default_rng(8)
    # turn the first rows of every sequence into supervised prompt rows (mask 2)
    for s in range(2 * w.n_pairs):
        rows = np.where(w.seq_id == s)[0]
        k = int(rng.integers(0, max(1, len(rows) // 3)))
        mask[rows[:k]] = 2
        mask[rows[-1]] = 1
    logp = workloads.synthetic_logp(6, w.seq_id, mask, scale=0.5, offset=-1.0)
    out, ell, g, st = run("orpo_full", logp, w.seq_id, mask, w.n_pairs, 0.1, 0.0, None)
    assert st == 0
    r = oracle.orpo_loss(logp.astype(np.float64), w.seq_id, mask, w.n_pairs, 0.1, scope="full")
    for a, b in zip(out, r.metrics()):
        assert abs(a - b) <= LOSS_RTOL * max(abs(b), 1e-6), (out, r.metrics())
    assert np.allclose(ell, r.ell, rtol=1e-6, atol=1e-6)
    assert np.allclose(g, r.g, rtol=1e-5, atol=1e-12)
    # response scope on the same mask: prompt rows carry no gradient
    out2, _, g2, st2 = run("orpo", logp, w.seq_id, mask, w.n_pairs, 0.1, 0.0, None)
    r2 = oracle.orpo_loss(logp.astype(np.float64), w.seq_id, mask, w.n_pairs, 0.1)
    assert st2 == 0 and np.allclose(g2, r2.g, rtol=1e-5, atol=1e-12) and np.all(g2[mask == 2] == 0)
