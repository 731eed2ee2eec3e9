"""Metamorphic checks of the whole chain (forward, loss, backward) on the GPU: rows that carry no
supervision (mask 0, sequence id -1) may be inserted anywhere, and the batch split differently into
row tiles, without changing the loss, the per-sequence means, the gradient of any real row, or dW
beyond fp32 reordering."""

import dataclasses

import numpy as np
import pytest
import torch

import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import relfro, to_dev

pytestmark = pytest.mark.gpu


def run_chain(w):
    t = to_dev(w)
    head = orpo.OrpoHead(w.M, w.V, w.d, w.n_pairs)
    head.step(t["h"].view(torch.bfloat16), t["W"].view(torch.bfloat16), t["targets"], t["mask"], t["seq_id"],
              w.softcap, w.lam)
    torch.cuda.synchronize()
    assert int(head.status.item()) == 0
    return {k: getattr(head, k).detach().cpu().numpy().copy() for k in ("logp", "lse", "out", "ell", "g", "dh", "dW")}


@pytest.mark.parametrize("name,kw", [("small", {}), ("e4b", dict(M=4096, d=256, V=65536 + 320))])
def test_unsupervised_rows_inserted_anywhere_change_nothing(name, kw):
    w = workloads.make(name, **kw)
    rng = np.random.default_rng(21)
    n_pad = 333
    at = np.sort(rng.integers(0, w.M + 1, size=n_pad))           # insertion points, repeats allowed
    pad_h = rng.integers(0, 1 << 16, size=(n_pad, w.d), dtype=np.uint64).astype(np.uint16)
    pad_h = (pad_h & np.uint16(0x3FFF)) | np.uint16(0x3C00)        # finite bf16 bits of moderate size
    ins = lambda a, v: np.insert(a, at, v, axis=0)
    wp = dataclasses.replace(
        w, h=ins(w.h, pad_h), targets=ins(w.targets, rng.integers(0, w.V, size=n_pad).astype(np.int32)),
        mask=ins(w.mask, np.zeros(n_pad, np.uint8)), seq_id=ins(w.seq_id, np.full(n_pad, -1, np.int32)))
    a, b = run_chain(w), run_chain(wp)
    real = np.ones(wp.M, dtype=bool)
    real[at + np.arange(n_pad)] = False                             # positions of the inserted rows
    assert real.sum() == w.M
    assert np.max(np.abs(b["logp"][real] - a["logp"])) < 1e-5
    assert np.max(np.abs(b["lse"][real] - a["lse"])) < 1e-5
    assert np.all(b["logp"][~real] == 0) and np.all(b["g"][~real] == 0) and np.all(b["dh"][~real] == 0)
    assert np.allclose(b["out"], a["out"], rtol=1e-5, atol=1e-7)
    assert np.allclose(b["ell"], a["ell"], rtol=1e-6, atol=1e-7)
    assert np.allclose(b["g"][real], a["g"], rtol=1e-5, atol=1e-12)
    assert relfro(b["dh"][real], a["dh"]) < 1e-4
    assert relfro(b["dW"], a["dW"]) < 1e-4
