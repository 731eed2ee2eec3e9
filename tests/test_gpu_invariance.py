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


def test_vocabulary_permutation_moves_only_dW_rows():
    # relabel the vocabulary: W'[j] = W[perm[j]], y' = perm^-1[y].  Every logit is the same number in
    # another column, so logp, lse, the loss and dh stay put (to fp32 reordering of the sums) and
    # dW'[j] = dW[perm[j]]; a wrong column offset in any split or vocabulary block would show here
    w = workloads.make("e4b", M=2048, d=128, V=65536 + 320)
    perm = np.random.default_rng(8).permutation(w.V)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(w.V)
    wp = dataclasses.replace(w, W=np.ascontiguousarray(w.W[perm]), targets=inv[w.targets].astype(np.int32))
    a, b = run_chain(w), run_chain(wp)
    assert np.max(np.abs(b["logp"] - a["logp"])) < 1e-5
    assert np.max(np.abs(b["lse"] - a["lse"])) < 1e-5
    assert np.allclose(b["out"], a["out"], rtol=1e-5, atol=1e-7)
    assert relfro(b["dh"], a["dh"]) < 1e-4
    assert relfro(b["dW"], a["dW"][perm]) < 1e-4


def test_pair_order_moves_only_rows():
    # reorder the pairs (rows of each sequence move with it, ids relabelled in the new order): the loss
    # is a mean over pairs and dW a sum over rows, so both stay put; per-row outputs move with the rows
    w = workloads.make("small")
    P = w.n_pairs
    sigma = np.random.default_rng(4).permutation(P)
    order, new_sid = [], []
    for q, p in enumerate(sigma):
        for k in (0, 1):
            rows = np.where(w.seq_id == 2 * p + k)[0]
            order.append(rows)
            new_sid.append(np.full(len(rows), 2 * q + k, np.int32))
    pad = np.where(w.seq_id < 0)[0]
    order = np.concatenate(order + [pad])
    new_sid = np.concatenate(new_sid + [np.full(len(pad), -1, np.int32)])
    assert len(order) == w.M
    wp = dataclasses.replace(w, h=np.ascontiguousarray(w.h[order]), targets=w.targets[order],
                             mask=w.mask[order], seq_id=new_sid)
    a, b = run_chain(w), run_chain(wp)
    assert np.max(np.abs(b["logp"] - a["logp"][order])) < 1e-5
    assert np.allclose(b["out"], a["out"], rtol=1e-5, atol=1e-7)
    ell_new = a["ell"].reshape(P, 2)[sigma].reshape(-1)
    assert np.allclose(b["ell"], ell_new, rtol=1e-6, atol=1e-7)
    assert np.allclose(b["g"], a["g"][order], rtol=1e-5, atol=1e-12)
    assert relfro(b["dh"], a["dh"][order]) < 1e-4
    assert relfro(b["dW"], a["dW"]) < 1e-4
