"""The seeded input generator: shapes, structure, determinism and bf16 rounding."""

import numpy as np
import torch

import workloads


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 3
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0]   # ties to even
    ours = workloads.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_tiny_structure_and_determinism():
    a = workloads.make("tiny")
    b = workloads.make("tiny")
    assert a.M == 256 and a.d == 256 and a.V == 4096 and a.n_pairs == 2
    assert np.array_equal(a.h, b.h) and np.array_equal(a.W, b.W)
    assert np.array_equal(a.targets, b.targets)
    # first 8 rows of each 64-row sequence are prompt rows
    for s in range(4):
        rows = np.where(a.seq_id == s)[0]
        assert len(rows) == 64 and a.mask[rows[:8]].sum() == 0 and a.mask[rows[8:]].all()
    std = workloads.bf16_to_f32(a.W).std()
    assert abs(std - (4.0 / 256) ** 0.5) < 0.01


def test_chunked_draw_is_thread_independent(monkeypatch):
    n = workloads.CHUNK * 3 + 17
    a = workloads.normal_bf16(1, 4, (n,), 1.0)
    monkeypatch.setattr(workloads, "_threads", lambda: 1)
    b = workloads.normal_bf16(1, 4, (n,), 1.0)
    assert np.array_equal(a, b)


def test_ragged_padding_and_small_lengths():
    w = workloads.make("ragged", M=4000, d=64, V=512)
    assert w.M % 128 == 0
    pad = w.seq_id < 0
    assert np.all(w.mask[pad] == 0)
    ids = w.seq_id[~pad]
    assert np.all(np.diff(ids) >= 0) and ids.max() == 2 * w.n_pairs - 1
    s = workloads.make("small", M=512, d=64, V=300)
    assert s.n_pairs == 8 and s.M == len(s.seq_id)


def test_zipf_targets_are_skewed():
    w = workloads.make("largev", M=2048, d=32, V=1000)
    counts = np.bincount(w.targets, minlength=1000)
    assert counts[0] > counts[10] > counts[500]
