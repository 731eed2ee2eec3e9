"""Pins for the backward skips in the oracle (coefficient filter and block maxima).

The skips are defined on the pages in words only ("Steel flash-CCE — handoff" §E;
"Training — design" §5.1, the Apple-CCE skips with eps 1e-5): a block of the
backward coefficient that lies wholly below eps is skipped, and the forward's
per-block logit maxima let the backward skip cold (token block, vocabulary block)
programs.  These pins fix the oracle's reading of that on inputs whose logits are
known in closed form (an orthonormal head), by an error bound that any correct
filter obeys, and by the two limits of eps.
"""

import math

import numpy as np
import pytest

import oracle
import workloads


def _onehot_head(a, y, V):
    """W = I (V x V) and h_t = a_t e_{y_t}: z[t, v] = a_t [v == y_t] exactly."""
    W = np.eye(V)
    h = np.zeros((len(y), V))
    h[np.arange(len(y)), y] = a
    return h, W


def test_filter_closed_form_orthonormal_head():
    V, a = 16, 5.0
    y = np.array([1, 6, 6, 13, 2, 9])
    g = np.array([0.3, -0.2, 0.0, 0.5, 0.1, -0.4])
    mask = np.ones(6, dtype=np.uint8)
    h, W = _onehot_head(np.full(6, a), y, V)
    lse = np.full(6, math.log(math.exp(a) + V - 1))
    p_y = math.exp(a) / (math.exp(a) + V - 1)
    p_o = 1.0 / (math.exp(a) + V - 1)
    eps = 1e-2
    assert p_o < eps <= 1 - p_y          # off-target coefficients are below eps, target ones are not
    tile = (2, 4)
    # kept tiles, from where the targets of rows with g != 0 fall (row 2 has g = 0: its
    # target must not keep tile (1, 1) alive)
    kept = set()
    for t in range(6):
        if g[t] != 0:
            kept.add((t // 2, y[t] // 4))
    assert kept == {(0, 0), (0, 1), (1, 3), (2, 0), (2, 2)}
    dZ = np.zeros((6, V))
    for t in range(6):
        for v in range(V):
            if (t // 2, v // 4) in kept:
                dZ[t, v] = g[t] * ((1.0 if v == y[t] else 0.0) - (p_y if v == y[t] else p_o))
    dh_exp = dZ                                   # W = I
    dW_exp = np.zeros((V, V))
    for t in range(6):
        dW_exp[:, y[t]] += a * dZ[t]              # dW = dZ^T h, h_t = a e_{y_t}
    dh, dW = oracle.head_backward(h, W, y, mask, lse, g, 0.0, filter_eps=eps, tile=tile)
    np.testing.assert_allclose(dh, dh_exp, rtol=0, atol=1e-15)
    np.testing.assert_allclose(dW, dW_exp, rtol=0, atol=1e-14)
    # eps above the target coefficient 1 - p_y drops every tile
    dh2, dW2 = oracle.head_backward(h, W, y, mask, lse, g, 0.0, filter_eps=0.1, tile=tile)
    assert 1 - p_y < 0.1
    assert not dh2.any() and not dW2.any()
    # the threshold sits exactly at the off-target coefficient p_o: just below it every tile
    # of an active row is kept, just above it only the target tiles are
    dh3, _ = oracle.head_backward(h, W, y, mask, lse, g, 0.0, filter_eps=p_o * (1 - 1e-9), tile=tile)
    full = g[:, None] * (np.eye(V)[y] - np.where(np.eye(V)[y] > 0, p_y, p_o))
    np.testing.assert_allclose(dh3, full, rtol=0, atol=1e-15)
    dh4, _ = oracle.head_backward(h, W, y, mask, lse, g, 0.0, filter_eps=p_o * (1 + 1e-9), tile=tile)
    np.testing.assert_allclose(dh4, dh_exp, rtol=0, atol=1e-15)


def test_filter_limits_of_eps():
    w = workloads.make("tiny", M=96, d=64, V=700)
    h, W = oracle.bf16_bits_to_f64(w.h), oracle.bf16_bits_to_f64(w.W)
    g = np.random.default_rng(3).standard_normal(w.M) * w.mask
    lse = oracle.head_forward(h, W, w.targets, w.mask)[1]
    dh0, dW0 = oracle.head_backward(h, W, w.targets, w.mask, lse, g)
    # no coefficient of an active row is exactly 0, so a vanishing eps keeps everything
    dh1, dW1 = oracle.head_backward(h, W, w.targets, w.mask, lse, g, filter_eps=1e-300)
    assert np.array_equal(dh0, dh1) and np.array_equal(dW0, dW1)
    # |onehot - p| <= 1 and sech^2 <= 1: eps = 2 drops every tile
    dh2, dW2 = oracle.head_backward(h, W, w.targets, w.mask, lse, g, 30.0, filter_eps=2.0)
    assert not dh2.any() and not dW2.any()


@pytest.mark.parametrize("softcap", [0.0, 30.0])
def test_filter_error_bound(softcap):
    # every dropped entry has |coefficient| < eps, so per row
    #   |dh_t - dh~_t| <= |g_t| eps sum_v |W_v|  and per head row  |dW_v - dW~_v| <= eps sum_t |g_t| |h_t|
    w = workloads.make("tiny", M=150, d=64, V=900)
    h, W = oracle.bf16_bits_to_f64(w.h) * 2.0, oracle.bf16_bits_to_f64(w.W)
    g = np.random.default_rng(5).standard_normal(w.M) * w.mask
    lse = oracle.head_forward(h, W, w.targets, w.mask, softcap)[1]
    eps, tile = 3e-3, (4, 16)
    dh0, dW0 = oracle.head_backward(h, W, w.targets, w.mask, lse, g, softcap)
    dh1, dW1 = oracle.head_backward(h, W, w.targets, w.mask, lse, g, softcap, filter_eps=eps, tile=tile)
    assert not np.array_equal(dh0, dh1)          # the filter drops something here
    bound_h = np.abs(g) * eps * np.linalg.norm(W, axis=1).sum()
    assert np.all(np.linalg.norm(dh0 - dh1, axis=1) <= bound_h + 1e-15)
    bound_w = eps * (np.abs(g) * np.linalg.norm(h, axis=1)).sum()
    assert np.all(np.linalg.norm(dW0 - dW1, axis=1) <= bound_w + 1e-15)
    # and the filtered gradient is still close in the relative Frobenius sense
    assert np.linalg.norm(dh0 - dh1) / np.linalg.norm(dh0) < 0.05


@pytest.mark.parametrize("softcap", [0.0, 4.0])
def test_block_max_closed_form(softcap):
    V, M = 14, 5                                   # ragged: last tile 2 columns, last group 1 row
    y = np.array([1, 6, 12, 3, 13])
    a = np.array([2.0, -3.0, 1.5, 7.0, 0.5])
    mask = np.array([1, 1, 0, 2, 1], dtype=np.uint8)   # row 2 unsupervised; row 3 a prompt row
    h, W = _onehot_head(a, y, V)
    bm = oracle.head_block_max(h, W, mask, softcap, group=(2, 4))
    assert bm.shape == (3, 4)
    zt = lambda x: softcap * math.tanh(x / softcap) if softcap > 0 else x
    exp = np.full((3, 4), -np.inf)
    for q in range(3):
        for j in range(4):
            for t in range(2 * q, min(M, 2 * q + 2)):
                if mask[t] == 0:
                    continue
                cols = range(4 * j, min(V, 4 * j + 4))
                # every tile has a column other than y_t, where z = 0
                m = max(zt(a[t]) if y[t] in cols else 0.0, 0.0)
                exp[q, j] = max(exp[q, j], m / math.log(2))
    np.testing.assert_allclose(bm, exp, rtol=0, atol=1e-14)


def test_block_max_bounds_the_softmax():
    # p[t, v] <= 2^(blockmax[q(t), j(v)] - lse_t log2 e) for every supervised row: the block skip's test
    w = workloads.make("tiny", M=100, d=64, V=600)
    h, W = oracle.bf16_bits_to_f64(w.h), oracle.bf16_bits_to_f64(w.W)
    lse = oracle.head_forward(h, W, w.targets, w.mask, 30.0)[1]
    bm = oracle.head_block_max(h, W, w.mask, 30.0)
    z = oracle.softcap_value(h @ W.T, 30.0)
    p = np.exp(z - lse[:, None])
    q = np.arange(w.M) // oracle.GROUP_ROWS
    j = np.arange(w.V) // oracle.TILE_COLS
    bound = np.exp2(bm[q][:, j] - lse[:, None] / math.log(2))
    rows = w.mask != 0
    assert np.all(p[rows] <= bound[rows] * (1 + 1e-12))


@pytest.mark.parametrize("eps", [0.0, 3e-3])
def test_vocab_slices_reassemble_the_whole(eps):
    # dW is separable over vocabulary rows and dh over columns: the slices add up to the whole
    w = workloads.make("tiny", M=70, d=32, V=600)
    h, W = oracle.bf16_bits_to_f64(w.h), oracle.bf16_bits_to_f64(w.W)
    g = np.random.default_rng(7).standard_normal(w.M) * w.mask
    lse = oracle.head_forward(h, W, w.targets, w.mask, 30.0)[1]
    tile = (8, 32)
    dh, dW = oracle.head_backward(h, W, w.targets, w.mask, lse, g, 30.0, filter_eps=eps, tile=tile)
    parts = [oracle.head_backward(h, W, w.targets, w.mask, lse, g, 30.0, filter_eps=eps, tile=tile, vocab=(c, min(600, c + 256)))
             for c in range(0, 600, 256)]
    np.testing.assert_allclose(sum(p[0] for p in parts), dh, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(np.concatenate([p[1] for p in parts]), dW, rtol=1e-12, atol=1e-15)
    with pytest.raises(oracle.OracleError):
        oracle.head_backward(h, W, w.targets, w.mask, lse, g, 30.0, tile=tile, vocab=(16, 64))
