"""Pins for the quantised head's weight definition in the oracle: hand-worked
values, nibble order, rounding against torch's bf16 conversion, and a fully
independent dequantisation through torch integer and float ops."""

import numpy as np
import pytest
import torch

import oracle
import workloads


def bf(x):
    return workloads.round_bf16(np.asarray(x, dtype=np.float32))


def test_hand_values_and_nibble_order():
    # one row, d = 8, group 8: q = 0..7 packed two per byte, low nibble = even column
    wq = np.array([[0x10, 0x32, 0x54, 0x76]], dtype=np.uint8)
    W = oracle.dequant_affine(wq, bf([[0.5]]), bf([[-1.0]]), 4, 8, 8)
    assert list(W[0]) == [-1.0, -0.5, 0.0, 0.5, 1.0, 1.5, 2.0, 2.5]
    W8 = oracle.dequant_affine(np.array([[0, 255, 3, 4]], dtype=np.uint8), bf([[0.25]]), bf([[2.0]]), 8, 4, 4)
    # 255 * 0.25 + 2 = 65.75 lies halfway between bf16 neighbours 65.5 and 66: nearest even is 66
    assert list(W8[0]) == [2.0, 66.0, 2.75, 3.0]


def test_single_rounding_to_bf16_matches_torch():
    # scale = 1 + 2^-7, q = 3: 3.0234375 is a tie between two bf16 values; nearest even wins
    s = np.float32(1 + 2 ** -7)
    W = oracle.dequant_affine(np.array([[3]], dtype=np.uint8), bf([[s]]), bf([[0.0]]), 8, 1, 1)
    ref = torch.tensor([3.0234375], dtype=torch.float32).to(torch.bfloat16).float().item()
    assert W[0, 0] == ref == 3.03125


@pytest.mark.parametrize("bits,group", [(4, 32), (4, 64), (8, 64)])
def test_matches_independent_torch_dequantisation(bits, group):
    w = workloads.make("tiny", d=128, V=96)
    wq, s, b = workloads.quantize_affine(w.W, bits, group)
    ours = oracle.dequant_affine(wq, s, b, bits, group, 128)
    t = torch.from_numpy(wq.astype(np.int32))
    q = torch.stack([t & 15, t >> 4], dim=2).reshape(96, 128) if bits == 4 else t
    st = torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).float().repeat_interleave(group, dim=1)
    bt = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().repeat_interleave(group, dim=1)
    ref = torch.addcmul(bt, st, q.float()).to(torch.bfloat16).double().numpy()
    assert np.array_equal(ours, ref)
    # the quantiser itself is faithful: every weight within half a step of its original
    Wt = workloads.bf16_to_f32(w.W).astype(np.float64)
    step = np.repeat(workloads.bf16_to_f32(s).astype(np.float64), group, axis=1)
    assert np.all(np.abs(ours - Wt) <= 0.51 * step + 1e-2 * np.abs(Wt))
