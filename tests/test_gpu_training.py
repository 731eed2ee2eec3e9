"""A short training run: h and W are fp32 parameters, each step feeds their bf16 rounding to the
head, and plain gradient descent applies the returned dh and dW.  The GPU run and the float64
oracle's own run (its own gradients and parameters from the same start) must give finite,
decreasing losses that agree step by step."""

import numpy as np
import pytest
import torch

import oracle
import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import dev

pytestmark = pytest.mark.gpu

STEPS = 8
LR_H, LR_W = 1.0, 1.0


def bf16_round(x32):
    """bf16 bit patterns (nearest even) of a float32 array, and their exact float64 values."""
    bits = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return bits, oracle.bf16_bits_to_f64(bits)


@pytest.mark.parametrize("name,softcap", [("tiny", None), ("tiny", 30.0)])
def test_gradient_descent_tracks_the_oracle(name, softcap):
    w = workloads.make(name)
    cap = w.softcap if softcap is None else softcap
    h0 = oracle.bf16_bits_to_f64(w.h).astype(np.float32)
    W0 = oracle.bf16_bits_to_f64(w.W).astype(np.float32)
    M, V, d, P = w.M, w.V, w.d, w.n_pairs
    head = orpo.OrpoHead(M, V, d, P)
    tg = torch.from_numpy(w.targets).to(dev())
    mk = torch.from_numpy(w.mask).to(dev())
    sq = torch.from_numpy(w.seq_id).to(dev())

    hg, Wg = torch.from_numpy(h0).to(dev()), torch.from_numpy(W0).to(dev())  # GPU run's parameters
    ho, Wo = h0.copy(), W0.copy()                                          # oracle run's parameters
    gpu_losses, ora_losses = [], []
    for _ in range(STEPS):
        head.step(hg.to(torch.bfloat16), Wg.to(torch.bfloat16), tg, mk, sq, cap, w.lam)
        torch.cuda.synchronize()
        assert int(head.status.item()) == 0
        gpu_losses.append(float(head.out[0].item()))
        hg -= LR_H * head.dh
        Wg -= LR_W * head.dW

        _, h64 = bf16_round(ho)
        _, W64 = bf16_round(Wo)
        _, _, res, dh, dW = oracle.full_chain(h64, W64, w.targets, w.mask, w.seq_id, P, w.lam, cap)
        ora_losses.append(res.loss)
        ho = (ho - LR_H * dh).astype(np.float32)
        Wo = (Wo - LR_W * dW).astype(np.float32)

    g, o = np.array(gpu_losses), np.array(ora_losses)
    assert np.all(np.isfinite(g))
    assert np.all(np.diff(g) < 0), g          # every step lowers the loss
    assert o[-1] < 0.1 * o[0], o               # the oracle's run learns the batch too
    assert abs(g[0] - o[0]) <= 1e-4 * abs(o[0])
    # the two runs round different parameters to bf16 after the first step, so they drift apart
    # slowly; a gradient with a wrong sign, scale or term would separate them within a step
    assert np.max(np.abs(g - o) / np.abs(o)) < 5e-3, (g, o)
