"""A whole head step (forward, loss, backward) captured once in a CUDA graph and replayed: the
library allocates nothing and enqueues only stream-ordered work, so replays must reproduce the
eager results bit for bit, here with a 16-block backward and with the backward skips."""

import numpy as np
import pytest
import torch

import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import dev, to_dev

pytestmark = pytest.mark.gpu


def outputs(head):
    return [x.detach().cpu().numpy().copy() for x in (head.logp, head.lse, head.out, head.g, head.dh, head.dW)]


@pytest.mark.parametrize("skip_eps", [0.0, 1e-5])
def test_step_replays_in_a_cuda_graph(skip_eps):
    w = workloads.make("e4b_sharp", M=16384 + 512, d=64, V=65536)   # 2 row blocks x 5 vocabulary blocks
    t = to_dev(w)
    h, W = t["h"].view(torch.bfloat16), t["W"].view(torch.bfloat16)
    head = orpo.OrpoHead(w.M, w.V, w.d, w.n_pairs, skip_eps=skip_eps)
    args = (h, W, t["targets"], t["mask"], t["seq_id"], w.softcap, w.lam)

    side = torch.cuda.Stream(dev())
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # eager warm-up off the default stream, then the reference
        head.step(*args)
        torch.cuda.synchronize()
        ref = outputs(head)
    torch.cuda.current_stream().wait_stream(side)
    assert int(head.status.item()) == 0

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        head.step(*args)
    for x in (head.logp, head.lse, head.out, head.g, head.dh, head.dW):
        x.fill_(float("nan"))
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        got = outputs(head)
        for a, b in zip(got, ref):
            assert np.array_equal(a, b)
    assert int(head.status.item()) == 0


def test_capture_replays_new_inputs_of_the_tiny_config():
    """OrpoHead.capture on the tiny config (a launch-bound step): a replay after new values are
    copied into the captured input tensors equals an eager step on those values, bit for bit."""
    w1 = workloads.make("tiny")
    w2 = workloads.make("tiny", seed=1)
    t1, t2 = to_dev(w1), to_dev(w2)
    bufs = {k: v.clone() for k, v in t1.items()}
    h, W = bufs["h"].view(torch.bfloat16), bufs["W"].view(torch.bfloat16)
    head = orpo.OrpoHead(w1.M, w1.V, w1.d, w1.n_pairs)
    graph = head.capture(h, W, bufs["targets"], bufs["mask"], bufs["seq_id"], w1.softcap, w1.lam)
    eager = orpo.OrpoHead(w1.M, w1.V, w1.d, w1.n_pairs)
    for t, w in ((t2, w2), (t1, w1)):
        for k in bufs:
            bufs[k].copy_(t[k])
        graph.replay()
        eager.step(t["h"].view(torch.bfloat16), t["W"].view(torch.bfloat16), t["targets"], t["mask"], t["seq_id"],
                   w.softcap, w.lam)
        torch.cuda.synchronize()
        for a, b in zip(outputs(head), outputs(eager)):
            assert np.array_equal(a, b)
    assert int(head.status.item()) == 0 and int(eager.status.item()) == 0
