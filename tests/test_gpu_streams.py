"""Independent head steps enqueued at once from several host threads, each on its own stream with its
own workspace and outputs, give the same bits as the same steps run one after the other.  The library
keeps no per-call state outside the caller's buffers, so concurrent calls of different shapes and
modes (exact, skips, quantised) neither race on the host nor share device memory."""

import threading

import numpy as np
import pytest
import torch

import orpo_preference_loss_gb300 as orpo
import workloads
from gpu_helpers import dev, to_dev

pytestmark = pytest.mark.gpu


def outputs(head):
    return [x.detach().cpu().numpy().copy() for x in (head.logp, head.lse, head.out, head.g, head.dh, head.dW)]


class QuantHead:
    """The same step on a 4-bit affine quantised head (groups of 64)."""

    def __init__(self, w, t):
        wq, qs, qb = workloads.quantize_affine(w.W, 4, 64)
        d = dev()
        self.wq = torch.from_numpy(wq).to(d)
        self.qs = torch.from_numpy(qs.view(np.int16)).to(d).view(torch.bfloat16)
        self.qb = torch.from_numpy(qb.view(np.int16)).to(d).view(torch.bfloat16)
        self.w, self.t = w, t
        M, V, dd, P = w.M, w.V, w.d, w.n_pairs
        self.workspace = torch.empty(orpo.orpo_head_q_workspace_bytes(M, V, dd), dtype=torch.uint8, device=d)
        self.status = torch.zeros(1, dtype=torch.int32, device=d)
        self.logp = torch.empty(M, device=d)
        self.lse = torch.empty(M, device=d)
        self.out = torch.empty(5, device=d)
        self.ell = torch.empty(2 * P, device=d)
        self.g = torch.empty(M, device=d)
        self.dh = torch.empty((M, dd), device=d)
        self.dW = torch.empty((V, dd), device=d)

    def step(self):
        w, t = self.w, self.t
        h = t["h"].view(torch.bfloat16)
        q = (self.wq, self.qs, self.qb, 4, 64)
        orpo.orpo_head_fwd_q(h, *q, t["targets"], t["mask"], w.softcap, self.logp, self.lse, self.workspace,
                             self.status)
        orpo.orpo_loss(self.logp, t["seq_id"], t["mask"], w.n_pairs, w.lam, self.out, self.ell, self.g, self.status)
        orpo.orpo_head_bwd_q(h, *q, t["targets"], t["mask"], self.lse, self.g, w.softcap, self.dh, self.dW, False,
                             self.workspace, self.status)


class BfHead:
    def __init__(self, w, t, skip_eps=0.0):
        self.head = orpo.OrpoHead(w.M, w.V, w.d, w.n_pairs, skip_eps=skip_eps)
        self.args = (t["h"].view(torch.bfloat16), t["W"].view(torch.bfloat16), t["targets"], t["mask"],
                     t["seq_id"], w.softcap, w.lam)
        for name in ("logp", "lse", "out", "g", "dh", "dW", "status"):
            setattr(self, name, getattr(self.head, name))

    def step(self):
        self.head.step(*self.args)


def test_concurrent_steps_on_separate_streams_match_serial_runs():
    cases = [
        ("small", {}, lambda w, t: BfHead(w, t)),
        ("e4b_sharp", dict(M=4096 + 256, d=128, V=32768 + 512), lambda w, t: BfHead(w, t, skip_eps=1e-5)),
        ("e4b", dict(M=2048, d=256, V=65536), lambda w, t: QuantHead(w, t)),
        ("tiny", {}, lambda w, t: BfHead(w, t)),
    ]
    heads = []
    for name, kw, make in cases:
        w = workloads.make(name, **kw)
        heads.append(make(w, to_dev(w)))

    ref = []
    for hd in heads:  # serial, on the default stream
        hd.step()
        torch.cuda.synchronize()
        assert int(hd.status.item()) == 0
        ref.append(outputs(hd))
        for x in (hd.logp, hd.lse, hd.out, hd.g, hd.dh, hd.dW):
            x.fill_(float("nan"))
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream(dev()) for _ in heads]
    start = threading.Barrier(len(heads))
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(dev())
            with torch.cuda.stream(streams[i]):
                start.wait()
                for _ in range(2):
                    heads[i].step()
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(heads))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for hd, r in zip(heads, ref):
        assert int(hd.status.item()) == 0
        for a, b in zip(outputs(hd), r):
            assert np.array_equal(a, b)
