"""Head steps shared by the bounds-checked-build test and the child process it starts: each case
runs forward, loss and backward through whichever library this process loaded and returns every
output with the status word."""

import numpy as np
import torch

import orpo_preference_loss_gb300 as orpo
import workloads

# (recipe, shape overrides, mode): edge shapes, a multi-block skip run, the quantised head
CASES = [
    ("tiny", {}, "exact"),
    ("e4b", dict(M=300, d=136, V=4160), "exact"),
    ("small", {}, "exact"),
    ("e4b_sharp", dict(M=16384 + 512, d=64, V=65536), "skip"),
    ("e4b", dict(M=2048, d=256, V=65536), "q4"),
]


def run_case(name, kw, mode):
    dev = torch.device("cuda:0")
    w = workloads.make(name, **kw)
    h = torch.from_numpy(np.ascontiguousarray(w.h).view(np.int16)).to(dev).view(torch.bfloat16)
    tg = torch.from_numpy(w.targets).to(dev)
    mk = torch.from_numpy(w.mask).to(dev)
    sq = torch.from_numpy(w.seq_id).to(dev)
    M, V, d, P = w.M, w.V, w.d, w.n_pairs
    if mode == "q4":
        wq, qs, qb = workloads.quantize_affine(w.W, 4, 64)
        q = (torch.from_numpy(wq).to(dev), torch.from_numpy(qs.view(np.int16)).to(dev).view(torch.bfloat16),
             torch.from_numpy(qb.view(np.int16)).to(dev).view(torch.bfloat16), 4, 64)
        ws = torch.empty(orpo.orpo_head_q_workspace_bytes(M, V, d), dtype=torch.uint8, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        logp, lse = torch.empty(M, device=dev), torch.empty(M, device=dev)
        out, ell, g = torch.empty(5, device=dev), torch.empty(2 * P, device=dev), torch.empty(M, device=dev)
        dh, dW = torch.empty((M, d), device=dev), torch.empty((V, d), device=dev)
        orpo.orpo_head_fwd_q(h, *q, tg, mk, w.softcap, logp, lse, ws, st)
        orpo.orpo_loss(logp, sq, mk, P, w.lam, out, ell, g, st)
        orpo.orpo_head_bwd_q(h, *q, tg, mk, lse, g, w.softcap, dh, dW, False, ws, st)
    else:
        W = torch.from_numpy(np.ascontiguousarray(w.W).view(np.int16)).to(dev).view(torch.bfloat16)
        head = orpo.OrpoHead(M, V, d, P, device=dev, skip_eps=1e-5 if mode == "skip" else 0.0)
        head.step(h, W, tg, mk, sq, w.softcap, w.lam)
        logp, lse, out, g, dh, dW, st = head.logp, head.lse, head.out, head.g, head.dh, head.dW, head.status
    torch.cuda.synchronize()
    res = {k: v.detach().cpu().numpy().copy() for k, v in
           dict(logp=logp, lse=lse, out=out, g=g, dh=dh, dW=dW).items()}
    res["status"] = np.array([int(st.item())])
    return res
