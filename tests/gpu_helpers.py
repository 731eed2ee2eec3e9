"""Shared helpers for the GPU parity tests: move a workload to the device, run
the library through its C ABI, and compare with the oracle."""

import numpy as np
import torch

import oracle
import orpo_preference_loss_gb300 as orpo
import workloads

# tolerances fixed by the acceptance bar of this head
LOGP_ATOL = 2e-3
LOSS_RTOL = 1e-4
GRAD_RELFRO = 1e-2


def dev():
    return torch.device("cuda:0")


def to_dev(w: workloads.Workload):
    d = dev()
    return dict(
        h=torch.from_numpy(np.ascontiguousarray(w.h).view(np.int16)).to(d).view(torch.bfloat16),
        W=torch.from_numpy(np.ascontiguousarray(w.W).view(np.int16)).to(d).view(torch.bfloat16),
        targets=torch.from_numpy(np.ascontiguousarray(w.targets)).to(d),
        mask=torch.from_numpy(np.ascontiguousarray(w.mask)).to(d),
        seq_id=torch.from_numpy(np.ascontiguousarray(w.seq_id)).to(d),
    )


def f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def relfro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def status_tensor():
    return torch.zeros(1, dtype=torch.int32, device=dev())


def workspace(M, V, d):
    return torch.empty(orpo.orpo_head_workspace_bytes(M, V, d), dtype=torch.uint8, device=dev())


def gpu_forward(t, M, V, d, softcap, ws=None, st=None):
    logp = torch.full((M,), float("nan"), dtype=torch.float32, device=dev())
    lse = torch.full((M,), float("nan"), dtype=torch.float32, device=dev())
    ws = workspace(M, V, d) if ws is None else ws
    st = status_tensor() if st is None else st
    orpo.orpo_head_fwd(t["h"], t["W"], t["targets"], t["mask"], softcap, logp, lse, ws, st)
    torch.cuda.synchronize()
    return logp.cpu().numpy(), lse.cpu().numpy(), int(st.item())


def gpu_loss(logp_t, seq_t, mask_t, P, lam):
    M = logp_t.shape[0]
    out = torch.full((5,), float("nan"), dtype=torch.float32, device=dev())
    ell = torch.empty(2 * P, dtype=torch.float32, device=dev())
    g = torch.full((M,), float("nan"), dtype=torch.float32, device=dev())
    st = status_tensor()
    orpo.orpo_loss(logp_t, seq_t, mask_t, P, lam, out, ell, g, st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ell.cpu().numpy(), g.cpu().numpy(), int(st.item())


def gpu_backward(t, lse_np, g_np, M, V, d, softcap, dW_init=None, accumulate=False, ws=None):
    lse = torch.from_numpy(np.asarray(lse_np, dtype=np.float32)).to(dev())
    g = torch.from_numpy(np.asarray(g_np, dtype=np.float32)).to(dev())
    dh = torch.full((M, d), float("nan"), dtype=torch.float32, device=dev())
    if dW_init is None:
        dW = torch.full((V, d), float("nan"), dtype=torch.float32, device=dev())
    else:
        dW = torch.from_numpy(np.asarray(dW_init, dtype=np.float32)).to(dev())
    ws = workspace(M, V, d) if ws is None else ws
    st = status_tensor()
    orpo.orpo_head_bwd(t["h"], t["W"], t["targets"], t["mask"], lse, g, softcap, dh, dW, accumulate, ws, st)
    torch.cuda.synchronize()
    return dh.cpu().numpy(), dW.cpu().numpy(), int(st.item())
