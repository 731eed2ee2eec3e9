"""GB300 (sm_103a) flash-CCE ORPO head: Python binding of liborpo_head.

The functions here carry the C entry points' names and only marshal arguments:
every step of the head runs in the library's CUDA kernels.  PyTorch supplies
device memory and the current CUDA stream.  If the library has not been built
(``python -c "import __graft_entry__ as g; g.build()"``) the calls raise; there
is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "OrpoError", "load", "lib_path", "orpo_head_workspace_bytes", "orpo_head_fwd", "orpo_loss",
    "orpo_head_bwd", "orpo_status_string", "orpo_debug_gemm", "OrpoHead", "STATUS_BITS",
    "orpo_profile_start", "orpo_profile_stop", "orpo_head_fwd_static", "orpo_debug_wait_timeout",
    "orpo_pref_loss", "PREF_KINDS", "orpo_head_q_workspace_bytes", "orpo_head_fwd_q", "orpo_head_bwd_q",
    "use_bounds_checked_library",
]

STATUS_BITS = {"target": 1 << 4, "seqid": 1 << 5, "empty": 1 << 6, "nonfinite": 1 << 7, "timeout": 1 << 8,
               "bounds": 1 << 9}
MAX_PAIRS = 2048

_lib = None


class OrpoError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {orpo_status_string(code)} (code {code})")
        self.code = code


_variant = "release"


def lib_path() -> str:
    return _build.DEBUG_LIB_PATH if _variant == "debug" else _build.LIB_PATH


def use_bounds_checked_library() -> None:
    """Bind this process to liborpo_head_debug.so (build(debug=True)) instead of liborpo_head.so.

    The bounds-checked build checks every computed index against its buffer and reports a miss
    as ORPO_STATUS_BOUNDS; its arithmetic is the release build's.  Call before the first use."""
    global _variant
    if _lib is not None and _variant != "debug":
        raise RuntimeError("the release library is already loaded in this process")
    _variant = "debug"


def load():
    """Load the library (built in-tree); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with orpo_preference_loss_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    L.orpo_head_workspace_bytes.argtypes = [i64, i64, i64]
    L.orpo_head_workspace_bytes.restype = sz
    L.orpo_head_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, vp, vp, vp, sz, vp, vp]
    L.orpo_head_fwd.restype = ctypes.c_int
    L.orpo_loss.argtypes = [vp, vp, vp, i64, i32, f32, vp, vp, vp, vp, vp]
    L.orpo_loss.restype = ctypes.c_int
    L.orpo_head_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, f32, vp, vp, ctypes.c_int, vp, sz, vp, vp]
    L.orpo_head_bwd.restype = ctypes.c_int
    L.orpo_status_string.argtypes = [ctypes.c_int]
    L.orpo_status_string.restype = ctypes.c_char_p
    L.orpo_debug_gemm.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int, ctypes.c_int, vp, vp]
    L.orpo_debug_gemm.restype = ctypes.c_int
    L.orpo_pref_loss.argtypes = [ctypes.c_int, vp, vp, vp, i64, i32, f32, f32, vp, vp, vp, vp, vp, vp]
    L.orpo_pref_loss.restype = ctypes.c_int
    L.orpo_head_q_workspace_bytes.argtypes = [i64, i64, i64]
    L.orpo_head_q_workspace_bytes.restype = sz
    L.orpo_head_fwd_q.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp, i64, i64, i64, f32, vp, vp, vp,
                                  sz, vp, vp]
    L.orpo_head_fwd_q.restype = ctypes.c_int
    L.orpo_head_bwd_q.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, i64, i64, i64, f32, vp,
                                  vp, ctypes.c_int, vp, sz, vp, vp]
    L.orpo_head_bwd_q.restype = ctypes.c_int
    L.orpo_head_fwd_static.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, vp, vp, vp, vp]
    L.orpo_head_fwd_static.restype = ctypes.c_int
    L.orpo_debug_wait_timeout.argtypes = [vp, i64, vp]
    L.orpo_debug_wait_timeout.restype = ctypes.c_int
    L.orpo_head_block_max_elems.argtypes = [i64, i64]
    L.orpo_head_block_max_elems.restype = sz
    L.orpo_head_fwd_bmax.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, vp, vp, vp, vp, sz, vp, vp]
    L.orpo_head_fwd_bmax.restype = ctypes.c_int
    L.orpo_head_bwd_skip.argtypes = [vp, vp, vp, vp, vp, vp, vp, f32, i64, i64, i64, f32, vp, vp, ctypes.c_int, vp,
                                     sz, vp, vp]
    L.orpo_head_bwd_skip.restype = ctypes.c_int
    L.orpo_head_fwd_q_bmax.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp, i64, i64, i64, f32, vp,
                                       vp, vp, vp, sz, vp, vp]
    L.orpo_head_fwd_q_bmax.restype = ctypes.c_int
    L.orpo_head_bwd_q_skip.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, f32, i64, i64,
                                       i64, f32, vp, vp, ctypes.c_int, vp, sz, vp, vp]
    L.orpo_head_bwd_q_skip.restype = ctypes.c_int
    L.orpo_profile_start.argtypes = []
    L.orpo_profile_start.restype = ctypes.c_int
    L.orpo_profile_stop.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64), ctypes.c_int]
    L.orpo_profile_stop.restype = ctypes.c_int
    L.orpo_profile_kind_name.argtypes = [ctypes.c_int]
    L.orpo_profile_kind_name.restype = ctypes.c_char_p
    _lib = L
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code, what):
    if code != 0:
        raise OrpoError(code, what)


def _dev(t, name, dtypes, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)


def orpo_status_string(code: int) -> str:
    return load().orpo_status_string(int(code)).decode()


def orpo_head_workspace_bytes(M: int, V: int, d: int) -> int:
    return int(load().orpo_head_workspace_bytes(M, V, d))


def orpo_head_fwd(h, W, targets, mask, softcap, logp, lse, workspace, status, stream=None):
    M, d = h.shape
    V = W.shape[0]
    _dev(h, "h", BF16)
    _dev(W, "W", BF16, (V, d))
    _dev(targets, "targets", (torch.int32,), (M,))
    _dev(mask, "mask", (torch.uint8, torch.bool), (M,))
    _dev(logp, "logp", (torch.float32,), (M,))
    _dev(lse, "lse", (torch.float32,), (M,))
    _dev(workspace, "workspace", (torch.uint8,))
    _dev(status, "status", (torch.int32,))
    _check(load().orpo_head_fwd(_ptr(h), _ptr(W), _ptr(targets), _ptr(mask), M, V, d, float(softcap),
                                _ptr(logp), _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(status),
                                _stream(stream)), "orpo_head_fwd")


FWD_STATIC_MAX_ROWS = 65536


def orpo_head_fwd_static(h, W, targets, mask, softcap, logp, lse, status, stream=None):
    """orpo_head_fwd without a workspace argument, for callers that may not allocate
    device memory: the split partials use a fixed array inside the library."""
    M, d = h.shape
    V = W.shape[0]
    _dev(h, "h", BF16)
    _dev(W, "W", BF16, (V, d))
    _dev(targets, "targets", (torch.int32,), (M,))
    _dev(mask, "mask", (torch.uint8, torch.bool), (M,))
    _dev(logp, "logp", (torch.float32,), (M,))
    _dev(lse, "lse", (torch.float32,), (M,))
    _dev(status, "status", (torch.int32,))
    _check(load().orpo_head_fwd_static(_ptr(h), _ptr(W), _ptr(targets), _ptr(mask), M, V, d, float(softcap),
                                       _ptr(logp), _ptr(lse), _ptr(status), _stream(stream)),
           "orpo_head_fwd_static")


def orpo_loss(logp, seq_id, mask, n_pairs, lam, out, ell, g, status, stream=None):
    M = logp.shape[0]
    _dev(logp, "logp", (torch.float32,), (M,))
    _dev(seq_id, "seq_id", (torch.int32,), (M,))
    _dev(mask, "mask", (torch.uint8, torch.bool), (M,))
    _dev(out, "out", (torch.float32,), (5,))
    _dev(ell, "ell", (torch.float32,), (2 * n_pairs,))
    _dev(g, "g", (torch.float32,), (M,))
    _dev(status, "status", (torch.int32,))
    _check(load().orpo_loss(_ptr(logp), _ptr(seq_id), _ptr(mask), M, int(n_pairs), float(lam), _ptr(out),
                            _ptr(ell), _ptr(g), _ptr(status), _stream(stream)), "orpo_loss")


PREF_KINDS = {"orpo": 0, "simpo": 1, "dpo": 2, "ipo": 3, "hinge": 4, "orpo_full": 5}


def orpo_pref_loss(kind, logp, seq_id, mask, n_pairs, beta, gamma, ref_logp, out, ell, g, status, stream=None):
    """Sibling preference objective `kind` (orpo, simpo, dpo, ipo, hinge) on per-token logp."""
    M = logp.shape[0]
    k = PREF_KINDS[kind] if isinstance(kind, str) else int(kind)
    _dev(logp, "logp", (torch.float32,), (M,))
    _dev(seq_id, "seq_id", (torch.int32,), (M,))
    _dev(mask, "mask", (torch.uint8, torch.bool), (M,))
    _dev(out, "out", (torch.float32,), (5,))
    _dev(ell, "ell", (torch.float32,), (2 * n_pairs,))
    _dev(g, "g", (torch.float32,), (M,))
    _dev(status, "status", (torch.int32,))
    if ref_logp is not None:
        _dev(ref_logp, "ref_logp", (torch.float32,), (2 * n_pairs,))
    _check(load().orpo_pref_loss(k, _ptr(logp), _ptr(seq_id), _ptr(mask), M, int(n_pairs), float(beta), float(gamma),
                                 _ptr(ref_logp), _ptr(out), _ptr(ell), _ptr(g), _ptr(status), _stream(stream)),
           "orpo_pref_loss")


def orpo_head_bwd(h, W, targets, mask, lse, g, softcap, dh, dW, accumulate_dW, workspace, status,
                  stream=None):
    M, d = h.shape
    V = W.shape[0]
    _dev(h, "h", BF16)
    _dev(W, "W", BF16, (V, d))
    _dev(targets, "targets", (torch.int32,), (M,))
    _dev(mask, "mask", (torch.uint8, torch.bool), (M,))
    _dev(lse, "lse", (torch.float32,), (M,))
    _dev(g, "g", (torch.float32,), (M,))
    _dev(dh, "dh", (torch.float32,), (M, d))
    if dW is not None:
        _dev(dW, "dW", (torch.float32,), (V, d))
    _dev(workspace, "workspace", (torch.uint8,))
    _dev(status, "status", (torch.int32,))
    _check(load().orpo_head_bwd(_ptr(h), _ptr(W), _ptr(targets), _ptr(mask), _ptr(lse), _ptr(g), M, V, d,
                                float(softcap), _ptr(dh), _ptr(dW), 1 if accumulate_dW else 0, _ptr(workspace),
                                workspace.numel(), _ptr(status), _stream(stream)), "orpo_head_bwd")


def orpo_head_block_max_elems(M: int, V: int) -> int:
    return int(load().orpo_head_block_max_elems(M, V))


def block_max_shape(M: int, V: int):
    """[ceil(M / 32), ceil(V / 256)]: the block-max array of the backward skips."""
    return (-(-M // 32), -(-V // 256))


def orpo_head_fwd_bmax(h, W, targets, mask, softcap, logp, lse, block_max, workspace, status, stream=None):
    """orpo_head_fwd that also writes the block maxima the backward's block skip reads."""
    M, d = h.shape
    V = W.shape[0]
    _dev(h, "h", BF16)
    _dev(W, "W", BF16, (V, d))
    _dev(targets, "targets", (torch.int32,), (M,))
    _dev(mask, "mask", (torch.uint8, torch.bool), (M,))
    _dev(logp, "logp", (torch.float32,), (M,))
    _dev(lse, "lse", (torch.float32,), (M,))
    _dev(block_max, "block_max", (torch.float32,), block_max_shape(M, V))
    _dev(workspace, "workspace", (torch.uint8,))
    _dev(status, "status", (torch.int32,))
    _check(load().orpo_head_fwd_bmax(_ptr(h), _ptr(W), _ptr(targets), _ptr(mask), M, V, d, float(softcap),
                                     _ptr(logp), _ptr(lse), _ptr(block_max), _ptr(workspace), workspace.numel(),
                                     _ptr(status), _stream(stream)), "orpo_head_fwd_bmax")


def orpo_head_bwd_skip(h, W, targets, mask, lse, g, block_max, eps, softcap, dh, dW, accumulate_dW, workspace,
                       status, stream=None):
    """orpo_head_bwd with the backward skips: the coefficient filter at eps, and the block skip when
    block_max (from orpo_head_fwd_bmax) is given (None: filter alone)."""
    M, d = h.shape
    V = W.shape[0]
    _dev(h, "h", BF16)
    _dev(W, "W", BF16, (V, d))
    _dev(targets, "targets", (torch.int32,), (M,))
    _dev(mask, "mask", (torch.uint8, torch.bool), (M,))
    _dev(lse, "lse", (torch.float32,), (M,))
    _dev(g, "g", (torch.float32,), (M,))
    if block_max is not None:
        _dev(block_max, "block_max", (torch.float32,), block_max_shape(M, V))
    _dev(dh, "dh", (torch.float32,), (M, d))
    if dW is not None:
        _dev(dW, "dW", (torch.float32,), (V, d))
    _dev(workspace, "workspace", (torch.uint8,))
    _dev(status, "status", (torch.int32,))
    _check(load().orpo_head_bwd_skip(_ptr(h), _ptr(W), _ptr(targets), _ptr(mask), _ptr(lse), _ptr(g),
                                     _ptr(block_max), float(eps), M, V, d, float(softcap), _ptr(dh), _ptr(dW),
                                     1 if accumulate_dW else 0, _ptr(workspace), workspace.numel(), _ptr(status),
                                     _stream(stream)), "orpo_head_bwd_skip")


def orpo_head_q_workspace_bytes(M: int, V: int, d: int) -> int:
    return int(load().orpo_head_q_workspace_bytes(M, V, d))


def _quant_args(wq, scales, biases, V, d, bits, group):
    _dev(wq, "wq", (torch.uint8,), (V, d * bits // 8))
    _dev(scales, "scales", BF16, (V, d // group))
    _dev(biases, "biases", BF16, (V, d // group))


def orpo_head_fwd_q(h, wq, scales, biases, bits, group, targets, mask, softcap, logp, lse, workspace, status,
                    stream=None):
    """orpo_head_fwd on an affine group-quantised head (wq, scales, biases)."""
    M, d = h.shape
    V = wq.shape[0]
    _dev(h, "h", BF16)
    _quant_args(wq, scales, biases, V, d, bits, group)
    _dev(targets, "targets", (torch.int32,), (M,))
    _dev(mask, "mask", (torch.uint8, torch.bool), (M,))
    _dev(logp, "logp", (torch.float32,), (M,))
    _dev(lse, "lse", (torch.float32,), (M,))
    _dev(workspace, "workspace", (torch.uint8,))
    _check(load().orpo_head_fwd_q(_ptr(h), _ptr(wq), _ptr(scales), _ptr(biases), int(bits), int(group), _ptr(targets),
                                  _ptr(mask), M, V, d, float(softcap), _ptr(logp), _ptr(lse), _ptr(workspace),
                                  workspace.numel(), _ptr(status), _stream(stream)), "orpo_head_fwd_q")


def orpo_head_bwd_q(h, wq, scales, biases, bits, group, targets, mask, lse, g, softcap, dh, dW, accumulate_dW,
                    workspace, status, stream=None):
    """orpo_head_bwd on an affine group-quantised head; dW (optional) is w.r.t. the dequantised weight."""
    M, d = h.shape
    V = wq.shape[0]
    _dev(h, "h", BF16)
    _quant_args(wq, scales, biases, V, d, bits, group)
    _dev(lse, "lse", (torch.float32,), (M,))
    _dev(g, "g", (torch.float32,), (M,))
    _dev(dh, "dh", (torch.float32,), (M, d))
    if dW is not None:
        _dev(dW, "dW", (torch.float32,), (V, d))
    _check(load().orpo_head_bwd_q(_ptr(h), _ptr(wq), _ptr(scales), _ptr(biases), int(bits), int(group), _ptr(targets),
                                  _ptr(mask), _ptr(lse), _ptr(g), M, V, d, float(softcap), _ptr(dh), _ptr(dW),
                                  1 if accumulate_dW else 0, _ptr(workspace), workspace.numel(), _ptr(status),
                                  _stream(stream)), "orpo_head_bwd_q")


def orpo_head_fwd_q_bmax(h, wq, scales, biases, bits, group, targets, mask, softcap, logp, lse, block_max,
                         workspace, status, stream=None):
    """orpo_head_fwd_q that also writes the block maxima of the backward skips."""
    M, d = h.shape
    V = wq.shape[0]
    _dev(h, "h", BF16)
    _quant_args(wq, scales, biases, V, d, bits, group)
    _dev(targets, "targets", (torch.int32,), (M,))
    _dev(mask, "mask", (torch.uint8, torch.bool), (M,))
    _dev(logp, "logp", (torch.float32,), (M,))
    _dev(lse, "lse", (torch.float32,), (M,))
    _dev(block_max, "block_max", (torch.float32,), block_max_shape(M, V))
    _dev(workspace, "workspace", (torch.uint8,))
    _check(load().orpo_head_fwd_q_bmax(_ptr(h), _ptr(wq), _ptr(scales), _ptr(biases), int(bits), int(group),
                                       _ptr(targets), _ptr(mask), M, V, d, float(softcap), _ptr(logp), _ptr(lse),
                                       _ptr(block_max), _ptr(workspace), workspace.numel(), _ptr(status),
                                       _stream(stream)), "orpo_head_fwd_q_bmax")


def orpo_head_bwd_q_skip(h, wq, scales, biases, bits, group, targets, mask, lse, g, block_max, eps, softcap, dh, dW,
                         accumulate_dW, workspace, status, stream=None):
    """orpo_head_bwd_q with the backward skips (block_max may be None: filter alone)."""
    M, d = h.shape
    V = wq.shape[0]
    _dev(h, "h", BF16)
    _quant_args(wq, scales, biases, V, d, bits, group)
    _dev(lse, "lse", (torch.float32,), (M,))
    _dev(g, "g", (torch.float32,), (M,))
    if block_max is not None:
        _dev(block_max, "block_max", (torch.float32,), block_max_shape(M, V))
    _dev(dh, "dh", (torch.float32,), (M, d))
    if dW is not None:
        _dev(dW, "dW", (torch.float32,), (V, d))
    _check(load().orpo_head_bwd_q_skip(_ptr(h), _ptr(wq), _ptr(scales), _ptr(biases), int(bits), int(group),
                                       _ptr(targets), _ptr(mask), _ptr(lse), _ptr(g), _ptr(block_max), float(eps), M, V,
                                       d, float(softcap), _ptr(dh), _ptr(dW), 1 if accumulate_dW else 0,
                                       _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream)),
           "orpo_head_bwd_q_skip")


def orpo_debug_gemm(A, B, C, M, N, K, a_mn_major, b_mn_major, status, stream=None):
    _dev(A, "A", BF16)
    _dev(B, "B", BF16)
    _dev(C, "C", (torch.float32,), (M, N))
    _check(load().orpo_debug_gemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(a_mn_major), int(b_mn_major),
                                  _ptr(status), _stream(stream)), "orpo_debug_gemm")


def orpo_debug_wait_timeout(status, limit_ns, stream=None):
    _dev(status, "status", (torch.int32,))
    _check(load().orpo_debug_wait_timeout(_ptr(status), int(limit_ns), _stream(stream)), "orpo_debug_wait_timeout")


PROFILE_KINDS = 8


def orpo_profile_start():
    _check(load().orpo_profile_start(), "orpo_profile_start")


def orpo_profile_stop():
    """Per kernel kind: {name: (total_ms, launches)} for the launches since orpo_profile_start()."""
    ms = (ctypes.c_double * PROFILE_KINDS)()
    cnt = (ctypes.c_int64 * PROFILE_KINDS)()
    _check(load().orpo_profile_stop(ms, cnt, PROFILE_KINDS), "orpo_profile_stop")
    return {load().orpo_profile_kind_name(k).decode(): (ms[k], int(cnt[k])) for k in range(PROFILE_KINDS)}


class OrpoHead:
    """Owns the per-size device buffers (workspace, outputs) and runs one head step.

    All tensors come from PyTorch's allocator; the step itself is the three C
    entry points in order on the current stream.
    """

    def __init__(self, M: int, V: int, d: int, n_pairs: int, device="cuda", skip_eps: float = 0.0):
        """skip_eps > 0 turns on the backward skips (coefficient filter and block skip) at that eps."""
        self.M, self.V, self.d, self.P = M, V, d, n_pairs
        self.skip_eps = float(skip_eps)
        dev = torch.device(device)
        self.block_max = (torch.empty(block_max_shape(M, V), dtype=torch.float32, device=dev)
                          if self.skip_eps > 0 else None)
        self.workspace = torch.empty(orpo_head_workspace_bytes(M, V, d), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.logp = torch.empty(M, dtype=torch.float32, device=dev)
        self.lse = torch.empty(M, dtype=torch.float32, device=dev)
        self.out = torch.empty(5, dtype=torch.float32, device=dev)
        self.ell = torch.empty(2 * n_pairs, dtype=torch.float32, device=dev)
        self.g = torch.empty(M, dtype=torch.float32, device=dev)
        self.dh = torch.empty((M, d), dtype=torch.float32, device=dev)
        self.dW = torch.empty((V, d), dtype=torch.float32, device=dev)

    def step(self, h, W, targets, mask, seq_id, softcap, lam, accumulate_dW=False, stream=None):
        if self.skip_eps > 0:
            orpo_head_fwd_bmax(h, W, targets, mask, softcap, self.logp, self.lse, self.block_max, self.workspace,
                               self.status, stream)
        else:
            orpo_head_fwd(h, W, targets, mask, softcap, self.logp, self.lse, self.workspace, self.status, stream)
        orpo_loss(self.logp, seq_id, mask, self.P, lam, self.out, self.ell, self.g, self.status, stream)
        if self.skip_eps > 0:
            orpo_head_bwd_skip(h, W, targets, mask, self.lse, self.g, self.block_max, self.skip_eps, softcap,
                               self.dh, self.dW, accumulate_dW, self.workspace, self.status, stream)
        else:
            orpo_head_bwd(h, W, targets, mask, self.lse, self.g, softcap, self.dh, self.dW, accumulate_dW,
                          self.workspace, self.status, stream)
        return self.out

    def capture(self, h, W, targets, mask, seq_id, softcap, lam, accumulate_dW=False):
        """Record one step on these tensors into a CUDA graph and return it.

        Each ``graph.replay()`` reruns the whole step (forward, loss, backward: 5 or more launches)
        on whatever the given tensors hold at that moment, for the price of one launch; this matters
        for small batches, whose step is a few launches of microseconds.  The step runs once eagerly
        first, on a side stream, so that the library's one-time device set-up happens outside the
        capture.  Fill the same input tensors before each replay; the outputs land in this head's
        buffers as with step()."""
        args = (h, W, targets, mask, seq_id, softcap, lam, accumulate_dW)
        side = torch.cuda.Stream(self.workspace.device)
        side.wait_stream(torch.cuda.current_stream(self.workspace.device))
        with torch.cuda.stream(side):
            self.step(*args)
        torch.cuda.current_stream(self.workspace.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.step(*args)
        return graph
