"""The C ABI without a GPU: the library builds, loads and exports every symbol
declared in include/*.h, and host-side argument checks return their codes
before any CUDA call is made."""

import ctypes
import glob
import math
import os
import re

import pytest

import orpo_preference_loss_gb300 as orpo
from orpo_preference_loss_gb300 import build as orpo_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_ARG, ERR_WS = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def lib():
    orpo_build.build()
    return orpo.load()


def declared_functions():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(orpo_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("orpo_head_fwd", "orpo_head_bwd", "orpo_loss", "orpo_head_workspace_bytes",
              "orpo_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared but not exported"


FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: every case fails before any CUDA call
MISALIGNED = ctypes.c_void_p(0x10008)
MAX_ROWS = (1 << 31) - (1 << 16)   # largest M and V the header documents


def fwd(lib, h=FAKE, W=FAKE, M=64, V=128, d=64, softcap=0.0, ws_bytes=1 << 30, tgt=FAKE, ws=FAKE):
    return lib.orpo_head_fwd(h, W, tgt, FAKE, M, V, d, softcap, FAKE, FAKE, ws, ws_bytes, FAKE, None)


def test_forward_host_checks(lib):
    assert fwd(lib, M=-1) == ERR_SHAPE
    assert fwd(lib, V=0) == ERR_SHAPE
    assert fwd(lib, d=4) == ERR_SHAPE
    assert fwd(lib, h=None) == ERR_NULL
    assert fwd(lib, tgt=None) == ERR_NULL
    assert fwd(lib, d=68) == ERR_ALIGN
    assert fwd(lib, W=MISALIGNED) == ERR_ALIGN
    assert fwd(lib, softcap=math.nan) == ERR_ARG
    assert fwd(lib, softcap=math.inf) == ERR_ARG
    assert fwd(lib, ws_bytes=16) == ERR_WS
    assert fwd(lib, M=0) == OK              # empty input: nothing to launch
    assert fwd(lib, M=MAX_ROWS + 1) == ERR_SHAPE
    assert fwd(lib, V=MAX_ROWS + 1) == ERR_SHAPE


def test_loss_host_checks(lib):
    call = lambda **k: lib.orpo_loss(k.get("logp", FAKE), FAKE, FAKE, k.get("M", 10), k.get("P", 1),
                                     k.get("lam", 0.1), FAKE, FAKE, FAKE, FAKE, None)
    assert call(P=0) == ERR_SHAPE
    assert call(P=orpo.MAX_PAIRS + 1) == ERR_SHAPE
    assert call(M=-3) == ERR_SHAPE
    assert call(M=MAX_ROWS + 1) == ERR_SHAPE
    assert call(logp=None) == ERR_NULL
    assert call(lam=-0.1) == ERR_ARG
    assert call(lam=math.nan) == ERR_ARG


def test_backward_host_checks(lib):
    def call(**k):
        return lib.orpo_head_bwd(k.get("h", FAKE), FAKE, FAKE, FAKE, FAKE, k.get("g", FAKE), k.get("M", 64), 128,
                                 k.get("d", 64), 0.0, k.get("dh", FAKE), FAKE, 0, FAKE, k.get("ws", 1 << 30),
                                 FAKE, None)
    assert call(M=-1) == ERR_SHAPE
    assert call(g=None) == ERR_NULL
    assert call(dh=MISALIGNED) == ERR_ALIGN
    assert call(d=12) == ERR_ALIGN
    assert call(ws=8) == ERR_WS


def test_status_strings(lib):
    assert orpo.orpo_status_string(0) == "ok"
    s = orpo.orpo_status_string(orpo.STATUS_BITS["target"] | orpo.STATUS_BITS["timeout"])
    assert "target" in s and "timed out" in s


def test_workspace_is_flat_in_M(lib):
    V, d = 262144, 2560
    base = lib.orpo_head_workspace_bytes(16384, V, d)
    # dZ block (padded pitch) + GEMM unit counters + the backward skips' plan slots
    assert base <= (258 << 20) + (16 << 10) + (4 << 20) + 1024
    # blocks are balanced (equal heights and widths), so the dZ block may be a little smaller than
    # at M = 16384, never larger
    for M in (16384, 20000, 65536, 131072, 16384 * 7 + 128):
        ws = lib.orpo_head_workspace_bytes(M, V, d)
        assert base * 0.9 <= ws <= base
    # far below any [M, V] buffer: 8192 x 262144 fp32 logits would be 8 GiB
    assert lib.orpo_head_workspace_bytes(8192, V, d) < (8192 * V * 4) // 16
    assert lib.orpo_head_workspace_bytes(-1, V, d) == 0
    # the documented limits: M, V <= 2^31 - 2^16
    assert lib.orpo_head_workspace_bytes(MAX_ROWS, V, d) > 0
    assert lib.orpo_head_workspace_bytes(8192, MAX_ROWS, 64) > 0
    assert lib.orpo_head_workspace_bytes(MAX_ROWS + 1, V, d) == 0
    assert lib.orpo_head_workspace_bytes(8192, MAX_ROWS + 1, 64) == 0


def test_skip_host_checks(lib):
    assert lib.orpo_head_block_max_elems(100, 1000) == 4 * 4
    assert lib.orpo_head_block_max_elems(8192, 262144) == 256 * 1024
    assert lib.orpo_head_block_max_elems(-1, 10) == 0
    assert orpo.block_max_shape(100, 1000) == (4, 4)

    def fwd_bm(bm=FAKE, M=64):
        return lib.orpo_head_fwd_bmax(FAKE, FAKE, FAKE, FAKE, M, 128, 64, 0.0, FAKE, FAKE, bm, FAKE, 1 << 30, FAKE,
                                      None)

    assert fwd_bm(bm=None) == ERR_NULL
    assert fwd_bm(bm=ctypes.c_void_p(0x10002)) == ERR_ALIGN
    assert fwd_bm(M=-1) == ERR_SHAPE

    def bwd_skip(eps=1e-5, bm=FAKE, ws=1 << 30):
        return lib.orpo_head_bwd_skip(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, bm, eps, 64, 128, 64, 0.0, FAKE, FAKE, 0,
                                      FAKE, ws, FAKE, None)

    assert bwd_skip(eps=-1e-5) == ERR_ARG
    assert bwd_skip(eps=float("nan")) == ERR_ARG
    assert bwd_skip(eps=float("inf")) == ERR_ARG
    assert bwd_skip(bm=ctypes.c_void_p(0x10002)) == ERR_ALIGN
    assert bwd_skip(ws=8) == ERR_WS


def test_quantised_skip_host_checks(lib):
    def fwd(bm=FAKE, M=64):
        return lib.orpo_head_fwd_q_bmax(FAKE, FAKE, FAKE, FAKE, 4, 64, FAKE, FAKE, M, 128, 64, 0.0, FAKE, FAKE, bm,
                                        FAKE, 1 << 30, FAKE, None)

    def bwd(eps=1e-5, bits=4):
        return lib.orpo_head_bwd_q_skip(FAKE, FAKE, FAKE, FAKE, bits, 64, FAKE, FAKE, FAKE, FAKE, FAKE, eps, 64, 128,
                                        64, 0.0, FAKE, FAKE, 0, FAKE, 1 << 30, FAKE, None)

    assert fwd(bm=None) == ERR_NULL
    assert fwd(bm=ctypes.c_void_p(0x10002)) == ERR_ALIGN
    assert bwd(eps=-1.0) == ERR_ARG
    assert bwd(bits=5) == ERR_ARG


def test_quantised_workspace_stays_bounded(lib):
    # the dequantised W block keeps to its 256 MiB budget at every M, also when few rows would let the
    # dZ block span the whole vocabulary; the whole quantised workspace stays far below a bf16 copy of W
    for V, d in ((262144, 2560), (128256, 4096), (32000, 2048)):
        for M in (1, 128, 512, 2048, 8192, 65536):
            q = orpo.orpo_head_q_workspace_bytes(M, V, d)
            b = orpo.orpo_head_workspace_bytes(M, V, d)
            assert 0 < q - b <= (256 << 20) + (192 << 20), (V, d, M, q, b)   # W block + larger split table
            assert q <= (520 << 20), (V, d, M, q)
