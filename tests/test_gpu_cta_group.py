"""The other forms of the tensor-core engine, held to the same oracle comparisons.

The engine kernels run as 2-CTA clusters (tcgen05.mma.cta_group::2) wherever
clusters fit, which every other GPU test exercises.  Single-CTA tiles remain for
the backward skips and for devices where no cluster fits; ORPO_CTA_GROUP=1
selects them everywhere.  The dh/dW GEMM takes 256 x 512 pair tiles (all of
TMEM for one accumulator) only for wide outputs with several waves of tiles, so
few test shapes reach them by default; ORPO_GEMM_WIDE=1 selects them wherever
they are legal (ragged widths included: the second half of a tile past the
output is loaded as zeros and never stored).  Each test reruns a set of parity
tests in a child process with its setting.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_single_cta_form_matches_oracle():
    files = ["test_gpu_engine.py", "test_gpu_forward.py", "test_gpu_backward.py", "test_gpu_edges.py",
             "test_gpu_split_k.py"]
    env = dict(os.environ, ORPO_CTA_GROUP="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        *[os.path.join(ROOT, "tests", f) for f in files]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_wide_gemm_tiles_match_oracle():
    files = ["test_gpu_engine.py", "test_gpu_backward.py", "test_gpu_edges.py", "test_gpu_dense_multiblock.py",
             "test_gpu_quant.py"]
    env = dict(os.environ, ORPO_GEMM_WIDE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        *[os.path.join(ROOT, "tests", f) for f in files]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
