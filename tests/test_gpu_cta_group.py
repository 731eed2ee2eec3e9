"""Both forms of the tensor-core engine, held to the same oracle comparisons.

The engine kernels run either on single CTAs or as 2-CTA clusters
(tcgen05.mma.cta_group::2).  By default only the dh / dW GEMM uses clusters;
ORPO_CTA_GROUP=1 selects single CTAs everywhere and ORPO_CTA_GROUP=2 clusters
everywhere (forward and recompute included).  This test reruns the engine,
forward, backward, edge-case and split-K parity tests in a child process under
each setting, so every kernel is checked in both forms.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("group", ["1", "2"])
def test_engine_form_matches_oracle(group):
    files = ["test_gpu_engine.py", "test_gpu_forward.py", "test_gpu_backward.py", "test_gpu_edges.py",
             "test_gpu_split_k.py"]
    env = dict(os.environ, ORPO_CTA_GROUP=group)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        *[os.path.join(ROOT, "tests", f) for f in files]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
