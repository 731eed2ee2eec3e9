"""The C ABI from a plain C program (no C++, no PyTorch): the header compiles as C99 and the
program links against liborpo_head.so and the CUDA runtime (CPU test); on a GPU it runs a whole
step on the tiny workload, and its outputs match the oracle (GPU test)."""

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import workloads
from orpo_preference_loss_gb300 import build as orpo_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_caller", "orpo_step.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_caller(out_dir):
    lib = orpo_build.build()
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = os.path.join(out_dir, "orpo_step")
    lib_dir = os.path.dirname(lib)
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), SRC, "-o", exe, "-L", lib_dir, "-lorpo_head",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{lib_dir}",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_header_compiles_as_c_and_links(tmp_path):
    assert os.path.exists(compile_caller(str(tmp_path)))


@pytest.mark.gpu
def test_c_caller_step_matches_oracle(tmp_path):
    exe = compile_caller(str(tmp_path))
    w = workloads.make("tiny")
    c = 30.0
    d = str(tmp_path)
    w.h.tofile(os.path.join(d, "h.bin"))
    w.W.tofile(os.path.join(d, "W.bin"))
    w.targets.astype(np.int32).tofile(os.path.join(d, "targets.bin"))
    w.mask.astype(np.uint8).tofile(os.path.join(d, "mask.bin"))
    w.seq_id.astype(np.int32).tofile(os.path.join(d, "seq_id.bin"))
    r = subprocess.run([exe, d, str(w.M), str(w.V), str(w.d), str(w.n_pairs), str(c), str(w.lam)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert open(os.path.join(d, "status.txt")).read().strip() == "0"
    rd = lambda name, shape: np.fromfile(os.path.join(d, name), dtype=np.float32).reshape(shape)
    logp, lse, res, dh, dW = oracle.full_chain(oracle.bf16_bits_to_f64(w.h), oracle.bf16_bits_to_f64(w.W), w.targets,
                                               w.mask, w.seq_id, w.n_pairs, w.lam, c)
    assert np.max(np.abs(rd("logp.bin", (w.M,)) - logp)) < 2e-3
    assert np.max(np.abs(rd("lse.bin", (w.M,)) - lse)) < 2e-3
    assert abs(rd("out.bin", (5,))[0] - res.loss) <= 1e-4 * abs(res.loss)
    relfro = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert relfro(rd("dh.bin", (w.M, w.d)), dh) < 1e-2
    assert relfro(rd("dW.bin", (w.V, w.d)), dW) < 1e-2
