"""The bounds-checked build (ORPO_DEBUG_BOUNDS: every computed index is tested against its buffer,
and a miss sets ORPO_STATUS_BOUNDS instead of touching memory) over edge shapes, a multi-block
run with the backward skips and the quantised head.  No index leaves its buffer, and the outputs
equal the release build's bit for bit: the checks change no arithmetic.  The checked library runs
in a child process, since one process binds one variant."""

import os
import subprocess
import sys

import numpy as np
import pytest

import orpo_preference_loss_gb300 as orpo
from bounds_cases import CASES, run_case

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import numpy as np
import orpo_preference_loss_gb300 as orpo
from orpo_preference_loss_gb300 import build
build.build(debug=True)
orpo.use_bounds_checked_library()
from bounds_cases import CASES, run_case
for i, (name, kw, mode) in enumerate(CASES):
    np.savez({out!r} + f"/case{{i}}.npz", **run_case(name, kw, mode))
print("loaded", orpo.lib_path())
"""


def test_bounds_checked_build_matches_release(tmp_path):
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), out=str(tmp_path))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "liborpo_head_debug.so" in r.stdout
    for i, (name, kw, mode) in enumerate(CASES):
        checked = np.load(tmp_path / f"case{i}.npz")
        st = int(checked["status"][0])
        assert st & orpo.STATUS_BITS["bounds"] == 0, (name, mode, orpo.orpo_status_string(st))
        assert st == 0, (name, mode, orpo.orpo_status_string(st))
        release = run_case(name, kw, mode)
        assert int(release["status"][0]) == 0
        for k in ("logp", "lse", "out", "g", "dh", "dW"):
            assert np.array_equal(checked[k], release[k], equal_nan=True), (name, mode, k)


def test_suite_runs_on_the_library_it_was_asked_for(request):
    # under --bounds-checked every test of the session goes through liborpo_head_debug.so
    lib = orpo.load()
    want = "liborpo_head_debug.so" if request.config.getoption("--bounds-checked") else "liborpo_head.so"
    assert os.path.basename(lib._name) == want
    assert os.path.basename(orpo.lib_path()) == want
