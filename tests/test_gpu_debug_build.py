"""The -DMUON_DEBUG build (libmuon_debug.so): its kernels check every tiled
TMA copy's innermost coordinate, the GEMM tiles' matrix, tile, split and
K-block indices, the split-K partial slots and the streaming kernels'
element ranges, and report a failed check as MUON_ERR_BOUNDS.  One case per
kernel (tests/debug_cases.py) runs in a process of its own under each
library: no call may report a status, and the results must agree bit for
bit (the checks guard accesses, they never change arithmetic)."""
import os
import subprocess
import sys
import time

import numpy as np
import pytest

from newton_schulz_gb300 import build

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def _run(tmp_path, name, lib):
    out = str(tmp_path / f"{name}.npz")
    env = dict(os.environ, MUON_LIB_PATH=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_cases.py"), out], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    return np.load(out)


def test_debug_build_checks_pass_and_match_release(tmp_path, cuda_ok):
    t0 = time.time()
    debug_lib = build.build(debug=True)
    print(f"debug build: {time.time() - t0:.1f} s")
    rel = _run(tmp_path, "release", build.LIB)
    dbg = _run(tmp_path, "debug", debug_lib)
    assert int(rel["debug_build"]) == 0 and int(dbg["debug_build"]) == 1
    names = list(dbg["names"])
    assert list(rel["names"]) == names
    for n, code_r, code_d in zip(names, rel["codes"], dbg["codes"]):
        assert code_d == 0 and code_r == 0, (n, int(code_r), int(code_d))
    meta = ("names", "codes", "debug_build")
    keys = sorted(k for k in rel.files if k not in meta)
    assert keys == sorted(k for k in dbg.files if k not in meta)
    for k in keys:
        assert np.array_equal(rel[k], dbg[k], equal_nan=True), k
