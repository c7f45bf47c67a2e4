"""The library's debug-bounds build (index checks in the kernels that record a
status bit and skip the access, never trap) runs small cases of every entry
point cleanly: parity with the oracle at the usual bars and no failed check.
The build is loaded in a child process (OPAM_LIBRARY), so the normal build
the other tests use is untouched; the child also shows that a deliberately
failed check is reported.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_bounds_build_runs_clean(cuda_lib):
    from outer_product_associative_chunked_b300 import build
    lib = build.build(debug_bounds=True)
    env = dict(os.environ, OPAM_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    print(r.stdout[-3000:])
    assert r.returncode == 0, r.stderr[-3000:]
    assert "all cases clean" in r.stdout
