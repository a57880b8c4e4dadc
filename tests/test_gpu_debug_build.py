"""The bounds-checking build (liblce_debug.so: the same sources compiled with
LCE_DEBUG) under the GPU parity tests of small shapes.  In that build every
kernel checks the indices it computes -- row maps, sorted label keys,
labels, chunk rows, partial and workspace offsets -- and the coordinates of
its TMA copies against the buffers they address; a check that fails skips
the access and raises LCE_ERR_BOUNDS in the call's status word.  The parity
tests assert LCE_OK after every call and check guard bytes around every
output, so any out-of-range index in these paths fails them.  This stands in
for a memory checker, which is not available here.  The tests run in a child
process that loads the debug library (LCE_LIBRARY=debug)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ["tests/test_gpu_parity.py", "tests/test_gpu_peaked.py", "tests/test_gpu_options.py",
         "tests/test_gpu_random_shapes.py", "tests/test_gpu_extremes.py", "tests/test_gpu_gradx_tail.py"]


def test_child_process_loads_the_debug_library():
    from lm_head_linear_chunked_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, LCE_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", "import lm_head_linear_chunked_gb300 as l; l.lib(); print(l.library_path)"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().endswith("liblce_debug.so")


def test_parity_tests_pass_on_the_bounds_checking_build():
    from lm_head_linear_chunked_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, LCE_LIBRARY="debug")
    env.pop("LCE_PARITY_REPORT", None)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *FILES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout
