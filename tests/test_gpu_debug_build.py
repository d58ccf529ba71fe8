"""The guard-band suite (tests/test_gpu_canaries.py) again, against the debug build of the library
(libgq_debug.so: the same sources with -DGQ_DEBUG, whose kernels check every store and bulk copy
against its buffer's logical extent and record a failure instead of trapping).  Every call must
leave the guard bands intact and the debug word at 0.  The normal build reports -1 (no checks
compiled in)."""
import os
import subprocess
import sys

import pytest

from gpu_common import gq_module

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_normal_build_has_no_checks():
    gq = gq_module()
    if os.environ.get("GQ_LIBRARY"):
        pytest.skip("running against another build")
    assert gq.gq_debug_status() == -1


def test_canaries_under_the_debug_build():
    gq_module()  # skips without a GPU
    from allreduce_compatible_gradient_gb300 import _build
    lib = _build.build_library(debug=True)
    env = dict(os.environ, GQ_LIBRARY=lib, GQ_EXPECT_DEBUG="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
                        os.path.join(ROOT, "tests", "test_gpu_canaries.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
