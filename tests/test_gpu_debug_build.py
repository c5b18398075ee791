"""The GQ_DEBUG build of the library (GPU only).

That build compiles the same kernels with device-side checks of the indices they derive from
their arguments; a failed check records GQ_ERR_DEVICE_CHECK in the device status word and the
kernel goes on (nothing traps).  This test builds it beside the normal library, runs every kernel
family through it in a child process (tests/debug_build_checks.py, which loads the build named by
GQ_LIBRARY) and requires correct results and a clean status word.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_runs_clean():
    from quantized_skinny_matmul_gb300 import _build
    path = _build.build(debug=True)
    env = dict(os.environ, GQ_LIBRARY=path)
    res = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_checks.py")], env=env,
                         capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "debug build clean" in res.stdout
