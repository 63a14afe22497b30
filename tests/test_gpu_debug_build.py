"""The bounds-checked build (BD_DEBUG), the stand-in for a memory checker.

compute-sanitizer is closed on this machine, so the library can be built with every
kernel checking the indices of its global accesses against the extents it was
given (a failed check skips the access and records BD_ERR_DEVICE_BOUNDS in the
device status word; nothing traps).  This test builds that variant and runs small
cases of every kernel family through it in a child process (so that the debug
library is the one loaded), each against the oracle and with the status word
read after every call."""
import os
import subprocess
import sys

import pytest

from bit_delta_tenant_gb300 import build as lib_build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_every_kernel_family_passes_its_bounds_checks():
    path = lib_build.build(debug=True)
    assert path.endswith("libbitdelta_debug.so")
    res = subprocess.run([sys.executable, os.path.join(HERE, "debug_child.py")], capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "debug build ok" in res.stdout
