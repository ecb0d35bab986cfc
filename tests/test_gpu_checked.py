"""The parity suites again, on the bounds-checked build.

The checked library tests every load and store of the flush kernels against
the task it belongs to, records DPRED_E_BOUNDS for any access outside it and
skips that access.  Here it is built, and the flush, fuzz, executor,
partitioned and collective suites run against it in a child process.  They
must all pass (results equal to the oracle's), and the device error word must
still be 0 when the session ends: no kernel access left its task on any of
these cases."""
import os
import subprocess
import sys

import pytest

from tests.conftest import ROOT

pytestmark = pytest.mark.gpu

SUITES = ["tests/test_gpu_flush.py", "tests/test_gpu_fuzz.py", "tests/test_gpu_executor.py",
          "tests/test_gpu_partitioned.py", "tests/test_gpu_collectives.py", "tests/test_gpu_status.py"]


def test_parity_suites_on_the_checked_build():
    sys.path.insert(0, ROOT)
    from zero_collectives_gb300 import build
    build.build(checked=True)
    env = dict(os.environ, DPRED_CHECKED="1")
    probe = subprocess.run([sys.executable, "-c", "import zero_collectives_gb300 as zc; print(zc.checked_build())"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.stdout.strip() == "True", probe.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITES, "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider",
                        "-p", "tests.status_plugin"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
