"""The parity suites run against the bounds-checked build of the library.

That build (LSDRS_CHECKED=1) tests every shared and global index of the
scatter, histogram and one-kernel sorts before the access and records a
failed test in the scratch header instead of performing the access; the
binding raises BoundsViolation when a sort recorded one.  It stands in for
memory checkers: the parity suites must pass against it with no recorded
failure, the outputs still equal to the oracle's.
"""
import os
import subprocess
import sys

import pytest

from tests.conftest import ROOT

pytestmark = pytest.mark.gpu

SUITES = ["tests/test_gpu_parity.py", "tests/test_gpu_small.py", "tests/test_gpu_typed.py",
          "tests/test_gpu_skip.py", "tests/test_gpu_rows_shapes.py", "tests/test_gpu_options.py"]


def test_parity_suites_record_no_bounds_violation(tmp_path):
    lib = tmp_path / "liblsdrs_checked.so"
    subprocess.run([sys.executable, "-m", "lsd_radix_sort_gb300.build", "--out", str(lib),
                    "-D", "LSDRS_CHECKED=1"], cwd=ROOT, check=True, capture_output=True)
    env = dict(os.environ, LSDRS_LIB=str(lib))
    probe = subprocess.run(
        [sys.executable, "-c",
         "import lsd_radix_sort_gb300 as rs; print(int(rs.checked_build()))"],
        cwd=ROOT, env=env, capture_output=True, text=True, check=True)
    assert probe.stdout.strip() == "1", "the checked build was not the library loaded"
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
                        "-p", "no:cacheprovider", *SUITES],
                       cwd=ROOT, env=env, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
