"""The bounds-checked build (libspconv_debug.so, -DSPCONV_DEBUG=1), the stand-in
for a device memory checker: every staged-tile read, weight-blob range,
shared-memory scratch index, distributed-shared-memory slot and global index
of the kernels is checked against its extent before the access; a failed
check skips the access and sets bit 2 of the handle's device error word
(spconv_device_status), with no trap.

The GPU test builds that library and runs, in a child process bound to it
(SPCONV_LIBRARY), the parity suites that exercise the staging, reduction and
write-back paths at their edges -- edge shapes, heavy and dense rows, empty
rows, both cluster reductions, tap pairs, plane staging, column blocks (one
image and image pairs, 3x3 and 5x5), tight-pitch tiles, the 32-bit word
format, the weight-stationary kernel and the seeded random layers.  Every
GPU helper of those suites asserts that the device error word is clear after
each forward, so a single failed check fails the run; outputs are compared
with the oracle as usual (a skipped access would also show there)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SUITES = [
    "tests/test_parity.py::test_edge_shapes",
    "tests/test_parity.py::test_heavy_rows_split_and_dense",
    "tests/test_parity.py::test_empty_rows_and_empty_matrix",
    "tests/test_parity.py::test_cluster_reduction_paths",
    "tests/test_parity.py::test_tap_pairs",
    "tests/test_parity.py::test_plane_staging",
    "tests/test_parity.py::test_column_blocks",
    "tests/test_parity.py::test_image_pair_column_blocks",
    "tests/test_parity.py::test_image_pair_5x5",
    "tests/test_parity.py::test_tight_pitch",
    "tests/test_parity.py::test_packed32_format",
    "tests/test_ws.py",
    "tests/test_random_shapes.py",
]


def test_debug_build_is_a_separate_library():
    """The checks live only in the debug build: the default library is built
    from the same sources without the macro, into its own objects."""
    from sparse_weight_direct_gb300 import build as b
    assert b.LIB_DEBUG != b.LIB and b.BUILD_DEBUG != b.BUILD
    src = open(os.path.join(b.CSRC, "spconv_kernel.cuh")).read()
    assert "#ifdef SPCONV_DEBUG" in src and "kErrBounds = 4u" in src


@pytest.mark.gpu
def test_bounds_checked_build_runs_the_edge_suites_clean():
    from sparse_weight_direct_gb300 import build as b
    lib = b.build(debug=True)
    assert os.path.exists(lib)
    env = dict(os.environ, SPCONV_LIBRARY=lib)
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           *SUITES]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
