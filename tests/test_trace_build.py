"""The trace build (libspconv_trace.so, -DSPCONV_TRACE=1): every forward block
records its start, first-stage-ready and pipeline-end times and its SM,
group and group flags, read back through spconv_trace_read; bench.py
--timeline summarises one launch from them.  The default library exports the
same entry point and answers that it does not trace."""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import sparse_weight_direct_gb300 as swd
from sparse_weight_direct_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_default_build_does_not_trace():
    lib = _lib.lib()
    buf = np.zeros(8, dtype=np.uint64)
    assert lib.spconv_trace_read(buf.ctypes.data, buf.nbytes) == _lib.SPCONV_ERR_UNSUPPORTED
    assert lib.spconv_trace_read(None, 64) == _lib.SPCONV_ERR_INVALID_ARG
    assert lib.spconv_trace_read(buf.ctypes.data, -1) == _lib.SPCONV_ERR_INVALID_ARG


def test_trace_build_is_a_separate_library():
    from sparse_weight_direct_gb300 import build as b
    assert b.LIB_TRACE not in (b.LIB, b.LIB_DEBUG) and b.BUILD_TRACE not in (b.BUILD, b.BUILD_DEBUG)
    with pytest.raises(ValueError):
        b.build(debug=True, trace=True)


@pytest.mark.gpu
@pytest.mark.parametrize("config", ["sweep90", "resnet3x3"])
def test_timeline_of_one_launch(config):
    """A child process bound to the trace build times the layer and prints
    the timeline: one record per block, every block started, reached its
    first stage and ended, in that order, within the launch's span; the
    parity helpers' device status stays clear."""
    from sparse_weight_direct_gb300 import build as b
    lib = b.build(trace=True)
    env = dict(os.environ, SPCONV_LIBRARY=lib)
    cmd = [sys.executable, "bench.py", "--timeline", "--config", config, "--steps", "3",
           "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (r.stdout + r.stderr)[-3000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("{")][-1]
    d = json.loads(line)
    assert d["timeline"] == config and d["launches"] == 3
    assert d["blocks"] == d["grid"][0] * d["grid"][1]
    lo, med, hi = d["block_us_min_med_max"]
    assert 0 < lo <= med <= hi <= d["span_us"] < 10000
    ready_med, ready_max = d["first_stage_ready_us_med_max"]
    assert 0 < ready_med <= ready_max <= hi
    assert sum(k["blocks"] for k in d["by_kind"].values()) == d["blocks"]
    assert 1 <= d["peak_running_blocks"] <= d["blocks"]
    assert d["ideal_span_us"] <= d["span_us"] * 1.01
    assert 1 <= d["sms_used"] <= 152 + 8


@pytest.mark.gpu
def test_trace_build_computes_the_same_convolution():
    """The records are a few stores per block: the traced kernel's outputs
    pass the same parity suite as the default build's."""
    from sparse_weight_direct_gb300 import build as b
    lib = b.build(trace=True)
    env = dict(os.environ, SPCONV_LIBRARY=lib)
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_parity.py::test_layer_full_size", "tests/test_parity.py::test_edge_shapes"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0 and " passed" in r.stdout, (r.stdout + r.stderr)[-3000:]
