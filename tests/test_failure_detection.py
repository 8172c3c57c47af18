"""Failure detection without a GPU fault.

The forward kernel's copy-pipeline waits are bounded by a timer; on expiry
the kernel records a flag and returns instead of hanging.  These tests make
such a wait run out on purpose (a barrier nothing completes, 20 ms limit) and
check that the status reaches the host and the context stays usable, and that
a clean forward leaves the handle's device error word clear.
"""
import ctypes

import numpy as np
import pytest

import workloads
import sparse_weight_direct_gb300 as swd
from sparse_weight_direct_gb300 import _lib

torch = pytest.importorskip("torch")


@pytest.mark.gpu
def test_bounded_wait_times_out_and_reports():
    L = _lib.lib()
    flags = ctypes.c_int32(0)
    rc = L.spconv_selftest_wait(0, None, ctypes.byref(flags))
    assert rc == _lib.SPCONV_ERR_DEVICE
    assert flags.value & 1 and not flags.value & 2
    # the context is still usable: a completed wait, then a real forward
    rc = L.spconv_selftest_wait(1, None, ctypes.byref(flags))
    assert rc == _lib.SPCONV_OK and flags.value == 2
    lay = workloads.LAYERS["tiny"]
    rowptr, colidx, value = workloads.make_weights(lay)
    w = swd.pack(rowptr, colidx, value, C=lay.C, H=lay.H, W=lay.W, M=lay.M, R=lay.R, S=lay.S,
                 stride=lay.stride, pad=lay.pad)
    y = swd.forward(torch.from_numpy(workloads.make_input(lay)).cuda(), w)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    assert w.device_status() == 0
    w.close()


@pytest.mark.gpu
def test_selftest_rejects_null_flags():
    assert _lib.lib().spconv_selftest_wait(0, None, None) == _lib.SPCONV_ERR_INVALID_ARG


def test_device_status_rejects_host_only_handle():
    w = swd.pack_host(np.array([0, 1], np.int32), np.array([4], np.int32),
                      np.array([1.0], np.float32), C=1, H=5, W=5, M=1, R=3, S=3, stride=1, pad=1)
    flags = ctypes.c_int32(0)
    rc = _lib.lib().spconv_device_status(w.handle, None, ctypes.byref(flags))
    assert rc == _lib.SPCONV_ERR_INVALID_ARG
    w.close()
