"""spconv_forward_host: the forward with the activation and the result in host
memory (copy in, forward, copy out, enqueued by one call).  GPU cases compare
its result with the oracle under the usual rule (bit-exact on integer-valued
layers, else |gpu - oracle| <= 1e-5 * sum|w*x| + 1e-7) and with the device
forward of the same inputs (identical bits: the same kernel on the same data).
CPU cases check the argument errors that need no device."""
import ctypes
import dataclasses

import numpy as np
import pytest

import oracle
import workloads
import sparse_weight_direct_gb300 as swd
from sparse_weight_direct_gb300 import _lib

torch = pytest.importorskip("torch")
P = ctypes.c_void_p


def _tiny_host_handle():
    return swd.pack_host(np.array([0, 1], np.int32), np.array([4], np.int32),
                         np.array([1.0], np.float32), C=1, H=5, W=5, M=1, R=3, S=3, stride=1, pad=1)


def test_rejects_host_only_handle_and_null_handle():
    L = _lib.lib()
    w = _tiny_host_handle()
    args = (1, 1, 5, 5, 1, 3, 3, 1, 1)
    rc = L.spconv_forward_host(*args, None, w.handle, None, 0, None, None, None, None)
    assert rc == _lib.SPCONV_ERR_MISMATCH
    rc = L.spconv_forward_host(*args, None, None, None, 0, None, None, None, None)
    assert rc == _lib.SPCONV_ERR_INVALID_ARG
    rc = L.spconv_forward_host(*args, None, w.handle, None, 5, None, None, None, None)
    assert rc == _lib.SPCONV_ERR_INVALID_ARG  # unknown activation
    w.close()


def test_binding_checks_tensors():
    w = _tiny_host_handle()
    x = torch.zeros((1, 1, 5, 5))
    y = torch.zeros((1, 1, 5, 5))
    with pytest.raises(swd.SpconvError):  # device workspaces must be CUDA tensors
        swd.forward_host(x, w, y, x, y)
    with pytest.raises(swd.SpconvError):
        swd.forward_host(x.double(), w, y, x, y)
    with pytest.raises(swd.SpconvError):
        swd.forward_host(x[:, :, :4], w, y, x, y)
    w.close()


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).pin_memory()


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "resnet3x3", "vgg3x3", "sweep99", "alex11x11",
                                  "conv5x5"])
@pytest.mark.parametrize("integer", [False, True])
def test_forward_host_parity(name, integer):
    L = dataclasses.replace(workloads.LAYERS[name], integer=integer)
    N = min(L.N, 2)
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L, N)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad, batch_hint=N)
    xh = _pinned(x)
    yh = torch.full((N, L.M, L.E, L.F), float("nan")).pin_memory()
    xd = torch.empty(xh.shape, device="cuda")
    yd = torch.empty(yh.shape, device="cuda")
    s = torch.cuda.Stream()
    yd.fill_(float("nan"))
    # the fill runs on the current stream, the forward on s: order them
    s.wait_stream(torch.cuda.current_stream())
    swd.forward_host(xh, w, yh, xd, yd, stream=s)
    s.synchronize()
    # page-locked buffers from torch are mapped on the device: the input went
    # through the copy kernel; a Y of at most 1 MiB went straight into the host
    # buffer (the device output workspace was never written), a larger one
    # through the workspace
    if yh.numel() * 4 <= 1 << 20:
        assert torch.isnan(yd).all()
    else:
        np.testing.assert_array_equal(yd.cpu().numpy(), yh.numpy())
    got = yh.numpy().astype(np.float64)
    ref, mag = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
    if integer:
        np.testing.assert_array_equal(got, ref)
    else:
        bad = ~(np.abs(got - ref) <= 1e-5 * mag + 1e-7)
        assert not bad.any(), f"{int(bad.sum())} of {bad.size} outputs off"
    y_dev = swd.forward(torch.from_numpy(x).cuda(), w)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y_dev.cpu().numpy(), yh.numpy())
    w.close()


@pytest.mark.gpu
@pytest.mark.parametrize("relu", [False, True])
def test_forward_host_bias_relu(relu):
    L = dataclasses.replace(workloads.LAYERS["resnet3x3"], integer=True)
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L, 1)
    bias = np.random.default_rng(5).integers(-20, 21, L.M).astype(np.float32)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad, batch_hint=1)
    xh = _pinned(x)
    yh = torch.empty((1, L.M, L.E, L.F)).pin_memory()
    xd = torch.empty(xh.shape, device="cuda")
    yd = torch.empty(yh.shape, device="cuda")
    swd.forward_host(xh, w, yh, xd, yd, bias=torch.from_numpy(bias).cuda(), relu=relu)
    torch.cuda.synchronize()
    ref, _ = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
    ref = ref + bias.astype(np.float64).reshape(1, -1, 1, 1)
    if relu:
        ref = np.maximum(ref, 0.0)
    np.testing.assert_array_equal(yh.numpy().astype(np.float64), ref)
    w.close()


@pytest.mark.gpu
def test_forward_host_argument_errors():
    L = workloads.LAYERS["tiny"]
    rowptr, colidx, value = workloads.make_weights(L)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad)
    lib = _lib.lib()
    xh = torch.zeros((1, L.C, L.H, L.W)).pin_memory()
    yh = torch.zeros((1, L.M, L.E, L.F)).pin_memory()
    xd = torch.zeros(xh.shape, device="cuda")
    yd = torch.zeros(yh.shape, device="cuda")
    args = (1, L.C, L.H, L.W, L.M, L.R, L.S, L.stride, L.pad)
    ptrs = dict(xh=P(xh.data_ptr()), yh=P(yh.data_ptr()), xd=P(xd.data_ptr()),
                yd=P(yd.data_ptr()))

    def call(a=args, **kw):
        q = {**ptrs, **kw}
        return lib.spconv_forward_host(*a, q["xh"], w.handle, None, 0, q["yh"], q["xd"],
                                       q["yd"], None)

    assert call() == 0
    torch.cuda.synchronize()
    assert call(xh=None) == _lib.SPCONV_ERR_INVALID_ARG
    assert call(yh=None) == _lib.SPCONV_ERR_INVALID_ARG
    assert call(yd=None) == _lib.SPCONV_ERR_INVALID_ARG
    assert call(xd=P(xd.data_ptr() + 4)) == _lib.SPCONV_ERR_INVALID_ARG  # not 16-byte aligned
    assert call(yd=P(xd.data_ptr())) == _lib.SPCONV_ERR_INVALID_ARG      # workspaces overlap
    assert call(yh=P(xh.data_ptr())) == _lib.SPCONV_ERR_INVALID_ARG      # host buffers overlap
    bad = (1, L.C, L.H + 1, L.W, L.M, L.R, L.S, L.stride, L.pad)
    assert call(a=bad) == _lib.SPCONV_ERR_MISMATCH
    # N = 0: nothing to do, nothing read
    assert call(a=(0,) + args[1:], xh=None, yh=None, xd=None, yd=None) == 0
    torch.cuda.synchronize()
    w.close()


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["resnet3x3", "sweep99"])
def test_forward_host_pageable_takes_copy_path(name):
    """Pageable host buffers (numpy arrays) are not mapped on the device: the
    call copies with cudaMemcpyAsync and runs the forward into dev_output."""
    L = dataclasses.replace(workloads.LAYERS[name], integer=True)
    N = 1
    rowptr, colidx, value = workloads.make_weights(L)
    x = np.ascontiguousarray(workloads.make_input(L, N), np.float32)
    y = np.full((N, L.M, L.E, L.F), np.nan, np.float32)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad, batch_hint=N)
    xd = torch.empty(x.shape, device="cuda")
    yd = torch.full(y.shape, float("nan"), device="cuda")
    rc = _lib.lib().spconv_forward_host(N, L.C, L.H, L.W, L.M, L.R, L.S, L.stride, L.pad,
                                        P(x.ctypes.data), w.handle, None, 0, P(y.ctypes.data),
                                        P(xd.data_ptr()), P(yd.data_ptr()), None)
    assert rc == 0
    torch.cuda.synchronize()
    ref, _ = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
    np.testing.assert_array_equal(y.astype(np.float64), ref)
    np.testing.assert_array_equal(yd.cpu().numpy(), y)  # the copy path went through dev_output
    w.close()
