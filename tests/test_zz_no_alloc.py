"""spconv_forward_host_noalloc: the host-buffer forward for callers that must
not allocate device memory when they run a layer (a plugin whose framework's
allocator owns the GPU's memory, a service with a fixed memory budget, a
latency-critical caller that cannot take cudaMalloc's implicit
synchronisation).  Its device workspaces are one array the library declares
statically, so these tests check, through the C ABI, that two calls in a row
give what spconv_forward_host gives with caller-provided workspaces, and that
a layer too large for the array is refused before anything runs.

(The file name sorts last, so a run that stops at its first failure has run
every other test before this one.)"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads
import sparse_weight_direct_gb300 as swd
from sparse_weight_direct_gb300 import _lib

MAX_BYTES = 32 << 20  # SPCONV_NOALLOC_MAX_BYTES


def _args(L, N):
    return (N, L.C, L.H, L.W, L.M, L.R, L.S, L.stride, L.pad)


def test_noalloc_rejects_a_layer_too_large_for_its_workspace():
    """The VGG-style layer (N=16: 25.7 MB in, 25.7 MB out) does not fit in
    32 MiB; the call says so without touching a GPU (host-only handle)."""
    L = workloads.LAYERS["vgg3x3"]
    assert 4 * L.N * (L.C * L.H * L.W + L.M * L.E * L.F) > MAX_BYTES
    rowptr, colidx, value = workloads.make_weights(L)
    w = swd.pack_host(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                      stride=L.stride, pad=L.pad)
    rc = _lib.lib().spconv_forward_host_noalloc(*_args(L, L.N), None, w.handle, None, 0, None,
                                                None)
    assert rc == _lib.SPCONV_ERR_UNSUPPORTED
    # a non-positive shape argument is an argument error
    rc = _lib.lib().spconv_forward_host_noalloc(L.N, 0, L.H, L.W, L.M, L.R, L.S, L.stride,
                                                L.pad, None, w.handle, None, 0, None, None)
    assert rc == _lib.SPCONV_ERR_INVALID_ARG
    w.close()


@pytest.mark.gpu
@pytest.mark.parametrize("name,pinned", [("resnet3x3", True), ("sweep90", True),
                                         ("sweep90", False)])
def test_noalloc_matches_host_forward_twice(name, pinned):
    """Two calls in a row on different inputs, each compared element by
    element with spconv_forward_host on the same input (caller-provided
    workspaces), under the parity rule |a - b| <= 1e-5 * sum|w x| + 1e-7.
    The one-image layer's Y (0.2 MB) goes straight to the host buffer; the
    sweep layer's (12.8 MB) goes through the array's output region.  Page-
    locked buffers take the mapped path, pageable ones the copy path."""
    import torch
    L = workloads.LAYERS[name]
    N = L.N
    rowptr, colidx, value = workloads.make_weights(L)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad, batch_hint=N)
    lib = _lib.lib()
    stream = torch.cuda.Stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    xd = torch.empty((N, L.C, L.H, L.W), device="cuda")
    yd = torch.empty((N, L.M, L.E, L.F), device="cuda")
    rng = np.random.default_rng(99)
    for call in range(2):
        x = workloads.make_input(L) if call == 0 else \
            workloads.random_input((N, L.C, L.H, L.W), rng)
        xh = torch.from_numpy(np.ascontiguousarray(x))
        want = torch.full((N, L.M, L.E, L.F), float("nan"))
        got = torch.full((N, L.M, L.E, L.F), float("nan"))
        if pinned:
            xh, want, got = xh.pin_memory(), want.pin_memory(), got.pin_memory()
        torch.cuda.synchronize()
        rc = lib.spconv_forward_host(*_args(L, N), ctypes.c_void_p(xh.data_ptr()), w.handle,
                                     None, 0, ctypes.c_void_p(want.data_ptr()),
                                     ctypes.c_void_p(xd.data_ptr()),
                                     ctypes.c_void_p(yd.data_ptr()), sp)
        assert rc == _lib.SPCONV_OK
        rc = lib.spconv_forward_host_noalloc(*_args(L, N), ctypes.c_void_p(xh.data_ptr()),
                                             w.handle, None, 0,
                                             ctypes.c_void_p(got.data_ptr()), sp)
        assert rc == _lib.SPCONV_OK, swd.status_string(rc)
        stream.synchronize()
        assert w.device_status(stream) == 0
        a = got.numpy().astype(np.float64)
        b = want.numpy().astype(np.float64)
        assert np.isfinite(a).all() and np.isfinite(b).all()
        _, mag = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
        bad = ~(np.abs(a - b) <= 1e-5 * mag + 1e-7)
        assert not bad.any(), f"call {call}: {int(bad.sum())} of {bad.size} outputs differ"
    w.close()
