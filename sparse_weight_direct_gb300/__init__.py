"""sparse_weight_direct_gb300 -- direct 2-D convolution with unstructured-sparse
weights on GB300 (sm_103a).

The whole computation runs in ``libspconv.so`` (hand-written CUDA behind the C
ABI of ``include/spconv.h``).  This package only marshals arguments: it passes
raw pointers, sizes and a stream to the library.  PyTorch provides device
memory and streams; no step of the convolution runs in Python or PyTorch, and
there is no CPU fallback -- if the library is missing, every call raises.

    from sparse_weight_direct_gb300 import pack, forward
    w = pack(rowptr, colidx, value, C=..., H=..., W=..., M=..., R=3, S=3,
             stride=1, pad=1)
    y = forward(x_cuda, w)            # x: (N, C, H, W) float32 on the GPU
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib
from ._lib import SpconvError, status_string

__all__ = ["pack", "pack_host", "forward", "forward_host", "PackedWeights", "SpconvError", "status_string",
           "out_extent", "library_path"]


def library_path() -> str:
    return _lib.LIB_PATH


def out_extent(size: int, k: int, stride: int, pad: int) -> int:
    """Output extent, floor((size + 2*pad - k) / stride) + 1."""
    return (size + 2 * pad - k) // stride + 1


class PackedWeights:
    """Owner of a ``spconv_packed`` handle (freed on close / garbage collection)."""

    def __init__(self, handle: ctypes.c_void_p, shape: dict):
        self._h = handle
        self.shape = shape  # C, H, W, M, R, S, stride, pad

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise SpconvError(_lib.SPCONV_ERR_INVALID_ARG, "packed weights already freed")
        return self._h

    def info(self) -> dict:
        info = _lib.PackedInfo()
        _lib.check(_lib.lib().spconv_packed_info_get(self.handle, ctypes.byref(info)),
                   "spconv_packed_info_get")
        return {name: getattr(info, name) for name, _ in _lib.PackedInfo._fields_}

    def launch_info(self, N: int) -> dict:
        """How a forward of N images would launch (grid, cluster size, reduction
        mode, shared memory, staging path, kernel); host logic only."""
        info = _lib.LaunchInfo()
        _lib.check(_lib.lib().spconv_launch_info_get(self.handle, int(N), ctypes.byref(info)),
                   "spconv_launch_info_get")
        return {name: getattr(info, name) for name, _ in _lib.LaunchInfo._fields_}

    def array(self, which: str) -> np.ndarray:
        """Copy of a packed host array: 'blobs' (raw bytes), 'blob_off'
        (uint32, 16-byte units), 'slot_oc', 'slot_next' or 'group_flags' (int32)."""
        code = {"blobs": 0, "blob_off": 1, "slot_oc": 2, "slot_next": 3, "group_flags": 4}[which]
        need = ctypes.c_int64(0)
        L = _lib.lib()
        _lib.check(L.spconv_packed_copy_array(self.handle, code, None, 0, ctypes.byref(need)),
                   "spconv_packed_copy_array")
        if which == "blobs":
            out = np.zeros(need.value, dtype=np.uint8)
        elif which == "blob_off":
            out = np.zeros(need.value // 4, dtype=np.uint32)
        else:
            out = np.zeros(need.value // 4, dtype=np.int32)
        _lib.check(L.spconv_packed_copy_array(self.handle, code, out.ctypes.data_as(ctypes.c_void_p),
                                              out.nbytes, None), "spconv_packed_copy_array")
        return out

    def device_status(self, stream=None) -> int:
        """Synchronise the stream and read/clear the device error flags
        (0 = clean; bit 0 = a pipeline wait of the forward kernel timed out;
        bit 1 = the wait for the block's copies in flight after that timeout
        ran out too: the context is then suspect and should be reset;
        bit 2 = bounds-checked build only: an access failed its check and was
        skipped)."""
        flags = ctypes.c_int32(0)
        rc = _lib.lib().spconv_device_status(self.handle, _stream_ptr(stream), ctypes.byref(flags))
        if rc not in (_lib.SPCONV_OK, _lib.SPCONV_ERR_DEVICE):
            _lib.check(rc, "spconv_device_status")
        return int(flags.value)

    def close(self) -> None:
        if self._h:
            _lib.lib().spconv_packed_free(self._h)
            self._h = None

    def __del__(self):  # pragma: no cover - best effort
        try:
            self.close()
        except Exception:
            pass


def _csr_arrays(rowptr, colidx, value):
    rowptr = np.ascontiguousarray(np.asarray(rowptr, dtype=np.int32))
    colidx = np.ascontiguousarray(np.asarray(colidx, dtype=np.int32))
    value = np.ascontiguousarray(np.asarray(value, dtype=np.float32))
    return rowptr, colidx, value


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


FORMATS = {"f32": 0, "packed32": 1, "ws": 2}


def _pack(rowptr, colidx, value, C, H, W, M, R, S, stride, pad, fmt, batch_hint, host_only,
          stream):
    rowptr, colidx, value = _csr_arrays(rowptr, colidx, value)
    if rowptr.size != M + 1:
        raise SpconvError(_lib.SPCONV_ERR_INVALID_ARG, "rowptr must have M + 1 entries")
    h = ctypes.c_void_p()
    _lib.check(_lib.lib().spconv_pack_ex(C, H, W, M, R, S, stride, pad, _ptr(rowptr),
                                         _ptr(colidx), _ptr(value), FORMATS[fmt],
                                         int(batch_hint), 1 if host_only else 0,
                                         None if host_only else _stream_ptr(stream),
                                         ctypes.byref(h)), "spconv_pack_ex")
    return PackedWeights(h, dict(C=C, H=H, W=W, M=M, R=R, S=S, stride=stride, pad=pad))


def pack(rowptr, colidx, value, *, C: int, H: int, W: int, M: int, R: int, S: int,
         stride: int = 1, pad: int = 0, stream=None, fmt: str = "f32",
         batch_hint: int = 0) -> PackedWeights:
    """CSR (host arrays) -> packed device layout on the current CUDA device.
    fmt: "f32" (fp32 values, precomputed offsets), "packed32" (the first page's
    32-bit words with FP16 values) or "ws" (weight-stationary: one output
    channel per block, input read in place; Escoin, Figs. 5-7).  batch_hint:
    the batch size the forwards will mostly use (0 = unknown); it only shapes
    the tiling plan."""
    return _pack(rowptr, colidx, value, C, H, W, M, R, S, stride, pad, fmt, batch_hint, False,
                 stream)


def pack_host(rowptr, colidx, value, *, C: int, H: int, W: int, M: int, R: int, S: int,
              stride: int = 1, pad: int = 0, fmt: str = "f32",
              batch_hint: int = 0) -> PackedWeights:
    """The same packing kept in host memory only (inspection; needs no GPU)."""
    return _pack(rowptr, colidx, value, C, H, W, M, R, S, stride, pad, fmt, batch_hint, True,
                 None)


def _stream_ptr(stream):
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def forward(x, packed: PackedWeights, out=None, stream=None, bias=None, relu: bool = False):
    """Y = conv(x, packed) on the GPU.  x: (N, C, H, W) contiguous float32
    CUDA tensor; out (optional): (N, M, E, F) float32 CUDA tensor, overwritten.
    bias (optional): (M,) float32 CUDA tensor added in the kernel's write-back;
    relu: apply max(y, 0) there too.  Asynchronous on ``stream`` (default: the
    current torch stream)."""
    import torch
    sh = packed.shape
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32
            and x.dim() == 4 and x.is_contiguous()):
        raise SpconvError(_lib.SPCONV_ERR_INVALID_ARG,
                          "x must be a contiguous 4-D float32 CUDA tensor")
    N = x.shape[0]
    E = out_extent(sh["H"], sh["R"], sh["stride"], sh["pad"])
    F = out_extent(sh["W"], sh["S"], sh["stride"], sh["pad"])
    if out is None:
        out = torch.empty((N, sh["M"], E, F), device=x.device, dtype=torch.float32)
    elif not (out.is_cuda and out.dtype == torch.float32 and out.is_contiguous()
              and tuple(out.shape) == (N, sh["M"], E, F)):
        raise SpconvError(_lib.SPCONV_ERR_INVALID_ARG, "out has the wrong shape/dtype/layout")
    if bias is None and not relu:
        rc = _lib.lib().spconv_forward(N, x.shape[1], x.shape[2], x.shape[3], sh["M"], sh["R"],
                                       sh["S"], sh["stride"], sh["pad"],
                                       ctypes.c_void_p(x.data_ptr()), packed.handle,
                                       ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream))
        _lib.check(rc, "spconv_forward")
        return out
    if bias is not None and not (bias.is_cuda and bias.dtype == torch.float32
                                 and bias.is_contiguous() and bias.numel() == sh["M"]):
        raise SpconvError(_lib.SPCONV_ERR_INVALID_ARG, "bias must be M contiguous float32 on the GPU")
    rc = _lib.lib().spconv_forward_ex(N, x.shape[1], x.shape[2], x.shape[3], sh["M"], sh["R"],
                                      sh["S"], sh["stride"], sh["pad"],
                                      ctypes.c_void_p(x.data_ptr()), packed.handle,
                                      ctypes.c_void_p(bias.data_ptr() if bias is not None else 0),
                                      1 if relu else 0, ctypes.c_void_p(out.data_ptr()),
                                      _stream_ptr(stream))
    _lib.check(rc, "spconv_forward_ex")
    return out


def forward_host(x_host, packed: PackedWeights, out_host, x_dev, out_dev, stream=None, bias=None,
                 relu: bool = False):
    """Y = conv(x_host, packed) with the activation and the result in host
    memory (spconv_forward_host): one call enqueues the copy of x_host into
    the device workspace x_dev, the forward into out_dev and the copy of
    out_dev into out_host, in that order on ``stream``.  x_host: (N, C, H, W)
    and out_host: (N, M, E, F) contiguous float32 CPU tensors in page-locked
    memory; x_dev / out_dev: CUDA tensors of the same shapes.  Asynchronous:
    out_host holds Y once the stream has passed this work."""
    import torch
    sh = packed.shape
    N = x_host.shape[0] if isinstance(x_host, torch.Tensor) and x_host.dim() == 4 else -1
    E = out_extent(sh["H"], sh["R"], sh["stride"], sh["pad"])
    F = out_extent(sh["W"], sh["S"], sh["stride"], sh["pad"])
    in_shape = (N, sh["C"], sh["H"], sh["W"])
    out_shape = (N, sh["M"], E, F)
    for t, shape, cuda, what in ((x_host, in_shape, False, "x_host"),
                                 (out_host, out_shape, False, "out_host"),
                                 (x_dev, in_shape, True, "x_dev"),
                                 (out_dev, out_shape, True, "out_dev")):
        if not (isinstance(t, torch.Tensor) and t.dtype == torch.float32 and t.is_contiguous()
                and t.is_cuda == cuda and tuple(t.shape) == shape):
            raise SpconvError(_lib.SPCONV_ERR_INVALID_ARG,
                              f"{what} must be a contiguous float32 {'CUDA' if cuda else 'CPU'} "
                              f"tensor of shape {shape}")
        if not cuda and not t.is_pinned():
            raise SpconvError(_lib.SPCONV_ERR_INVALID_ARG, f"{what} must be in page-locked memory")
    if bias is not None and not (bias.is_cuda and bias.dtype == torch.float32
                                 and bias.is_contiguous() and bias.numel() == sh["M"]):
        raise SpconvError(_lib.SPCONV_ERR_INVALID_ARG, "bias must be M contiguous float32 on the GPU")
    rc = _lib.lib().spconv_forward_host(
        N, sh["C"], sh["H"], sh["W"], sh["M"], sh["R"], sh["S"], sh["stride"], sh["pad"],
        ctypes.c_void_p(x_host.data_ptr()), packed.handle,
        ctypes.c_void_p(bias.data_ptr() if bias is not None else 0), 1 if relu else 0,
        ctypes.c_void_p(out_host.data_ptr()), ctypes.c_void_p(x_dev.data_ptr()),
        ctypes.c_void_p(out_dev.data_ptr()), _stream_ptr(stream))
    _lib.check(rc, "spconv_forward_host")
    return out_host
