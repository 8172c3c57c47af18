"""Fused epilogue (bias + ReLU in the write-back, spconv_forward_ex) and layer
chaining, against the oracle's convolution followed by the same bias and
activation written out here (y = max(conv + b, 0)).

Tolerance: |gpu - ref| <= 1e-5 * (sum|w*x| + |b|) + 1e-7 (ReLU is
1-Lipschitz, so the bound carries through it); integer-valued cases exact.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads
import sparse_weight_direct_gb300 as swd
from sparse_weight_direct_gb300 import _lib

torch = pytest.importorskip("torch")


def _ref(x, rowptr, colidx, value, L, bias, relu):
    y, mag = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
    y = y + np.asarray(bias, np.float64).reshape(1, -1, 1, 1)
    if relu:
        y = np.maximum(y, 0.0)
    return y, mag + np.abs(np.asarray(bias, np.float64)).reshape(1, -1, 1, 1)


def _check(got, ref, mag, exact):
    if exact:
        np.testing.assert_array_equal(got, ref)
    else:
        bad = ~(np.abs(got - ref) <= 1e-5 * mag + 1e-7)
        assert not bad.any(), f"{int(bad.sum())} outputs off"


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "resnet3x3", "vgg3x3", "sweep95", "sweep50",
                                  "conv5x5"])
@pytest.mark.parametrize("relu", [False, True])
@pytest.mark.parametrize("integer", [False, True])
def test_bias_relu_epilogue(name, relu, integer):
    import dataclasses
    L = dataclasses.replace(workloads.LAYERS[name], integer=integer)
    N = min(L.N, 2)
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L, N)
    rng = np.random.default_rng(3)
    bias = (rng.integers(-20, 21, L.M) if integer else rng.normal(0, 0.5, L.M)).astype(np.float32)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad)
    y = swd.forward(torch.from_numpy(x).cuda(), w, bias=torch.from_numpy(bias).cuda(), relu=relu)
    torch.cuda.synchronize()
    ref, mag = _ref(x, rowptr, colidx, value, L, bias, relu)
    _check(y.cpu().numpy().astype(np.float64), ref, mag, integer)
    if relu:
        assert (y >= 0).all()
    w.close()


@pytest.mark.gpu
def test_relu_without_bias():
    L = workloads.LAYERS["tiny"]
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad)
    y = swd.forward(torch.from_numpy(x).cuda(), w, relu=True)
    torch.cuda.synchronize()
    ref, mag = _ref(x, rowptr, colidx, value, L, np.zeros(L.M), True)
    _check(y.cpu().numpy().astype(np.float64), ref, mag, False)
    w.close()


@pytest.mark.gpu
@pytest.mark.parametrize("integer", [True, False])
def test_chain_of_three_layers(integer):
    """A ResNet-like chain: 3x3 conv + bias + ReLU three times, activations
    staying on the GPU.  Integer: the whole chain is exact.  fp32: every stage
    is checked against the oracle applied to the GPU's previous output."""
    shapes = [(1, 32, 14, 14, 64, 0.10), (1, 64, 14, 14, 64, 0.05), (1, 64, 14, 14, 32, 0.10)]
    rng = np.random.default_rng(11)
    x = workloads.random_input((1, 32, 14, 14), rng, integer=integer)
    xd = torch.from_numpy(x).cuda()
    ref = x.astype(np.float64)
    for i, (N, C, H, W, M, d) in enumerate(shapes):
        L = workloads.Layer(f"chain{i}", N, C, H, W, M, 3, 3, 1, 1, d, integer=integer)
        rowptr, colidx, value = workloads.random_csr(M, C * 9, d, rng, integer=integer)
        bias = (rng.integers(-5, 6, M) if integer else rng.normal(0, 0.1, M)).astype(np.float32)
        w = swd.pack(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=3, S=3, stride=1, pad=1)
        yd = swd.forward(xd, w, bias=torch.from_numpy(bias).cuda(), relu=True)
        torch.cuda.synchronize()
        got = yd.cpu().numpy().astype(np.float64)
        prev = ref if integer else xd.cpu().numpy().astype(np.float64)
        ref, mag = _ref(prev, rowptr, colidx, value, L, bias, True)
        _check(got, ref, mag, integer)
        xd = yd
        w.close()


def test_forward_ex_rejects_unknown_activation():
    w = swd.pack_host(np.array([0, 1], np.int32), np.array([4], np.int32),
                      np.array([1.0], np.float32), C=1, H=5, W=5, M=1, R=3, S=3, stride=1, pad=1)
    rc = _lib.lib().spconv_forward_ex(1, 1, 5, 5, 1, 3, 3, 1, 1, None, w.handle, None, 7, None,
                                      None)
    assert rc == _lib.SPCONV_ERR_INVALID_ARG
    rc = _lib.lib().spconv_forward_ex(1, 1, 5, 5, 1, 3, 3, 1, 1, None, w.handle, None, 1, None,
                                      None)
    assert rc == _lib.SPCONV_ERR_MISMATCH  # host-only handle
    w.close()


@pytest.mark.gpu
@pytest.mark.parametrize("hw", [14, 16])  # 14: cp.async staging + cluster; 16: TMA staging
def test_ping_pong_chain_back_to_back(hw):
    """Ten layers launched back to back on one stream, alternating between two
    buffers: each layer reads what the previous one wrote and overwrites what
    the one before it read.  A kernel may start while the previous one
    finishes (programmatic dependent launch) and must still see that order.
    Each row has two nonzeros of +-1 (the centre tap of one permuted channel,
    the corner tap of another), so values at most double per layer and stay
    exact: the result must equal the oracle applied layer by layer."""
    rng = np.random.default_rng(21 + hw)
    N, C, H, W, K = 1, 64, hw, hw, 3
    layers = []
    for _ in range(10):
        perm, perm2 = rng.permutation(C), rng.permutation(C)
        rows = [sorted({(int(perm[m]) * K + 1) * K + 1, (int(perm2[m]) * K) * K}) for m in range(C)]
        rowptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
        colidx = np.concatenate(rows).astype(np.int32)
        value = rng.choice(np.array([-1, 1], np.float32), size=colidx.size)
        layers.append((rowptr, colidx, value))
    x0 = rng.integers(0, 8, size=(N, C, H, W)).astype(np.float32)
    ws = [swd.pack(rp, ci, v, C=C, H=H, W=W, M=C, R=K, S=K, stride=1, pad=1, batch_hint=1)
          for rp, ci, v in layers]
    a = torch.from_numpy(x0).cuda()
    b = torch.empty_like(a)
    torch.cuda.synchronize()
    src, dst = a, b
    for w in ws:
        swd.forward(src, w, out=dst)
        src, dst = dst, src
    torch.cuda.synchronize()
    got = src.cpu().numpy().astype(np.float64)
    ref = x0.astype(np.float64)
    for rp, ci, v in layers:
        ref, _ = oracle.csr(ref, rp, ci, v, C, K, K, 1, 1)
    assert np.array_equal(got, ref)
    for w in ws:
        w.close()
