"""The weight-stationary format (one output channel per thread block, its
entries staged in shared memory, the input read in place; Escoin, arXiv
1802.10280, Figs. 5-7): its packed layout on the CPU, and its forward against
the oracle on the GPU with the same rule as the tiled path --
|gpu - oracle| <= 1e-5 * sum|w*x| + 1e-7 per output, bit-exact for integer
layers.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads
import sparse_weight_direct_gb300 as swd
from sparse_weight_direct_gb300 import _lib

from test_parity import EDGE, check

WS_LAYERS = ["tiny", "resnet3x3", "vgg3x3", "sweep50", "sweep90", "sweep99", "alex11x11",
             "conv5x5"]


def pack_ws_host(L, rowptr, colidx, value):
    return swd.pack_host(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                         stride=L.stride, pad=L.pad, fmt="ws")


# ---------------------------------------------------------------- CPU: layout


@pytest.mark.parametrize("name", ["tiny", "resnet3x3", "sweep99", "alex11x11", "conv5x5"])
def test_ws_layout_decodes_to_csr(name):
    """Every row's entries decode back to its CSR nonzeros: value, and the
    stretched offset c*H*W + r*W + s with the tap (r, s) of column
    (c*R + r)*S + s (Escoin's weight stretching against the input tensor)."""
    L = workloads.LAYERS[name]
    rowptr, colidx, value = workloads.make_weights(L)
    w = pack_ws_host(L, rowptr, colidx, value)
    raw = w.array("blobs")
    vals = raw.view(np.float32)[0::2]
    words = raw.view(np.uint32)[1::2]
    info = w.array("blob_off").reshape(L.M, 2)
    order = w.array("slot_oc")
    counts = np.diff(rowptr)
    assert sorted(order.tolist()) == list(range(L.M))
    assert np.all(np.diff(counts[order]) <= 0), "rows must run heaviest first"
    RS = L.R * L.S
    for m in range(L.M):
        first, cnt = int(info[m, 0]), int(info[m, 1])
        assert first % 2 == 0 and cnt == counts[m]
        cols = colidx[rowptr[m]:rowptr[m + 1]]
        srt = np.argsort(cols, kind="stable")
        c, rem = cols[srt] // RS, cols[srt] % RS
        r, s = rem // L.S, rem % L.S
        wd = words[first:first + cnt]
        np.testing.assert_array_equal(wd >> 8, c * L.H * L.W + r * L.W + s)
        np.testing.assert_array_equal((wd >> 4) & 15, r)
        np.testing.assert_array_equal(wd & 15, s)
        np.testing.assert_array_equal(vals[first:first + cnt], value[rowptr[m]:rowptr[m + 1]][srt])
    assert w.array("slot_next").size == 0 and w.array("group_flags").size == 0
    w.close()


@pytest.mark.parametrize("name", WS_LAYERS)
def test_ws_plan_covers_layer(name):
    L = workloads.LAYERS[name]
    rowptr, colidx, value = workloads.make_weights(L)
    w = pack_ws_host(L, rowptr, colidx, value)
    i = w.info()
    assert i["format"] == 2 and i["warps"] == 8
    assert i["tiles_y"] * 8 * i["lane_rows"] * i["tile_rows"] >= L.E
    assert i["tiles_x"] * i["tile_cols"] == i["tiles_x"] * 32 // i["lane_rows"] >= L.F
    assert i["tile_rows"] in (1, 2, 4, 7, 8)
    longest = int(np.diff(rowptr).max())
    assert i["chunk"] % 2 == 0 and i["chunk"] * i["num_chunks"] >= longest
    assert i["max_warp_nnz"] == longest
    w.close()


def test_ws_limits():
    lib = _lib.lib()
    rng = np.random.default_rng(3)

    def pack_rc(C, H, W, M, R, S, stride=1, pad=0, rowptr=None, colidx=None, value=None):
        if rowptr is None:
            rowptr, colidx, value = workloads.random_csr(M, C * R * S, 0.1, rng)
        h = ctypes.c_void_p()
        P = ctypes.c_void_p
        rc = lib.spconv_pack_ex(C, H, W, M, R, S, stride, pad,
                                P(rowptr.ctypes.data), P(colidx.ctypes.data),
                                P(value.ctypes.data), 2, 0, 1, None, ctypes.byref(h))
        if rc == 0:
            lib.spconv_packed_free(h)
        return rc

    assert pack_rc(4, 20, 20, 3, 17, 3) == _lib.SPCONV_ERR_UNSUPPORTED   # R > 16
    assert pack_rc(4, 20, 20, 3, 3, 17) == _lib.SPCONV_ERR_UNSUPPORTED   # S > 16
    # stretched offsets need C*H*W + R*W + S <= 2^24
    assert pack_rc(257, 256, 256, 2, 1, 1) == _lib.SPCONV_ERR_UNSUPPORTED
    assert pack_rc(255, 256, 256, 2, 1, 1) == _lib.SPCONV_OK
    # a repeated column is malformed CSR
    rp = np.array([0, 2], np.int32)
    assert pack_rc(2, 5, 5, 1, 3, 3, rowptr=rp, colidx=np.array([4, 4], np.int32),
                   value=np.ones(2, np.float32)) == _lib.SPCONV_ERR_BAD_CSR


def test_ws_long_rows_take_several_stages():
    """Rows longer than one stage (4096 entries) are streamed in pieces."""
    rng = np.random.default_rng(5)
    C, M = 600, 6
    rowptr, colidx, value = workloads.random_csr(M, C * 9, 0.9, rng)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=6, W=6, M=M, R=3, S=3, stride=1, pad=1,
                      fmt="ws")
    i = w.info()
    assert i["chunk"] == 4096 and i["num_chunks"] == 2
    w.close()


# ---------------------------------------------------------------- GPU: parity

torch = pytest.importorskip("torch")


def run_ws(x, rowptr, colidx, value, C, H, W, M, R, S, stride, pad, bias=None, relu=False):
    w = swd.pack(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=R, S=S, stride=stride, pad=pad,
                 fmt="ws")
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    E, F = swd.out_extent(H, R, stride, pad), swd.out_extent(W, S, stride, pad)
    out = torch.full((x.shape[0], M, E, F), float("nan"), device="cuda")
    bd = torch.from_numpy(bias).cuda() if bias is not None else None
    swd.forward(xd, w, out=out, bias=bd, relu=relu)
    torch.cuda.synchronize()
    assert w.device_status() == 0
    w.close()
    return out.cpu().numpy().astype(np.float64)


def ws_layer_case(L, N=None):
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L, N)
    got = run_ws(x, rowptr, colidx, value, L.C, L.H, L.W, L.M, L.R, L.S, L.stride, L.pad)
    ref, mag = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
    check(got, ref, mag, exact=L.integer, what=L.name + " ws")


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(workloads.LAYERS))
def test_ws_layer_full_size(name):
    ws_layer_case(workloads.LAYERS[name])


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["resnet3x3", "vgg3x3", "sweep90", "alex11x11", "conv5x5"])
def test_ws_integer_bit_exact(name):
    import dataclasses
    L = dataclasses.replace(workloads.LAYERS[name], integer=True, name=name + "_int")
    ws_layer_case(L, N=min(L.N, 4))


@pytest.mark.gpu
@pytest.mark.parametrize("case", EDGE, ids=[str(c) for c in EDGE])
@pytest.mark.parametrize("integer", [False, True])
def test_ws_edge_shapes(case, integer):
    N, C, H, W, M, R, S, st, pad, d = case
    rng = np.random.default_rng(abs(hash(case)) % (2 ** 32))
    rowptr, colidx, value = workloads.random_csr(M, C * R * S, d, rng, integer=integer)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    got = run_ws(x, rowptr, colidx, value, C, H, W, M, R, S, st, pad)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, R, S, st, pad)
    check(got, ref, mag, exact=integer, what=str(case) + " ws")


@pytest.mark.gpu
@pytest.mark.parametrize("integer", [False, True])
def test_ws_long_rows_parity(integer):
    rng = np.random.default_rng(5)
    N, C, H, W, M = 2, 600, 6, 6, 6
    rowptr, colidx, value = workloads.random_csr(M, C * 9, 0.9, rng, integer=integer)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    got = run_ws(x, rowptr, colidx, value, C, H, W, M, 3, 3, 1, 1)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, 3, 3, 1, 1)
    check(got, ref, mag, exact=integer, what="long rows ws")


@pytest.mark.gpu
def test_ws_empty_rows_and_epilogue():
    rng = np.random.default_rng(11)
    N, C, H, W, M = 2, 5, 10, 12, 9
    rowptr, colidx, value = workloads.random_csr(M, C * 9, 0.3, rng)
    keep = np.ones(colidx.size, bool)
    for m in (1, 4):
        keep[rowptr[m]:rowptr[m + 1]] = False
    counts = np.array([keep[rowptr[m]:rowptr[m + 1]].sum() for m in range(M)])
    rp = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ci, va = colidx[keep], value[keep]
    x = workloads.random_input((N, C, H, W), rng)
    ref, mag = oracle.csr(x, rp, ci, va, M, 3, 3, 1, 1)
    got = run_ws(x, rp, ci, va, C, H, W, M, 3, 3, 1, 1)
    check(got, ref, mag, what="empty rows ws")
    assert not got[:, [1, 4]].any()
    bias = rng.normal(0, 0.1, size=M).astype(np.float32)
    got = run_ws(x, rp, ci, va, C, H, W, M, 3, 3, 1, 1, bias=bias, relu=True)
    refb = np.maximum(ref + bias.astype(np.float64)[None, :, None, None], 0.0)
    check(got, refb, mag + np.abs(bias.astype(np.float64))[None, :, None, None],
          what="bias+relu ws")
    z = run_ws(x, np.zeros(M + 1, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float32),
               C, H, W, M, 3, 3, 1, 1)
    assert np.all(z == 0)


@pytest.mark.gpu
def test_ws_batch_limits():
    """Images run along grid z: N = 65535 works, N = 65536 is UNSUPPORTED,
    N = 0 is a no-op."""
    rowptr = np.array([0, 1], np.int32)
    colidx = np.array([0], np.int32)
    value = np.array([2.0], np.float32)
    w = swd.pack(rowptr, colidx, value, C=1, H=1, W=1, M=1, R=1, S=1, fmt="ws")
    x = torch.arange(65536, dtype=torch.float32, device="cuda").reshape(65536, 1, 1, 1)
    y = swd.forward(x[:65535].contiguous(), w)
    torch.cuda.synchronize()
    assert torch.equal(y.reshape(-1), 2.0 * x[:65535].reshape(-1))
    with pytest.raises(swd.SpconvError) as e:
        swd.forward(x, w)
    assert e.value.status == _lib.SPCONV_ERR_UNSUPPORTED
    assert swd.forward(x[:0], w).shape == (0, 1, 1, 1)
    w.close()


@pytest.mark.gpu
def test_ws_p1_sweep_sampled():
    """A first-page sweep shape at full size (N=32, 32 -> 128, 256x256):
    sampled outputs against the oracle evaluated one output at a time, and
    every output written."""
    L = workloads.P1_LAYERS["p1_oc128_s94"]
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad, fmt="ws")
    xd = torch.from_numpy(x).cuda()
    out = torch.full((L.N, L.M, L.E, L.F), float("nan"), device="cuda")
    swd.forward(xd, w, out=out)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    rng = np.random.default_rng(8)
    idx = rng.integers(0, out.numel(), size=20000)
    got = out.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().numpy().astype(np.float64)
    ref, mag = oracle.csr_points(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad, idx)
    check(got, ref, mag, what=L.name + " ws")
    w.close()
