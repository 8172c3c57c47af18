"""The tensor-memory window path (SPCONV_FORMAT_TMEM): host-side plan and
layout checks (CPU), and GPU parity against the CPU oracle under the same
rule as the shared-memory path (|gpu - oracle| <= 1e-5 * sum|w*x| + 1e-7,
bit-exact on integer-valued layers)."""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads
import sparse_weight_direct_gb300 as swd
from sparse_weight_direct_gb300 import _lib

from test_parity import check, run_gpu

torch = pytest.importorskip("torch")

FULL = ["vgg3x3", "sweep50", "sweep80", "sweep90", "sweep95", "sweep99"]


def _pack_host(L, rowptr, colidx, value):
    return swd.pack_host(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                         stride=L.stride, pad=L.pad, fmt="tmem")


# ------------------------------------------------------------------ host (CPU)

@pytest.mark.parametrize("name", ["tiny", "resnet3x3", "alex11x11", "conv5x5"])
def test_unsupported_shapes_rejected(name):
    """Only 3x3 stride-1 layers wider than 16 output columns take the path:
    tiny and resnet3x3 (16 and 14 columns: two lane rows), 11x11/4 and 5x5
    are refused with SPCONV_ERR_UNSUPPORTED."""
    L = workloads.LAYERS[name]
    rowptr, colidx, value = workloads.make_weights(L)
    with pytest.raises(swd.SpconvError) as ei:
        _pack_host(L, rowptr, colidx, value)
    assert ei.value.status == _lib.SPCONV_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", FULL)
def test_plan_has_no_dense_groups_and_no_cluster(name):
    L = workloads.LAYERS[name]
    rowptr, colidx, value = workloads.make_weights(L)
    w = _pack_host(L, rowptr, colidx, value)
    info = w.info()
    assert info["format"] == 3 and info["dense_groups"] == 0
    assert info["slots_per_warp"] in (4, 8)
    assert info["smem_bytes"] >= 80 * 1024  # at most two blocks (2 x 256 columns) per SM
    for n in (1, L.N):
        li = w.launch_info(n)
        assert li["kernel"] == 2 and li["cluster"] == 1 and li["push"] == 0
    w.close()


# ------------------------------------------------------------------ GPU parity

def tm_case(L, N=None):
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L, N)
    got = run_gpu(x, rowptr, colidx, value, L.C, L.H, L.W, L.M, L.R, L.S, L.stride, L.pad,
                  fmt="tmem", batch_hint=L.N)
    ref, mag = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
    check(got, ref, mag, exact=L.integer, what=L.name + ":tmem")


@pytest.mark.gpu
@pytest.mark.parametrize("name", FULL)
def test_full_size(name):
    """The eligible seeded layers at full size, as bench.py --fmt tmem runs them."""
    tm_case(workloads.LAYERS[name])


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["vgg3x3", "sweep50", "sweep90", "sweep99"])
def test_integer_variant_bit_exact(name):
    L = dataclasses.replace(workloads.LAYERS[name], integer=True, name=name + "_int")
    tm_case(L, N=min(L.N, 4))


EDGE = [
    # (N, C, H, W, M, pad, density)
    (2, 40, 30, 30, 70, 1, 0.2),     # ragged groups and chunks, 30 of 32 columns
    (1, 80, 20, 37, 33, 1, 0.1),     # two column tiles, the second 5 wide
    (3, 7, 17, 17, 9, 1, 0.5),       # 17 columns, one channel chunk
    (2, 600, 18, 18, 40, 1, 0.05),   # many chunks
    (1, 24, 40, 40, 64, 0, 0.3),     # no padding (E = H - 2)
    (1, 24, 19, 21, 64, 2, 0.3),     # pad 2 (E = H + 2)
    (2, 16, 24, 24, 16, 1, 1.0),     # fully dense rows (9 taps per channel)
    (1, 33, 26, 26, 130, 1, 0.02),   # very sparse, several empty (warp, channel) words
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", EDGE, ids=[str(c) for c in EDGE])
@pytest.mark.parametrize("integer", [False, True])
def test_edge_shapes(case, integer):
    N, C, H, W, M, pad, d = case
    rng = np.random.default_rng(abs(hash(case)) % (2 ** 32) + integer)
    rowptr, colidx, value = workloads.random_csr(M, C * 9, d, rng, integer=integer)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, 3, 3, 1, pad, fmt="tmem")
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, 3, 3, 1, pad)
    check(got, ref, mag, exact=integer, what=str(case))


@pytest.mark.gpu
@pytest.mark.parametrize("integer", [False, True])
def test_split_rows_and_empty_rows(integer):
    """A few very heavy rows (split into parts over several warps, summed in
    the epilogue) and empty rows (written as zeros) on the path."""
    rng = np.random.default_rng(11 + integer)
    N, C, H, W, M = 2, 48, 20, 20, 96
    CRS = C * 9
    rows = []
    for m in range(M):
        d = 0.9 if m % 40 == 0 else (0.0 if m % 13 == 5 else 0.05)
        rows.append(np.nonzero(rng.random(CRS) < d)[0])
    rowptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    colidx = np.concatenate(rows).astype(np.int32)
    if integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], np.float32), size=colidx.size)
    else:
        value = rng.normal(0, 0.05, size=colidx.size).astype(np.float32)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=3, S=3, stride=1, pad=1,
                      fmt="tmem")
    assert (w.array("group_flags") & 2).any()
    w.close()
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, 3, 3, 1, 1, fmt="tmem")
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, 3, 3, 1, 1)
    check(got, ref, mag, exact=integer, what="split rows")
    assert not got[:, 5::13].any()


@pytest.mark.gpu
def test_repeated_forwards_and_streams():
    """One handle, several forwards on two streams: identical results (the
    block's tensor memory is allocated and freed by every launch)."""
    L = workloads.LAYERS["sweep90"]
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L, 2)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=3, S=3, stride=1, pad=1,
                 fmt="tmem", batch_hint=2)
    xd = torch.from_numpy(x).cuda()
    outs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for i in range(6):
        out = torch.empty((2, L.M, L.E, L.F), device="cuda")
        swd.forward(xd, w, out=out, stream=streams[i % 2])
        outs.append(out)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert w.device_status() == 0
    w.close()
    ref, mag = oracle.csr(x, rowptr, colidx, value, L.M, 3, 3, 1, 1)
    check(outs[0].cpu().numpy().astype(np.float64), ref, mag, what="sweep90 x2")
