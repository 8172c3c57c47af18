"""GPU parity: spconv_forward (CUDA, through the C ABI) against the CPU oracle,
element by element, on the seeded layers and on edge cases.

Rule (fp32 layers): |gpu - oracle| <= 1e-5 * sum|w*x| + 1e-7 per output, the
oracle in fp64.  Integer-valued layers: bit-exact (every fp32 partial sum is
an exact integer below 2^24, so any summation order gives the same result).
"""
import numpy as np
import pytest

import oracle
import workloads
import sparse_weight_direct_gb300 as swd

torch = pytest.importorskip("torch")

RTOL = 1e-5
ATOL = 1e-7


def run_gpu(x, rowptr, colidx, value, C, H, W, M, R, S, stride, pad, stream=None,
            prefill=float("nan"), fmt="f32", batch_hint=0):
    w = swd.pack(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=R, S=S, stride=stride, pad=pad,
                 fmt=fmt, batch_hint=batch_hint)
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    E = swd.out_extent(H, R, stride, pad)
    F = swd.out_extent(W, S, stride, pad)
    out = torch.full((x.shape[0], M, E, F), prefill, device="cuda", dtype=torch.float32)
    swd.forward(xd, w, out=out, stream=stream)
    torch.cuda.synchronize()
    # no kernel reported a failure (a timed-out wait, or a failed check of the
    # bounds-checked build)
    assert w.device_status(stream) == 0
    w.close()
    return out.cpu().numpy().astype(np.float64)


def check(got, ref, mag, exact=False, what=""):
    assert got.shape == ref.shape, what
    if exact:
        bad = got != ref
    else:
        bad = ~(np.abs(got - ref) <= RTOL * mag + ATOL)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outputs off; first at "
                             f"{tuple(i)}: gpu={got[tuple(i)]!r} oracle={ref[tuple(i)]!r} "
                             f"abs_sum={mag[tuple(i)]!r}")


def layer_case(L, N=None, batch_hint=None):
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L, N)
    hint = L.N if batch_hint is None else batch_hint
    got = run_gpu(x, rowptr, colidx, value, L.C, L.H, L.W, L.M, L.R, L.S, L.stride, L.pad,
                  batch_hint=hint)
    ref, mag = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
    check(got, ref, mag, exact=L.integer, what=L.name)
    return got, ref, mag


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(workloads.LAYERS))
def test_layer_full_size(name):
    """Every seeded layer at its full size, planned for its batch as bench.py
    plans it (the benchmark's launch configuration)."""
    layer_case(workloads.LAYERS[name])


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["resnet3x3", "vgg3x3", "sweep99", "conv5x5"])
@pytest.mark.parametrize("hint", [0, 1, 32])
def test_plan_independent_of_batch_hint(name, hint):
    """Any plan (batch hint unknown, too small or too large for the launch)
    computes the same convolution."""
    layer_case(workloads.LAYERS[name], N=min(workloads.LAYERS[name].N, 4), batch_hint=hint)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["resnet3x3", "vgg3x3", "sweep90", "sweep95", "sweep50",
                                  "alex11x11", "conv5x5"])
def test_integer_variant_bit_exact(name):
    """The same shapes with integer weights in {-3..3}\\{0} and inputs in
    {0..7}: the GPU result must equal the oracle exactly."""
    import dataclasses
    L = dataclasses.replace(workloads.LAYERS[name], integer=True, name=name + "_int")
    layer_case(L, N=min(workloads.LAYERS[name].N, 4))


EDGE = [
    # (N, C, H, W, M, R, S, stride, pad, density)
    (2, 3, 5, 37, 7, 3, 3, 1, 1, 0.3),       # F > 32: two column tiles, ragged
    (1, 1, 1, 1, 1, 1, 1, 1, 0, 1.0),        # 1x1 everything
    (3, 4, 9, 9, 5, 1, 1, 1, 0, 0.5),        # 1x1 conv
    (2, 5, 11, 13, 6, 2, 2, 1, 0, 0.4),      # even kernel
    (2, 4, 17, 19, 9, 7, 7, 2, 3, 0.2),      # generic 7x7 stride 2
    (2, 6, 15, 15, 8, 3, 3, 2, 1, 0.3),      # 3x3 stride 2
    (1, 3, 12, 40, 4, 1, 3, 1, 0, 0.5),      # 1x3
    (1, 3, 40, 12, 4, 3, 1, 1, 1, 0.5),      # 3x1 with pad
    (2, 600, 6, 6, 40, 3, 3, 1, 1, 0.05),    # many input channels: several chunks
    (1, 8, 10, 10, 300, 3, 3, 1, 1, 0.2),    # M not a multiple of the group size
    (1, 2, 30, 30, 3, 5, 5, 3, 2, 0.5),      # 5x5 stride 3
    (2, 3, 23, 23, 4, 11, 11, 4, 1, 0.3),    # 11x11/4 with padding
    (1, 16, 16, 16, 32, 3, 3, 1, 2, 0.1),    # pad larger than needed (E > H)
    (5, 4, 8, 8, 6, 3, 3, 1, 1, 1.0),        # fully dense rows
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", EDGE, ids=[str(c) for c in EDGE])
@pytest.mark.parametrize("integer", [False, True])
def test_edge_shapes(case, integer):
    N, C, H, W, M, R, S, st, pad, d = case
    rng = np.random.default_rng(abs(hash(case)) % (2 ** 32))
    rowptr, colidx, value = workloads.random_csr(M, C * R * S, d, rng, integer=integer)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, R, S, st, pad)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, R, S, st, pad)
    check(got, ref, mag, exact=integer, what=str(case))


HEAVY = [  # (N, C, H, W, M), heavy-row density, every, group flag the plan must hold
    ((8, 128, 28, 28, 256), 0.95, 3, 1),   # a third of the rows near-dense: dense-tap groups
    ((4, 128, 56, 56, 128), 0.8, 2, 1),    # half the rows at 0.8: dense-tap groups
    ((8, 128, 28, 28, 256), 0.95, 7, 2),   # too few for dense groups to pay: split rows
    ((2, 24, 12, 12, 96), 0.6, 7, 2),
    ((2, 24, 12, 12, 96), 0.6, 40, 2),
    ((2, 24, 12, 12, 96), 0.95, 40, 2),
]


@pytest.mark.gpu
@pytest.mark.parametrize("integer", [False, True])
@pytest.mark.parametrize("shape,heavy_density,every,want_flag", HEAVY,
                         ids=[f"{c[0]}-{c[1]}-{c[2]}" for c in HEAVY])
def test_heavy_rows_split_and_dense(shape, heavy_density, every, want_flag, integer):
    """Very heavy rows among sparse ones (0.05).  Where they carry most of a
    large layer's work, the planner's estimate puts them in dense-tap groups
    (flag 1); where they are few, or the layer is small, the all-sparse plan
    is estimated faster and each heavy row is split into parts in several
    warps, summed in the epilogue (flag 2)."""
    rng = np.random.default_rng(int(heavy_density * 100) + integer + every)
    N, C, H, W, M = shape
    K = 3
    CRS = C * K * K
    rows = []
    for m in range(M):
        d = heavy_density if m % every == 0 else 0.05
        keep = np.nonzero(rng.random(CRS) < d)[0]
        rows.append(keep)
    rowptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    colidx = np.concatenate(rows).astype(np.int32)
    if integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], np.float32), size=colidx.size)
    else:
        value = rng.normal(0, 0.05, size=colidx.size).astype(np.float32)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=K, S=K, stride=1, pad=1,
                      batch_hint=N)
    assert (w.array("group_flags") & want_flag).any()
    w.close()
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, K, K, 1, 1, batch_hint=N)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, K, K, 1, 1)
    check(got, ref, mag, exact=integer, what=f"heavy {shape} {heavy_density} {every}")


@pytest.mark.gpu
def test_empty_rows_and_empty_matrix():
    rng = np.random.default_rng(1)
    N, C, H, W, M = 2, 4, 9, 9, 10
    rowptr, colidx, value = workloads.random_csr(M, C * 9, 0.3, rng)
    # empty out rows 0, 3, 9
    keep = np.ones(colidx.size, bool)
    for m in (0, 3, 9):
        keep[rowptr[m]:rowptr[m + 1]] = False
    counts = np.array([keep[rowptr[m]:rowptr[m + 1]].sum() for m in range(M)])
    rowptr2 = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = workloads.random_input((N, C, H, W), rng)
    got = run_gpu(x, rowptr2, colidx[keep], value[keep], C, H, W, M, 3, 3, 1, 1)
    ref, mag = oracle.csr(x, rowptr2, colidx[keep], value[keep], M, 3, 3, 1, 1)
    check(got, ref, mag)
    assert not got[:, [0, 3, 9]].any()
    # no nonzeros at all: all outputs written as zero
    z = run_gpu(x, np.zeros(M + 1, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float32),
                C, H, W, M, 3, 3, 1, 1)
    assert np.all(z == 0)


@pytest.mark.gpu
def test_batch_zero_is_noop():
    L = workloads.LAYERS["tiny"]
    rowptr, colidx, value = workloads.make_weights(L)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad)
    x = torch.zeros((0, L.C, L.H, L.W), device="cuda")
    y = swd.forward(x, w)
    assert y.shape == (0, L.M, L.E, L.F)
    w.close()


@pytest.mark.gpu
def test_streams_and_shared_handle():
    """One handle, two forwards on two non-default streams at once."""
    L = workloads.LAYERS["vgg3x3"]
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L, N=4)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad)
    xd = torch.from_numpy(x).cuda()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        y1 = swd.forward(xd, w, stream=s1)
    with torch.cuda.stream(s2):
        y2 = swd.forward(xd[2:], w, stream=s2)
    torch.cuda.synchronize()
    ref, mag = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
    check(y1.cpu().numpy().astype(np.float64), ref, mag, what="stream 1")
    check(y2.cpu().numpy().astype(np.float64), ref[2:], mag[2:], what="stream 2")
    w.close()


@pytest.mark.gpu
def test_forward_argument_errors():
    L = workloads.LAYERS["tiny"]
    rowptr, colidx, value = workloads.make_weights(L)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad)
    lib = swd._lib.lib()
    x = torch.zeros((1, L.C, L.H, L.W), device="cuda")
    y = torch.zeros((1, L.M, L.E, L.F), device="cuda")
    args = (1, L.C, L.H, L.W, L.M, L.R, L.S, L.stride, L.pad)
    import ctypes
    P = ctypes.c_void_p
    ok = lib.spconv_forward(*args, P(x.data_ptr()), w.handle, P(y.data_ptr()), None)
    assert ok == 0
    # misaligned input (not 16-byte aligned)
    assert lib.spconv_forward(*args, P(x.data_ptr() + 4), w.handle, P(y.data_ptr()), None) == -1
    # null output
    assert lib.spconv_forward(*args, P(x.data_ptr()), w.handle, None, None) == -1
    # shape differs from the packed handle
    bad = (1, L.C, L.H + 1, L.W, L.M, L.R, L.S, L.stride, L.pad)
    assert lib.spconv_forward(*bad, P(x.data_ptr()), w.handle, P(y.data_ptr()), None) == -6
    # negative batch
    neg = (-1,) + args[1:]
    assert lib.spconv_forward(*neg, P(x.data_ptr()), w.handle, P(y.data_ptr()), None) == -1
    # overlapping input and output
    assert lib.spconv_forward(*args, P(x.data_ptr()), w.handle, P(x.data_ptr()), None) == -1
    torch.cuda.synchronize()
    w.close()


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["p1_oc64_s90", "p1_oc128_s98", "p1_oc256_s94"])
def test_p1_sweep_sampled(name):
    """The first page's A100 sweep shapes at full size (N=32, 32 -> OC,
    256x256): 20 000 sampled outputs against the oracle evaluated one output
    at a time (Eq.(3)), and every output written (the buffer is prefilled
    with NaN)."""
    L = workloads.P1_LAYERS[name]
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad, batch_hint=L.N)
    xd = torch.from_numpy(x).cuda()
    out = torch.full((L.N, L.M, L.E, L.F), float("nan"), device="cuda")
    swd.forward(xd, w, out=out)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    rng = np.random.default_rng(7)
    idx = rng.integers(0, out.numel(), size=20000)
    got = out.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().numpy().astype(np.float64)
    ref, mag = oracle.csr_points(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad, idx)
    check(got, ref, mag, what=name)
    w.close()


@pytest.mark.gpu
@pytest.mark.parametrize("integer", [False, True])
@pytest.mark.parametrize("name", ["tiny", "resnet3x3", "vgg3x3", "sweep90", "sweep95",
                                  "alex11x11", "conv5x5"])
def test_packed32_format(name, integer):
    """The first page's 32-bit packed words (FP16 values): parity against the
    oracle on the FP16-rounded weights (round to nearest even, once)."""
    import dataclasses
    L = dataclasses.replace(workloads.LAYERS[name], integer=integer)
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L, min(L.N, 4))
    v16 = value.astype(np.float16).astype(np.float32)
    got = run_gpu(x, rowptr, colidx, value, L.C, L.H, L.W, L.M, L.R, L.S, L.stride, L.pad,
                  fmt="packed32")
    ref, mag = oracle.csr(x, rowptr, colidx, v16, L.M, L.R, L.S, L.stride, L.pad)
    check(got, ref, mag, exact=integer, what=name + " packed32")


def _cluster_case(rng, heavy: bool, integer: bool):
    """N=1, 128 channels in 8 chunks, 64 output channels: a small grid whose
    chunks are split over a cluster.  heavy: rows 0 and 40 are 90 % dense and
    get split into parts (which keeps the cluster on the reduction by reads)."""
    C, H, W, M, K = 128, 14, 14, 64, 3
    CRS = C * K * K
    rows = [np.nonzero(rng.random(CRS) < (0.9 if heavy and m in (0, 40) else 0.1))[0]
            for m in range(M)]
    rowptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    colidx = np.concatenate(rows).astype(np.int32)
    if integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], np.float32), size=colidx.size)
    else:
        value = rng.normal(0, 0.05, size=colidx.size).astype(np.float32)
    x = workloads.random_input((1, C, H, W), rng, integer=integer)
    return x, rowptr, colidx, value, C, H, W, M, K


@pytest.mark.gpu
@pytest.mark.parametrize("integer", [False, True])
@pytest.mark.parametrize("heavy", [False, True])
def test_cluster_reduction_paths(heavy, integer):
    """Both cluster reductions against the oracle: partial sums pushed into
    the owning block (no split rows) and read from every rank (split rows)."""
    rng = np.random.default_rng(17 + heavy * 2 + integer)
    x, rowptr, colidx, value, C, H, W, M, K = _cluster_case(rng, heavy, integer)
    w = swd.pack(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=K, S=K, stride=1, pad=1,
                 batch_hint=1)
    plan = w.launch_info(1)
    assert plan["cluster"] > 1 and plan["push"] == (0 if heavy else 1)
    assert bool((w.array("group_flags") & 2).any()) == heavy
    xd = torch.from_numpy(x).cuda()
    out = torch.full((1, M, H, W), float("nan"), device="cuda")
    swd.forward(xd, w, out=out)
    torch.cuda.synchronize()
    assert w.device_status() == 0
    w.close()
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, K, K, 1, 1)
    check(out.cpu().numpy().astype(np.float64), ref, mag, exact=integer,
          what=f"cluster heavy={heavy}")


PAIR_CASES = [
    # (N, C, H, W, M, R, S, stride, pad, density): plans with tap pairs (a fifth or
    # more of the nonzeros share their tap with another output channel of the warp)
    (4, 40, 30, 30, 128, 3, 3, 1, 1, 0.2),     # 3x3, ragged chunks, 30 of 32 columns
    (4, 24, 27, 27, 128, 5, 5, 1, 2, 0.2),     # 5x5
    (8, 3, 99, 99, 128, 11, 11, 4, 0, 0.2),    # 11x11 stride 4
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", PAIR_CASES, ids=[str(c) for c in PAIR_CASES])
@pytest.mark.parametrize("integer", [False, True])
@pytest.mark.parametrize("heavy", [False, True])
def test_tap_pairs(case, integer, heavy):
    """Layers planned with tap-pair entries (one set of shared loads feeding two
    output channels of a warp), with uniform rows and with a few very dense
    rows among them."""
    N, C, H, W, M, R, S, st, pad, d = case
    rng = np.random.default_rng(abs(hash(case)) % (2 ** 32) + 2 * integer + heavy)
    CRS = C * R * S
    rows = [np.nonzero(rng.random(CRS) < (0.95 if heavy and m % 17 == 3 else d))[0]
            for m in range(M)]
    rowptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    colidx = np.concatenate(rows).astype(np.int32)
    if integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], np.float32), size=colidx.size)
    else:
        value = rng.normal(0, 0.05, size=colidx.size).astype(np.float32)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=R, S=S, stride=st, pad=pad,
                      batch_hint=N)
    info = w.info()
    w.close()
    assert info["tap_pairs"] == 1 and info["dense_groups"] == 0
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, R, S, st, pad, batch_hint=N)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, R, S, st, pad)
    check(got, ref, mag, exact=integer, what=f"pairs {case}")


PLANE_CASES = [
    # (N, C, H, W, M, density, heavy): whole-image tiles whose rows TMA cannot address,
    # staged as raw planes with the padding applied to the weights
    (1, 40, 14, 10, 24, 0.3, False),    # W = 10, ragged chunks
    (2, 33, 16, 13, 20, 0.3, False),    # P = 8, odd width, odd channel count
    (1, 64, 14, 6, 70, 0.2, False),     # W = 6, M not a multiple of the group size
    (1, 20, 14, 2, 9, 0.5, False),      # W = 2: every lane but two reads spare banks
    (1, 128, 14, 14, 64, 0.1, True),    # very dense rows split into parts
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", PLANE_CASES, ids=[str(c) for c in PLANE_CASES])
@pytest.mark.parametrize("integer", [False, True])
def test_plane_staging(case, integer):
    N, C, H, W, M, d, heavy = case
    rng = np.random.default_rng(abs(hash(case)) % (2 ** 32) + integer)
    CRS = C * 9
    rows = [np.nonzero(rng.random(CRS) < (0.9 if heavy and m % 20 == 0 else d))[0]
            for m in range(M)]
    rowptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    colidx = np.concatenate(rows).astype(np.int32)
    if integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], np.float32), size=colidx.size)
    else:
        value = rng.normal(0, 0.05, size=colidx.size).astype(np.float32)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=3, S=3, stride=1, pad=1,
                      batch_hint=N)
    info = w.info()
    assert info["plane_stage"] == 1
    assert not heavy or (w.array("group_flags") & 2).any()
    w.close()
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, 3, 3, 1, 1, batch_hint=N)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, 3, 3, 1, 1)
    check(got, ref, mag, exact=integer, what=f"plane {case}")


COLS_CASES = [
    # (N, C, H, W, M, pad, density, heavy): 3x3 stride-1 layers whose output width is a
    # multiple of 28 but not of 32, tiled in column blocks (8 x 28 tiles, each lane seven
    # consecutive outputs of one row)
    (2, 20, 56, 56, 40, 1, 0.1, False),      # two column tiles, one ragged chunk
    (1, 9, 16, 28, 17, 1, 0.3, False),       # one column tile, M not a multiple of 8
    (3, 9, 44, 84, 17, 1, 0.2, False),       # ragged rows (44), three column tiles
    (1, 6, 58, 58, 12, 0, 0.3, False),       # pad 0 (no alignment shift), cp.async staging
    (1, 7, 54, 54, 10, 2, 0.3, False),       # pad 2, cp.async staging
    (2, 32, 112, 112, 16, 1, 0.1, False),    # 112 wide: four column tiles
    (1, 128, 16, 56, 16, 1, 0.2, False),     # two-block clusters, push reduction
    (1, 96, 24, 28, 24, 1, 0.1, False),      # push reduction, one column tile
    (1, 128, 56, 56, 128, 1, 0.05, False),   # two-block clusters, four channels per warp
    (1, 128, 56, 56, 64, 1, 0.1, True),      # very dense rows split into parts, clusters
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", COLS_CASES, ids=[str(c) for c in COLS_CASES])
@pytest.mark.parametrize("integer", [False, True])
@pytest.mark.parametrize("fmt", ["f32", "packed32"])
def test_column_blocks(case, integer, fmt):
    N, C, H, W, M, pad, d, heavy = case
    rng = np.random.default_rng(abs(hash(case)) % (2 ** 32) + integer)
    CRS = C * 9
    rows = [np.nonzero(rng.random(CRS) < (0.9 if heavy and m % 20 == 0 else d))[0]
            for m in range(M)]
    rowptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    colidx = np.concatenate(rows).astype(np.int32)
    if integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], np.float32), size=colidx.size)
    else:
        value = rng.normal(0, 0.05, size=colidx.size).astype(np.float32)
    if fmt == "packed32":  # the 32-bit word holds FP16 values
        value = value.astype(np.float16).astype(np.float32)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=3, S=3, stride=1, pad=pad,
                      batch_hint=N, fmt=fmt)
    assert w.info()["col_blocks"] == 1
    # heavy rows: split into parts, or (dense enough) on the dense-tap path
    assert not heavy or (w.array("group_flags") & 3).any()
    w.close()
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, 3, 3, 1, pad, batch_hint=N, fmt=fmt)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, 3, 3, 1, pad)
    check(got, ref, mag, exact=integer, what=f"column blocks {case}")


PAIR_IMG_CASES = [
    # (N run, N planned, C, H, W, M, pad, sparse density, dense rows, dense groups planned):
    # 3x3 stride-1 layers 22..28 outputs wide planned for a batch, whose dense rows
    # (density 0.6) hold most nonzeros, tiled in image-pair column blocks (lanes 0..3 of a
    # row on image 2n, 4..7 on image 2n + 1, seven consecutive outputs each).  On the two
    # large layers the planner's estimate keeps dense-tap groups beside the sparse ones; on
    # the small ones an all-sparse plan is estimated faster and the heavy rows are split.
    (16, 16, 100, 28, 28, 256, 1, 0.05, 64, True),  # the sweep layers' 28 x 28: chunks
    (15, 16, 100, 28, 28, 256, 1, 0.05, 64, True),  # odd batch: last pair's second half empty
    (8, 8, 40, 28, 28, 72, 1, 0.05, 24, False),     # M not a multiple of 32
    (3, 8, 24, 28, 28, 40, 1, 0.05, 16, False),     # odd batch, small grid
    (1, 8, 24, 28, 28, 40, 1, 0.05, 16, False),     # one image on a pair plan
    (4, 4, 20, 30, 25, 33, 0, 0.05, 16, False),     # 28 x 23 outputs, pad 0 (no shift)
    (6, 6, 16, 26, 28, 24, 1, 0.05, 16, False),     # 26 x 28: the last row band half used
    (2, 2, 600, 28, 28, 16, 1, 0.05, 8, False),     # many chunks, channel-split clusters
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", PAIR_IMG_CASES, ids=[str(c) for c in PAIR_IMG_CASES])
@pytest.mark.parametrize("integer", [False, True])
def test_image_pair_column_blocks(case, integer):
    N, hint, C, H, W, M, pad, d, ndense, want_dense = case
    rng = np.random.default_rng(abs(hash(case[:9])) % (2 ** 32) + integer)
    CRS = C * 9
    rows = [np.nonzero(rng.random(CRS) < (0.6 if m < ndense else d))[0] for m in range(M)]
    rowptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    colidx = np.concatenate(rows).astype(np.int32)
    if integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], np.float32), size=colidx.size)
    else:
        value = rng.normal(0, 0.05, size=colidx.size).astype(np.float32)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=3, S=3, stride=1, pad=pad,
                      batch_hint=hint)
    info = w.info()
    assert info["col_blocks"] == 1 and info["tile_images"] == 2 and info["lane_rows"] == 4
    assert (info["dense_groups"] > 0) == want_dense
    w.close()
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, 3, 3, 1, pad, batch_hint=hint)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, 3, 3, 1, pad)
    check(got, ref, mag, exact=integer, what=f"image pairs {case}")


PAIR5_CASES = [
    # (N run, N planned, C, H, W, M, pad, density, tap pairs, Q): 5x5 stride-1 layers 22..28
    # outputs wide in image-pair column blocks.  Rows that a tensor map can address (W a
    # multiple of 4) are staged by one tensor copy with a ninth staged row; the others by
    # cp.async with the gap between the two images' sub-tiles padded to 16 mod 32 words.
    (16, 16, 96, 27, 27, 256, 2, 0.2, 1, 4),  # the 5x5 layer's shape: tap pairs, 7 chunks
    (9, 10, 48, 27, 27, 128, 2, 0.2, 1, 4),   # odd batch, tap pairs
    (8, 8, 8, 28, 28, 300, 2, 0.25, 1, 4),    # tensor copies, tap pairs, chunk past C
    (4, 4, 24, 28, 28, 64, 2, 0.2, 0, 2),     # tensor copies, two channels per warp
    (3, 4, 16, 24, 24, 40, 2, 0.05, 0, 2),    # odd batch, tensor copies, 24 x 24
    (2, 2, 40, 26, 26, 33, 1, 0.3, 0, 1),     # pad 1: 24 x 24 outputs, M not a multiple of 8
    (5, 6, 12, 22, 22, 16, 2, 0.3, 0, 1),     # 22 x 22: each lane row's last lanes idle
    (1, 4, 24, 27, 27, 64, 2, 0.2, 0, 2),     # one image on a pair plan
    (16, 16, 64, 27, 27, 512, 2, 0.01, 0, 8), # eight channels per warp
    (2, 2, 300, 28, 28, 24, 2, 0.1, 0, 1),    # many chunks, channel-split clusters
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", PAIR5_CASES, ids=[str(c) for c in PAIR5_CASES])
@pytest.mark.parametrize("integer", [False, True])
def test_image_pair_5x5(case, integer):
    N, hint, C, H, W, M, pad, d, want_pairs, want_q = case
    rng = np.random.default_rng(abs(hash(case[:8])) % (2 ** 32))
    rowptr, colidx, value = workloads.random_csr(M, C * 25, d, rng, integer=integer)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=5, S=5, stride=1, pad=pad,
                      batch_hint=hint)
    info = w.info()
    assert info["tile_images"] == 2 and info["lane_rows"] == 4 and info["col_blocks"] == 1
    assert info["tap_pairs"] == want_pairs and info["slots_per_warp"] == want_q
    assert info["pair_off"] % 32 == 16
    if (W * 4) % 16 == 0:  # one tensor copy: the second sub-tile right after the first
        assert info["pair_off"] == info["chunk"] * info["plane"]
    w.close()
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, 5, 5, 1, pad, batch_hint=hint)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, 5, 5, 1, pad)
    check(got, ref, mag, exact=integer, what=f"5x5 image pairs {case}")


TIGHT_CASES = [
    # (N run, N planned, C, H, W, M, density, heavy every, heavy density, Q, chunks, cluster):
    # 3x3 pad-1 layers up to 31 wide in one column-per-lane tile column, staged from column 0
    # at a 32-word pitch (the copy's zero fill stands in for the halo columns; the first
    # row's left tap reads the zeroed lead)
    (8, 8, 64, 28, 28, 96, 0.1, 0, 0.0, 4, 1, 1),        # one chunk
    (6, 8, 300, 28, 28, 64, 0.03, 0, 0.0, 4, 5, 5),      # partial last chunk, cluster split
    (3, 3, 77, 35, 20, 40, 0.15, 0, 0.0, 4, 1, None),    # 20 wide: eight columns of zeros
    (16, 16, 64, 28, 28, 512, 0.01, 0, 0.0, 8, 1, 1),    # eight channels per warp
    (2, 0, 48, 28, 28, 24, 0.2, 0, 0.0, 1, 1, None),     # batch unknown at pack time
    (4, 4, 64, 28, 28, 64, 0.05, 16, 0.9, 4, 1, None),   # heavy rows split over warps
    (1, 1, 300, 28, 28, 16, 0.1, 0, 0.0, 1, 8, 8),       # one image: 8-block cluster (push)
    (1, 1, 300, 28, 28, 32, 0.05, 8, 0.8, 1, 8, 8),      # cluster + split rows (pull)
    (8, 8, 256, 28, 28, 512, 0.15, 5, 0.7, 4, 13, 1),    # dense-tap groups (window at pitch 32)
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", TIGHT_CASES, ids=[str(c[:9]) for c in TIGHT_CASES])
@pytest.mark.parametrize("integer", [False, True])
@pytest.mark.parametrize("fmt", ["f32", "packed32"])
def test_tight_pitch(case, integer, fmt):
    N, hint, C, H, W, M, d, every, hd, want_q, want_nch, want_cluster = case
    rng = np.random.default_rng(abs(hash(case[:9])) % (2 ** 32) + integer)
    rows = [np.nonzero(rng.random(C * 9) < (hd if every and m % every == 0 else d))[0]
            for m in range(M)]
    rowptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    colidx = np.concatenate(rows).astype(np.int32)
    if integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], np.float32), size=colidx.size)
    else:
        value = rng.normal(0, 0.05, size=colidx.size).astype(np.float32)
    if fmt == "packed32":  # the 32-bit word holds FP16 values
        value = value.astype(np.float16).astype(np.float32)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=3, S=3, stride=1, pad=1,
                      batch_hint=hint, fmt=fmt)
    info = w.info()
    assert info["shift"] == -1 and info["row_pitch"] == 32 and info["col_blocks"] == 0
    if fmt == "f32":
        assert info["slots_per_warp"] == want_q and info["num_chunks"] == want_nch
        if want_cluster is not None:
            assert w.launch_info(N)["cluster"] == want_cluster
    w.close()
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, 3, 3, 1, 1, batch_hint=hint, fmt=fmt)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, 3, 3, 1, 1)
    check(got, ref, mag, exact=integer, what=f"tight pitch {fmt} {case[:9]}")


@pytest.mark.gpu
def test_dense_dominated_split_bit_exact():
    """The 50 % lognormal layer at its batch: most groups are dense-tap, so every
    tile's chunks are split over a two-block cluster and the dense-tap
    partial sums meet in the cluster reduction.  Integer weights and inputs:
    bit-exact against the oracle."""
    import dataclasses
    L = dataclasses.replace(workloads.LAYERS["sweep50"], integer=True, name="sweep50_int")
    rowptr, colidx, value = workloads.make_weights(L)
    w = swd.pack_host(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                      stride=L.stride, pad=L.pad, batch_hint=L.N)
    info, launch = w.info(), w.launch_info(L.N)
    assert launch["cluster"] == 2 and 2 * info["dense_groups"] >= info["groups"]
    w.close()
    layer_case(L)
