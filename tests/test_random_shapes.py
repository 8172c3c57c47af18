"""Seeded random layers across every plan the packer makes: kernel sizes 1..11
(square or not), strides 1 / 2 / 4, any padding, widths and heights up to 64,
1..320 channels, densities from 0.5 % to dense, a batch hint that is unknown,
too small, exact or too large, and all three weight formats.  Half the
shapes are drawn uniformly; the other half aim at a particular plan (tight
pitch, plane staging, column blocks, image pairs in 3x3 and 5x5, tap pairs,
dense-tap groups, split rows, channel-split clusters), with the rest of
their parameters random.

CPU: every packed layout (F32 and 32-bit words) decodes back to the CSR
input, and the launch of each batch size is planned.  GPU: the forward
matches the oracle element by element (integer layers bit-exact)."""
import numpy as np
import pytest

import oracle
import workloads
import sparse_weight_direct_gb300 as swd

from test_abi import decode_layout


def _rows(M, CRS, d, rng, heavy_every, heavy_d, integer):
    rows = [np.nonzero(rng.random(CRS) < (heavy_d if heavy_every and m % heavy_every == 0
                                          else d))[0] for m in range(M)]
    rowptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    colidx = np.concatenate(rows).astype(np.int32) if rows else np.zeros(0, np.int32)
    if integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], np.float32), size=colidx.size)
    else:
        value = rng.normal(0, 0.05, size=colidx.size).astype(np.float32)
    return rowptr, colidx, value.astype(np.float32)


def random_layer(seed):
    """(N, hint, C, H, W, M, R, S, stride, pad, fmt, integer, rowptr, colidx, value)."""
    rng = np.random.default_rng(seed)
    aim = seed % 2 == 1 and rng.integers(0, 9)
    heavy_every, heavy_d = 0, 0.0
    fmt = str(rng.choice(["f32", "f32", "f32", "packed32", "ws"]))
    N = int(rng.integers(1, 7))
    if not aim:
        K = int(rng.choice([1, 2, 3, 3, 5, 7, 11]))
        R, S = (K, K) if rng.random() < 0.8 else (int(rng.choice([1, 3, 5])),
                                                  int(rng.choice([1, 3, 5])))
        stride = int(rng.choice([1, 1, 2, 4]))
        pad = int(rng.integers(0, max(R, S) // 2 + 2))
        H = int(rng.integers(max(1, R - 2 * pad), 49))
        W = int(rng.integers(max(1, S - 2 * pad), 49))
        C, M = int(rng.integers(1, 160)), int(rng.integers(1, 160))
        d = float(rng.choice([0.005, 0.05, 0.2, 0.6, 1.0]))
    else:
        R = S = 3
        stride, pad = 1, 1
        C, M = int(rng.integers(8, 200)), int(rng.integers(8, 160))
        d = float(rng.choice([0.02, 0.1, 0.25]))
        if aim == 1:    # tight pitch: one tile column, 16-byte rows
            H, W = int(rng.integers(8, 40)), int(rng.choice([20, 28]))
        elif aim == 2:  # plane staging: one image, 14 x 14
            N, H, W, fmt = 1, 14, 14, "f32"
        elif aim == 3:  # column blocks: 56 / 84 wide
            H, W = int(rng.integers(8, 40)), int(rng.choice([56, 84]))
        elif aim == 4:  # image pairs (3x3): 22..28 wide, dense-tap rows holding most nonzeros
            N, H, W, fmt = int(rng.integers(2, 7)), int(rng.integers(10, 30)), 28, "f32"
            heavy_every, heavy_d, d = 2, 0.7, 0.03
        elif aim == 5:  # image pairs (5x5)
            R = S = 5
            pad = 2
            N, H, W = int(rng.integers(2, 7)), int(rng.integers(10, 30)), int(rng.choice([24, 27]))
        elif aim == 6:  # tap pairs: dense enough for shared taps
            R = S = int(rng.choice([3, 5]))
            pad, d, fmt = R // 2, 0.5, "f32"
            H, W = int(rng.integers(10, 40)), int(rng.integers(33, 64))
        elif aim == 7:  # heavy rows: split parts, or dense-tap groups
            H, W = int(rng.integers(10, 40)), int(rng.integers(10, 64))
            heavy_every, heavy_d, d = int(rng.choice([3, 16])), 0.9, 0.02
        else:           # one image, many channels: channel-split clusters
            N, H, W = 1, int(rng.integers(6, 20)), int(rng.integers(6, 40))
            C = int(rng.integers(200, 600))
    hint = int(rng.choice([0, 1, N, 2 * N]))
    integer = bool(rng.random() < 0.4)
    rowptr, colidx, value = _rows(M, C * R * S, d, rng, heavy_every, heavy_d, integer)
    if fmt == "packed32":  # the 32-bit word holds FP16 values
        value = value.astype(np.float16).astype(np.float32)
    return N, hint, C, H, W, M, R, S, stride, pad, fmt, integer, rowptr, colidx, value


CPU_SEEDS = list(range(120))
GPU_SEEDS = list(range(1000, 1060))


@pytest.mark.parametrize("seed", CPU_SEEDS)
def test_random_layout_decodes_to_csr(seed):
    N, hint, C, H, W, M, R, S, st, pad, fmt, integer, rowptr, colidx, value = random_layer(seed)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=R, S=S, stride=st, pad=pad,
                      fmt=fmt, batch_hint=hint)
    for n in (1, N, 2 * N + 1):
        launch = w.launch_info(n)
        assert launch["smem_bytes"] <= 227 * 1024 and launch["grid_x"] >= 1
    if fmt != "ws":
        _, rows, _ = decode_layout(w)
        for m in range(M):
            lo, hi = rowptr[m], rowptr[m + 1]
            want = sorted((c, v) for c, v in zip(colidx[lo:hi].tolist(),
                                                  value[lo:hi].astype(np.float64).tolist())
                          if v != 0)
            assert [(c, v) for c, v in rows.get(m, []) if v != 0] == want, m
    w.close()


def test_random_layers_reach_every_plan():
    """The aimed half of the seeds does reach the plans it aims at."""
    seen = set()
    for seed in CPU_SEEDS + GPU_SEEDS:
        N, hint, C, H, W, M, R, S, st, pad, fmt, _, rowptr, colidx, value = random_layer(seed)
        if fmt == "ws":
            continue
        w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=R, S=S, stride=st,
                          pad=pad, fmt=fmt, batch_hint=hint)
        i, launch = w.info(), w.launch_info(N)
        flags = set(w.array("group_flags").tolist())
        seen |= {k for k, on in (("tight", i["shift"] == -1), ("plane", i["plane_stage"] == 1),
                                 ("cols", i["col_blocks"] == 1 and i["tile_images"] == 1),
                                 ("pairs3", i["tile_images"] == 2 and R == 3),
                                 ("pairs5", i["tile_images"] == 2 and R == 5),
                                 ("tap_pairs", i["tap_pairs"] == 1),
                                 ("dense", 1 in flags), ("split_rows", 2 in flags),
                                 ("cluster", launch["cluster"] > 1)) if on}
        w.close()
    assert seen == {"tight", "plane", "cols", "pairs3", "pairs5", "tap_pairs", "dense",
                    "split_rows", "cluster"}, seen


@pytest.mark.gpu
@pytest.mark.parametrize("seed", GPU_SEEDS)
def test_random_layer_parity(seed):
    from test_parity import run_gpu, check
    N, hint, C, H, W, M, R, S, st, pad, fmt, integer, rowptr, colidx, value = random_layer(seed)
    rng = np.random.default_rng(seed + 7)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, R, S, st, pad, fmt=fmt, batch_hint=hint)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, R, S, st, pad)
    check(got, ref, mag, exact=integer,
          what=f"seed {seed}: N={N} hint={hint} C={C} {H}x{W} M={M} {R}x{S}/{st} pad {pad} {fmt}")
