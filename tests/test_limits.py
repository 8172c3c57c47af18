"""GPU parity at the extremes of the tiling plan: very wide and very tall
images (many column / row tiles), thousands of output channels (over a
thousand channel groups along grid y), a large batch (thousands of tiles along
grid x) and a single input channel.  Full comparison against the CPU oracle
under the usual rule (bit-exact on integer-valued data)."""
import numpy as np
import pytest

import oracle
import workloads
import sparse_weight_direct_gb300 as swd

from test_parity import check, run_gpu

torch = pytest.importorskip("torch")

CASES = [
    # (name, N, C, H, W, M, R, S, stride, pad, density)
    ("wide", 1, 4, 5, 2000, 6, 3, 3, 1, 1, 0.5),        # 63 column tiles, TMA rows of 8000 B
    ("wide_odd", 1, 3, 4, 1999, 5, 3, 3, 1, 1, 0.5),    # odd width: cp.async staging
    ("tall", 1, 4, 3000, 8, 6, 3, 3, 1, 1, 0.5),        # hundreds of row tiles
    ("many_m", 1, 2, 6, 6, 12000, 3, 3, 1, 1, 0.3),     # ~1500 channel groups on grid y
    ("big_batch", 3000, 2, 6, 6, 4, 3, 3, 1, 1, 0.5),   # 3000 images along grid x
    ("one_channel", 4, 1, 40, 40, 64, 5, 5, 1, 2, 0.6), # C = 1 (one chunk of one channel)
    ("strided_wide", 2, 3, 9, 1500, 4, 11, 11, 4, 2, 0.2),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("integer", [False, True])
def test_plan_extremes(case, integer):
    name, N, C, H, W, M, R, S, st, pad, d = case
    rng = np.random.default_rng(sum(map(ord, name)) + integer)
    rowptr, colidx, value = workloads.random_csr(M, C * R * S, d, rng, integer=integer)
    x = workloads.random_input((N, C, H, W), rng, integer=integer)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=R, S=S, stride=st, pad=pad)
    li = w.launch_info(N)
    assert li["grid_x"] * li["grid_y"] >= 1 and li["grid_y"] <= 65535
    w.close()
    got = run_gpu(x, rowptr, colidx, value, C, H, W, M, R, S, st, pad, batch_hint=N)
    ref, mag = oracle.csr(x, rowptr, colidx, value, M, R, S, st, pad)
    check(got, ref, mag, exact=integer, what=name)
