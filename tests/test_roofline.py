"""The per-launch accounting bench.py reports (useful FLOPs, algorithmic
bytes, the roofline time), pinned to figures worked out by hand for the
one-image ResNet-style layer (N=1, C=M=256, 14x14, 3x3, pad 1, 58 972
nonzeros): useful FLOPs = 2 * nnz * N * E * F (the first page's Eq.(8) with
the realised nonzero count); bytes = input once + output once + 8 bytes per
nonzero + the (M + 1) offsets (its Eq.(7) form)."""
import pytest

import workloads
from sparse_weight_direct_gb300 import roofline


def test_one_image_layer_by_hand():
    N, C, H, W, M, nnz = 1, 256, 14, 14, 256, 58972
    E = F = roofline.out_extent(14, 3, 1, 1)
    assert E == 14
    # 2 * 58972 * 196
    assert roofline.useful_flops(nnz, N, E, F) == 23_117_024
    # 4 * (256*196 + 256*196) + 8 * 58972 + 4 * 257 = 401408 + 471776 + 1028
    assert roofline.algorithmic_bytes(N, C, H, W, M, E, F, nnz) == 874_212
    # dense 3x3: 2 * 196 * 256 * 256 * 9
    assert roofline.dense_equiv_flops(N, E, F, M, C, 3, 3) == 231_211_008


def test_roofline_time_is_the_larger_bound():
    # 1 GFLOP at 1 TFLOP/s = 1 ms; 1 GB at 1 TB/s = 1 ms; the larger wins
    assert roofline.roofline_time(1e9, 5e8, 1e12, 1e12) == pytest.approx(1e-3)
    assert roofline.roofline_time(5e8, 2e9, 1e12, 1e12) == pytest.approx(2e-3)


def test_workload_nnz_matches_the_layer_density():
    L = workloads.LAYERS["resnet3x3"]
    rowptr, colidx, value = workloads.make_weights(L)
    assert rowptr[-1] == colidx.size == 58972  # the count the figures above use
    assert abs(colidx.size / (L.M * L.C * 9) - L.density) < 0.01
