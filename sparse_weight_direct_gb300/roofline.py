"""Traffic and FLOP accounting for the sparse direct convolution (host-side).

Tuteja et al., "Theoretical and Empirical Analysis of Sparse Convolution",
Sec. 4 ("Roofline Modelling"):

* Eq.(4)  AI = FLOPs / bytes.
* Eq.(5)  FLOPs_dense  = 2 N Hout Wout OC K^2 IC.
* Eq.(6)  Mem_dense    = (N H W IC + K^2 IC OC + Hout Wout N OC) * P.
* Eq.(7)  Mem_sparse   = (N H W IC + N Hout Wout OC) * P
                         + (1 - S) K^2 IC OC (P + P_idx).
* Eq.(8)  FLOPs_sparse = 2 N Hout Wout OC (1 - S) K^2 IC.
* Ridge point = peak FLOP/s / bandwidth (A100: 19.5 TFLOP/s / 2 TB/s).

Table 1 of that page is reproduced only with 4-byte activations and 4-byte
packed weight entries (P = 4, P + P_idx = 4); the text's "P = 2" describes the
FP16 weight half of the packed word.  This library stores 8 bytes per nonzero
(fp32 value + int32 precomputed offset), so its algorithmic bytes use 8.
Non-square kernels use R*S in place of K^2.
"""
from __future__ import annotations


def out_extent(size: int, k: int, stride: int, pad: int) -> int:
    return (size + 2 * pad - k) // stride + 1


def flops_dense(N, E, F, M, C, R, S) -> float:
    return 2.0 * N * E * F * M * R * S * C


def mem_dense(N, H, W, C, M, R, S, E, F, P=4) -> float:
    return float(N * H * W * C + R * S * C * M + E * F * N * M) * P


def flops_sparse(N, E, F, M, C, R, S, sparsity) -> float:
    return 2.0 * N * E * F * M * (1.0 - sparsity) * R * S * C


def mem_sparse(N, H, W, C, M, R, S, E, F, sparsity, P=4, P_entry=4) -> float:
    return float(N * H * W * C + N * E * F * M) * P + (1.0 - sparsity) * R * S * C * M * P_entry


def ai_sparse(N, H, W, C, M, K, sparsity, pad=None, stride=1, P=4, P_entry=4) -> float:
    pad = (K - 1) // 2 if pad is None else pad
    E, F = out_extent(H, K, stride, pad), out_extent(W, K, stride, pad)
    return (flops_sparse(N, E, F, M, C, K, K, sparsity)
            / mem_sparse(N, H, W, C, M, K, K, E, F, sparsity, P, P_entry))


def ai_dense(N, H, W, C, M, K, pad=None, stride=1, P=4) -> float:
    pad = (K - 1) // 2 if pad is None else pad
    E, F = out_extent(H, K, stride, pad), out_extent(W, K, stride, pad)
    return flops_dense(N, E, F, M, C, K, K) / mem_dense(N, H, W, C, M, K, K, E, F, P)


def ridge(peak_flops: float, bandwidth: float) -> float:
    return peak_flops / bandwidth


# ---- per-launch figures of one layer, with the realised nonzero count ----

ENTRY_BYTES = 8  # fp32 value + int32 precomputed input offset


def useful_flops(nnz: int, N: int, E: int, F: int) -> float:
    """Eq.(8) with the realised nonzero count: 2 * nnz * N * E * F."""
    return 2.0 * nnz * N * E * F


def dense_equiv_flops(N, E, F, M, C, R, S) -> float:
    return flops_dense(N, E, F, M, C, R, S)


def algorithmic_bytes(N, C, H, W, M, E, F, nnz, entry_bytes=ENTRY_BYTES) -> float:
    """Input read once + output written once + each nonzero read once + the
    (M + 1)-entry per-output-channel offset array (Eq.(7) form)."""
    return 4.0 * (N * C * H * W + N * M * E * F) + entry_bytes * nnz + 4.0 * (M + 1)


def roofline_time(flops: float, nbytes: float, peak_flops: float, bandwidth: float) -> float:
    """max(T_comp, T_comm): the time bound min(peak, AI * BW) implies."""
    return max(flops / peak_flops, nbytes / bandwidth)
