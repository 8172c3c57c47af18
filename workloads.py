"""Seeded synthetic layers for the sparse-weight direct convolution.

This module only draws random numbers and lays them out as the method's inputs:
a dense NCHW fp32 activation tensor and an M x (C*R*S) CSR weight matrix
(rowptr / colidx / value).  It holds none of the convolution's arithmetic, so
both the CPU oracle's tests and the CUDA path's tests and benchmark can use it.

Layer shapes follow the workloads the sparse-convolution pages measure on
(ResNet-, VGG- and AlexNet-like layers, a 512-channel sparsity sweep); the
pages publish no dataset, so every tensor here is synthetic:

* activations: max(0, N(0, 1)) in fp32 (a post-ReLU feature map);
* kept weight values: N(0, sigma=0.05) in fp32;
* "uniform unstructured sparsity" at density d: each of the M*C*R*S weights is
  kept independently with probability d (Bernoulli);
* "lognormal" rows: per-output-channel density d_m = d * L_m / mean(L) with
  L_m ~ lognormal(0, 1), clipped to [1/CRS, 1] with the clipped excess spread
  over the unclipped rows until the mean is d, then round(d_m * CRS) column
  positions per row drawn uniformly without replacement;
* integer variant: kept weights uniform in {-3..3} minus {0}, inputs uniform
  in {0..7}; every fp32 partial sum of such a layer is an exact integer.

Column index convention (the M x CRS lowered filter matrix of Escoin,
"Sparse convolution" section, Fig. 3): colidx = (c * R + r) * S + s.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class Layer:
    name: str
    N: int
    C: int
    H: int
    W: int
    M: int
    R: int
    S: int
    stride: int
    pad: int
    density: float          # mean fraction of kept weights (1 - sparsity)
    rows: str = "bernoulli"  # "bernoulli" | "lognormal"
    integer: bool = False
    seed: int = 1234

    @property
    def E(self) -> int:
        return (self.H + 2 * self.pad - self.R) // self.stride + 1

    @property
    def F(self) -> int:
        return (self.W + 2 * self.pad - self.S) // self.stride + 1

    @property
    def CRS(self) -> int:
        return self.C * self.R * self.S

    def with_batch(self, N: int) -> "Layer":
        return dataclasses.replace(self, N=N)


def _layers() -> List[Layer]:
    L = []
    # 0: tiny correctness layer (+ its integer variant)
    L.append(Layer("tiny", 1, 16, 16, 16, 32, 3, 3, 1, 1, 0.10))
    L.append(Layer("tiny_int", 1, 16, 16, 16, 32, 3, 3, 1, 1, 0.10, integer=True))
    # 1: ResNet-style 3x3 layer
    L.append(Layer("resnet3x3", 1, 256, 14, 14, 256, 3, 3, 1, 1, 0.10))
    # 2: VGG-style 3x3 layer, batched
    L.append(Layer("vgg3x3", 16, 128, 56, 56, 128, 3, 3, 1, 1, 0.05))
    # 3: sparsity / imbalance sweep, lognormal per-row density
    for sp in (50, 80, 90, 95, 99):
        L.append(Layer(f"sweep{sp}", 8, 512, 28, 28, 512, 3, 3, 1, 1,
                       round(1.0 - sp / 100.0, 4), rows="lognormal"))
    # 4: large-kernel strided layers
    L.append(Layer("alex11x11", 32, 3, 227, 227, 96, 11, 11, 4, 0, 0.20))
    L.append(Layer("conv5x5", 32, 96, 27, 27, 256, 5, 5, 1, 2, 0.20))
    return [dataclasses.replace(l, seed=1234 + i) for i, l in enumerate(L)]


LAYERS: Dict[str, Layer] = {l.name: l for l in _layers()}


def _p1_sweep() -> List[Layer]:
    """The first page's A100 sweep (Tuteja et al., Sec. 6.1, Fig. 5a/6a/7a):
    N=32, IC=32, H=W=256, 3x3, stride 1, same-size output, OC 48..256,
    sparsity 90..98 %.  The page's weight generator draws positions with
    Python's random module and states no value distribution; Bernoulli
    positions and N(0, 0.05) values stand in."""
    out = []
    for oc in (48, 64, 80, 96, 112, 128, 256):
        for sp in (90, 92, 94, 96, 98):
            out.append(Layer(f"p1_oc{oc}_s{sp}", 32, 32, 256, 256, oc, 3, 3, 1, 1,
                             round(1.0 - sp / 100.0, 4), seed=5000 + oc * 100 + sp))
    return out


# Shapes of the pages' own dense-vs-sparse comparison (not part of the
# default parity sweep: each input is 268 MB).
P1_LAYERS: Dict[str, Layer] = {l.name: l for l in _p1_sweep()}
ALL_LAYERS: Dict[str, Layer] = {**LAYERS, **P1_LAYERS}

# The layer the benchmark times by default: the largest one-GPU layer of the
# 90-99 % sparsity range (N=8, C=M=512, 28x28, 3x3, 90 %, lognormal rows).
BENCH_DEFAULT = "sweep90"


def _lognormal_row_counts(M: int, K: int, density: float,
                          rng: np.random.Generator) -> np.ndarray:
    L = rng.lognormal(mean=0.0, sigma=1.0, size=M)
    d = density * L / L.mean()
    lo, hi = 1.0 / K, 1.0
    for _ in range(100):
        d = np.clip(d, lo, hi)
        err = density * M - d.sum()
        if abs(err) <= 1e-3 * density * M:
            break
        free = (d > lo) & (d < hi) if err < 0 else (d < hi)
        if not free.any():
            break
        d[free] += err * d[free] / d[free].sum()
    counts = np.rint(d * K).astype(np.int64)
    return np.clip(counts, 1, K)


def make_weights(layer: Layer) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Return (rowptr int32[M+1], colidx int32[nnz], value float32[nnz]).

    Columns are sorted ascending within each row."""
    rng = np.random.default_rng(layer.seed)
    M, K = layer.M, layer.CRS
    if layer.rows == "bernoulli":
        mask = rng.random((M, K)) < layer.density
        counts = mask.sum(axis=1)
        cols = [np.nonzero(mask[m])[0] for m in range(M)]
    elif layer.rows == "lognormal":
        counts = _lognormal_row_counts(M, K, layer.density, rng)
        cols = [np.sort(rng.choice(K, size=int(k), replace=False)) for k in counts]
    else:
        raise ValueError(layer.rows)
    rowptr = np.zeros(M + 1, dtype=np.int64)
    rowptr[1:] = np.cumsum(counts)
    nnz = int(rowptr[-1])
    colidx = (np.concatenate(cols) if nnz else np.zeros(0)).astype(np.int32)
    if layer.integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], dtype=np.float32), size=nnz)
    else:
        value = rng.normal(0.0, 0.05, size=nnz).astype(np.float32)
    return rowptr.astype(np.int32), colidx, value.astype(np.float32)


def make_input(layer: Layer, N: int | None = None) -> np.ndarray:
    """Return the NCHW float32 activation tensor (post-ReLU)."""
    n = layer.N if N is None else N
    rng = np.random.default_rng(layer.seed + 1_000_003)
    shape = (n, layer.C, layer.H, layer.W)
    if layer.integer:
        return rng.integers(0, 8, size=shape).astype(np.float32)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return np.maximum(x, np.float32(0.0))


def random_csr(M: int, K: int, density: float, rng: np.random.Generator,
               integer: bool = False) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Bernoulli CSR of an M x K matrix for ad-hoc (small) test shapes."""
    mask = rng.random((M, K)) < density
    rowptr = np.zeros(M + 1, dtype=np.int32)
    rowptr[1:] = np.cumsum(mask.sum(axis=1))
    colidx = np.nonzero(mask)[1].astype(np.int32)
    nnz = colidx.size
    if integer:
        value = rng.choice(np.array([-3, -2, -1, 1, 2, 3], dtype=np.float32), size=nnz)
    else:
        value = rng.normal(0.0, 0.05, size=nnz).astype(np.float32)
    return rowptr, colidx, value.astype(np.float32)


def random_input(shape, rng: np.random.Generator, integer: bool = False) -> np.ndarray:
    if integer:
        return rng.integers(0, 8, size=shape).astype(np.float32)
    return np.maximum(rng.standard_normal(size=shape, dtype=np.float32), np.float32(0))
