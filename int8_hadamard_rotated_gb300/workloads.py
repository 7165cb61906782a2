"""Seeded synthetic inputs for the convrot linear workloads.

This module only draws random numbers and fixes shapes. It holds none of the
method's arithmetic (no rotation, no quantization, no GEMM), so that both the
CPU oracle and the CUDA path can be fed from it without sharing any code.

Every array is drawn from ``numpy.random.Generator(PCG64(seed))`` in a fixed
order (activation values, then the outlier pattern, then each weight matrix,
then each bias vector), row-major, so the same seed always gives the same
bytes on every machine.

The shapes follow diffusion-model linears: a tiny correctness case, a pack-only
sweep over the group size, a UNet-like 64x64-latent linear, the three DiT
attention projections sharing one input, and the DiT MLP pair.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "get",
    "rng_for",
    "activations",
    "weights",
    "biases",
    "make_case",
    "random_codes",
]


@dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one synthetic workload."""

    name: str
    M: int
    K: int
    G: int
    Ns: Tuple[int, ...]            # output features of each linear sharing X
    seed: int
    x_dtype: str = "f32"           # "f32" or "f16"
    outlier_kind: str = "element"  # "element" (Bernoulli mask) or "channel"
    outlier_frac: float = 0.01
    outlier_mult: float = 50.0
    x_std: float = 1.0
    w_std: float = 0.02
    b_std: float = 0.01
    groups: Tuple[int, ...] = field(default=())  # pack sweep: G values
    chain: bool = False            # MLP pair: second linear consumes GELU(Y_1)

    @property
    def gemm_ops(self) -> int:
        """2*M*N*K summed over the linears (multiply and add each count)."""
        if self.chain:
            n_up = self.Ns[0]
            return 2 * self.M * n_up * self.K + 2 * self.M * self.K * n_up
        return sum(2 * self.M * n * self.K for n in self.Ns)


WORKLOADS = {
    "tiny": Workload("tiny", M=16, K=256, G=256, Ns=(128,), seed=0,
                     outlier_frac=0.01, outlier_mult=50.0),
    "pack_sweep": Workload("pack_sweep", M=4096, K=3072, G=256, Ns=(), seed=1,
                           outlier_kind="channel", outlier_frac=0.005,
                           outlier_mult=30.0, groups=(4, 16, 64, 256, 1024)),
    "unet": Workload("unet", M=4096, K=1280, G=256, Ns=(1280,), seed=2,
                     x_dtype="f16", outlier_frac=0.01, outlier_mult=20.0),
    "dit_qkv": Workload("dit_qkv", M=4608, K=3072, G=256,
                        Ns=(3072, 3072, 3072), seed=3,
                        outlier_frac=0.01, outlier_mult=40.0),
    "dit_mlp": Workload("dit_mlp", M=4608, K=3072, G=256, Ns=(12288, 3072),
                        seed=4, outlier_frac=0.01, outlier_mult=40.0,
                        chain=True),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def activations(rng: np.random.Generator, M: int, K: int, *, std: float = 1.0,
                outlier_kind: str = "element", outlier_frac: float = 0.01,
                outlier_mult: float = 50.0, dtype: str = "f32") -> np.ndarray:
    """X ~ N(0, std) with outliers.

    ``element``: each entry is independently multiplied by ``outlier_mult``
    with probability ``outlier_frac``. ``channel``: round(outlier_frac*K)
    distinct columns, drawn uniformly, are multiplied by ``outlier_mult``.
    """
    x = rng.standard_normal((M, K), dtype=np.float32) * np.float32(std)
    if outlier_frac > 0:
        if outlier_kind == "element":
            mask = rng.random((M, K), dtype=np.float32) < np.float32(outlier_frac)
            x[mask] *= np.float32(outlier_mult)
        elif outlier_kind == "channel":
            n = int(round(outlier_frac * K))
            cols = rng.choice(K, size=n, replace=False)
            x[:, cols] *= np.float32(outlier_mult)
        else:
            raise ValueError(outlier_kind)
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype != "f32":
        raise ValueError(dtype)
    return x


def weights(rng: np.random.Generator, N: int, K: int, std: float = 0.02) -> np.ndarray:
    return rng.standard_normal((N, K), dtype=np.float32) * np.float32(std)


def biases(rng: np.random.Generator, N: int, std: float = 0.01) -> np.ndarray:
    return rng.standard_normal((N,), dtype=np.float32) * np.float32(std)


@dataclass
class Case:
    X: np.ndarray
    Ws: List[np.ndarray]
    bs: List[np.ndarray]


def make_case(w: Workload, *, M: Optional[int] = None) -> Case:
    """Draw X, the weights and the biases of workload ``w``.

    ``M`` optionally draws fewer activation rows (a prefix of the full draw is
    NOT implied; a smaller M is its own seeded draw of the same recipe).
    For the chained MLP pair the second weight has shape [K, N_up].
    """
    rng = rng_for(w.seed)
    m = w.M if M is None else M
    X = activations(rng, m, w.K, std=w.x_std, outlier_kind=w.outlier_kind,
                    outlier_frac=w.outlier_frac, outlier_mult=w.outlier_mult,
                    dtype=w.x_dtype)
    Ws, bs = [], []
    if w.chain:
        shapes = [(w.Ns[0], w.K), (w.Ns[1], w.Ns[0])]
    else:
        shapes = [(n, w.K) for n in w.Ns]
    for (n, k) in shapes:
        Ws.append(weights(rng, n, k, w.w_std))
    for (n, _k) in shapes:
        bs.append(biases(rng, n, w.b_std))
    return Case(X=X, Ws=Ws, bs=bs)


def modulation(rng: np.random.Generator, K: int):
    """Per-channel vectors of the pack's modulation prologue: a norm weight
    ~ 1 + N(0, 0.1), a modulation scale ~ N(0, 0.2) and shift ~ N(0, 0.05)."""
    w = (1.0 + 0.1 * rng.standard_normal(K)).astype(np.float32)
    sc = (0.2 * rng.standard_normal(K)).astype(np.float32)
    sh = (0.05 * rng.standard_normal(K)).astype(np.float32)
    return w, sc, sh


def packed_int4(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    """Uniform random bytes [N, K/2]: two signed 4-bit weights each."""
    return rng.integers(0, 256, size=(N, K // 2), dtype=np.int64).astype(np.uint8)


def random_codes(rng: np.random.Generator, rows: int, cols: int,
                 low: int = -127, high: int = 127) -> np.ndarray:
    """Uniform int8 codes in [low, high] (for GEMM-only cases)."""
    return rng.integers(low, high + 1, size=(rows, cols), dtype=np.int64).astype(np.int8)
