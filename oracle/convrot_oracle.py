"""CPU oracle for the INT8 convrot linear layer — TEST INFRASTRUCTURE ONLY.

This module is the plain, slow, obviously-correct statement of what the
convrot linear computes. Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import it; the library never does, and it
shares no code with the CUDA kernels.

Sources (stable-diffusion.cpp documentation pages):
  * "INT8 Convrot Safetensors", section "How INT8 convrot works": the H4
    matrix, the normalized Kronecker power for G = 4^n applied to every
    contiguous group of G input features, R R^T = I, X_rot = X R,
    W_rot = W R, and X_rot W_rot^T = X W^T.
  * same page, "Checkpoint format": G is a power of four dividing K.
  * same page, "Weight quantization": s_w and Q_w per output row.
  * same page, "Runtime activation quantization": s_x per row over the whole
    rotated row, Q_x, the int32 accumulation A, and Y ~= A*s_x*s_w + b.
  * "ggml operator extensions", section "sd.cpp integration": the output is
    float(int32_dot) * X_scale * W_scale + bias, evaluated in that order, with
    the weight scale and the bias optional.

Readings where the pages leave a step open (each listed in the design notes):
  * "round" is round-half-to-even (IEEE rint).
  * X_rot is the exact product X R rounded once to fp32; here it is formed in
    fp64 (every product x * (+-2^-n) is exact in fp64, the sums carry ~53-bit
    precision) and then rounded to fp32.
  * s = amax / 127 and X_rot / s are each one IEEE fp32 division.
  * An all-zero row has s = 0 and Q = 0.
  * Y is rounded to fp32 after every operation: ((float(A) * s_x) * s_w) + b.
  * The MLP pair's GELU is the exact-erf GELU, formed in fp64, rounded to fp32.
  * Split SwiGLU is h = silu(gate) * up with silu(g) = g / (1 + exp(-g)),
    gate and up each the output of a convrot linear, formed in fp64 from
    their fp32 values and rounded once to fp32.

Every function is pinned in tests/test_oracle_pins.py against facts the pages
or mathematics fix (the printed H4, orthogonality, closed forms, brute force).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "H4",
    "is_valid_group",
    "hadamard_matrix",
    "rotate",
    "quantize_rows",
    "pack",
    "prepare_weight",
    "gemm_s32",
    "reconstruct",
    "linear",
    "linear_scaled",
    "prologue",
    "unpack_w4",
    "gelu",
    "silu_mul",
    "linear_swiglu",
]

# "INT8 Convrot Safetensors" -- How INT8 convrot works: the regular Hadamard
# matrix with its 1/2 normalisation (rows are orthonormal).
H4 = np.array([[1, 1, 1, -1],
               [1, 1, -1, 1],
               [1, -1, 1, 1],
               [-1, 1, 1, 1]], dtype=np.float64) / 2.0

QMAX = 127
INT32_MAX = 2**31 - 1


def is_valid_group(G: int, K: int) -> bool:
    """G = 4^n (n >= 0) and G divides K ("Checkpoint format")."""
    if G < 1 or K < 1:
        return False
    g = G
    while g % 4 == 0:
        g //= 4
    return g == 1 and K % G == 0


def hadamard_matrix(G: int) -> np.ndarray:
    """R_G = H4^{(x) n}, the normalized Kronecker power, as a dense fp64 matrix.

    Entry (i, j) of a Kronecker power of a 4x4 matrix is the product over the
    base-4 digits of i and j: R[i, j] = prod_k H4[digit_k(i), digit_k(j)].
    ("How INT8 convrot works".)  G = 1 gives the 1x1 identity.
    """
    if not is_valid_group(G, G):
        raise ValueError(f"group size {G} is not a power of four")
    n = 0
    while 4**n < G:
        n += 1
    R = np.ones((G, G), dtype=np.float64)
    idx = np.arange(G)
    for k in range(n):
        d = (idx // 4**k) % 4
        R *= H4[d[:, None], d[None, :]]
    return R


def rotate(X: np.ndarray, G: int) -> np.ndarray:
    """X_rot = X R with R block-diagonal over contiguous groups of G features.

    Returns fp32: the fp64 group products rounded once to fp32.
    ("How INT8 convrot works": applied independently to every contiguous group
    of G input features.)
    """
    X = np.asarray(X)
    M, K = X.shape
    if not is_valid_group(G, K):
        raise ValueError(f"group size {G} must be a power of four dividing K={K}")
    R = hadamard_matrix(G)
    x64 = X.astype(np.float64).reshape(M, K // G, G)
    y64 = np.einsum("rgi,ij->rgj", x64, R, optimize=True)
    return y64.reshape(M, K).astype(np.float32)


def quantize_rows(Xrot: np.ndarray):
    """Per-row absmax INT8 quantization of an fp32 matrix.

    s[r] = max_i |X_rot[r, i]| / 127  (one fp32 division)
    Q[r, i] = clamp(round(X_rot[r, i] / s[r]), -127, 127)  (fp32 division,
    round half to even). ("Runtime activation quantization"; the weight rows
    use the same rule, "Weight quantization".)  A zero row gives s = 0, Q = 0.
    """
    Xrot = np.asarray(Xrot, dtype=np.float32)
    amax = np.max(np.abs(Xrot), axis=1) if Xrot.shape[1] else np.zeros(Xrot.shape[0], np.float32)
    s = (amax.astype(np.float32) / np.float32(QMAX)).astype(np.float32)
    Q = np.zeros(Xrot.shape, dtype=np.int8)
    nz = s > 0
    if np.any(nz):
        q = Xrot[nz] / s[nz][:, None]          # fp32 / fp32 -> fp32 (IEEE)
        assert q.dtype == np.float32
        q = np.rint(q)                          # round half to even
        q = np.clip(q, -QMAX, QMAX)
        Q[nz] = q.astype(np.int8)
    return Q, s


def pack(X: np.ndarray, G: int):
    """Rotate then quantize activation rows: returns (Q_x int8 [M,K], s_x f32 [M])."""
    return quantize_rows(rotate(X, G))


def prepare_weight(W: np.ndarray, G: int):
    """Offline weight path: W_rot = W R, then per-output-row quantization.

    Returns (Q_w int8 [N,K], s_w f32 [N]). ("Weight quantization".)
    """
    return quantize_rows(rotate(W, G))


def gemm_s32(Qx: np.ndarray, Qw: np.ndarray) -> np.ndarray:
    """A[r, o] = sum_i Q_x[r, i] * Q_w[o, i] in signed 32-bit integers.

    Formed with an fp64 matrix product, which is exact here: every product is
    an integer of magnitude <= 127^2 and every partial sum is an integer below
    2^31 < 2^53. The result is checked to fit int32.
    ("Runtime activation quantization": the matrix multiplication accumulates
    into signed 32-bit integers.)
    """
    Qx = np.asarray(Qx)
    Qw = np.asarray(Qw)
    if Qx.shape[1] != Qw.shape[1]:
        raise ValueError("inner dimensions differ")
    bound = Qx.shape[1] * QMAX * QMAX
    if bound > INT32_MAX:
        raise OverflowError(f"K={Qx.shape[1]} can overflow int32")
    A = Qx.astype(np.float64) @ Qw.astype(np.float64).T
    A = np.rint(A)
    if A.size and np.max(np.abs(A)) > INT32_MAX:
        raise OverflowError("int32 overflow")
    return A.astype(np.int32)


def reconstruct(A: np.ndarray, s_x: np.ndarray, s_w=None, bias=None) -> np.ndarray:
    """Y = float(A) * s_x[r] * s_w[o] + b[o], one fp32 rounding per operation,
    in that order; a missing weight scale or bias is left out.
    ("ggml operator extensions", sd.cpp integration; "INT8 Convrot
    Safetensors", Runtime activation quantization.)
    """
    Y = np.asarray(A).astype(np.float32)
    Y = (Y * np.asarray(s_x, np.float32)[:, None]).astype(np.float32)
    if s_w is not None:
        Y = (Y * np.asarray(s_w, np.float32)[None, :]).astype(np.float32)
    if bias is not None:
        Y = (Y + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
    return Y


def linear(X: np.ndarray, Qw: np.ndarray, s_w, bias, G: int) -> np.ndarray:
    """One convrot linear: pack X, integer GEMM against Q_w, reconstruct."""
    Qx, s_x = pack(X, G)
    return reconstruct(gemm_s32(Qx, Qw), s_x, s_w, bias)


def linear_scaled(X: np.ndarray, Qw: np.ndarray, s_w, bias, G: int, input_scale: float) -> np.ndarray:
    """One convrot linear with an input scale a ("Runtime activation
    quantization": for input scales other than 1 the activations are scaled
    before the convrot quantization and the output is unscaled before the
    bias): X' = fp32(a * X), Q_x', s_x' = pack(X'), and
    Y = (((float(A) * s_x') * s_w) / a) + b with one fp32 rounding per step.
    """
    a = np.float32(input_scale)
    Xs = (np.asarray(X).astype(np.float32) * a).astype(np.float32)
    Qx, s_x = pack(Xs, G)
    Y = gemm_s32(Qx, Qw).astype(np.float32)
    Y = (Y * np.asarray(s_x, np.float32)[:, None]).astype(np.float32)
    if s_w is not None:
        Y = (Y * np.asarray(s_w, np.float32)[None, :]).astype(np.float32)
    Y = (Y / a).astype(np.float32)
    if bias is not None:
        Y = (Y + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
    return Y


def prologue(X: np.ndarray, rmsnorm: bool = False, eps: float = 1e-6, weight=None, scale=None,
             shift=None) -> np.ndarray:
    """The normalization / modulation producers fused into the pack
    ("ggml operator extensions", sd.cpp integration: Modulate computes
    (x + x * scale) + shift with separate fp32 multiply/add rounding, and
    RMSNorm -> Mul(weight) -> Modulate -> ConvRot is one of the fused chains).
    In order, each operation rounded to fp32:
      rmsnorm: r = 1 / sqrt(mean(x^2) + eps) per row (the sum of squares
               formed in fp64 and rounded to fp32, then the mean, the sum
               with eps, the square root and the reciprocal in fp32), x * r;
      weight:  x * w[k];   scale: x + x * s[k];   shift: x + h[k].
    """
    x = np.asarray(X).astype(np.float32)
    f32 = np.float32
    if rmsnorm:
        ss = (x.astype(np.float64) ** 2).sum(axis=1).astype(f32)
        mean = (ss / f32(x.shape[1])).astype(f32)
        d = (mean + f32(eps)).astype(f32)
        r = (f32(1.0) / np.sqrt(d).astype(f32)).astype(f32)
        x = (x * r[:, None]).astype(f32)
    if weight is not None:
        x = (x * np.asarray(weight, f32)[None, :]).astype(f32)
    if scale is not None:
        t = (x * np.asarray(scale, f32)[None, :]).astype(f32)
        x = (x + t).astype(f32)
    if shift is not None:
        x = (x + np.asarray(shift, f32)[None, :]).astype(f32)
    return x


def unpack_w4(packed: np.ndarray) -> np.ndarray:
    """Weights of the packed INT4 convrot format ("INT8 Convrot Safetensors",
    Packed INT4 convrot: signed 4-bit values, low nibble first): byte j of a
    row holds element 2j in its low and element 2j+1 in its high four bits,
    each a two's-complement value in [-8, 7]. Returns int8 [N, 2 * bytes]."""
    b = np.asarray(packed, dtype=np.uint8).astype(np.int16)
    lo = b & 0xF
    hi = b >> 4
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty((b.shape[0], 2 * b.shape[1]), dtype=np.int8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def gelu(Y: np.ndarray) -> np.ndarray:
    """Exact-erf GELU 0.5*y*(1+erf(y/sqrt 2)), formed in fp64, rounded to fp32.

    The pages do not name the MLP activation; this is the standard definition.
    """
    from scipy.special import erf  # library erf, fp64
    y = np.asarray(Y, dtype=np.float64)
    return (0.5 * y * (1.0 + erf(y / math.sqrt(2.0)))).astype(np.float32)


def silu_mul(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """Split SwiGLU: h = silu(gate) * up, silu(g) = g / (1 + exp(-g)), formed in
    fp64 from the fp32 inputs and rounded once to fp32. ("ggml operator
    extensions", sd.cpp integration: two INT8 GEMMs sharing a quantized input
    fuse with split SwiGLU; the gate and up weights stay separate.)"""
    g = np.asarray(gate, dtype=np.float32).astype(np.float64)
    u = np.asarray(up, dtype=np.float32).astype(np.float64)
    with np.errstate(over="ignore"):
        sg = g / (1.0 + np.exp(-g))
    return (sg * u).astype(np.float32)


def linear_swiglu(X: np.ndarray, Qg: np.ndarray, s_g, b_g, Qu: np.ndarray, s_u, b_u, G: int) -> np.ndarray:
    """The split-SwiGLU pair on one packed input: h = silu(gate) * up, gate and
    up each the convrot linear of X (the same pack) with its own weight."""
    Qx, s_x = pack(X, G)
    gate = reconstruct(gemm_s32(Qx, Qg), s_x, s_g, b_g)
    up = reconstruct(gemm_s32(Qx, Qu), s_x, s_u, b_u)
    return silu_mul(gate, up)
