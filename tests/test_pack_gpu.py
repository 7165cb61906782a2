"""GPU parity of the pack kernel (rotation + row absmax + quantization) against
the oracle, through the C ABI, on the workloads' seeded inputs and edge cases.
"""
import numpy as np
import pytest
import torch

import oracle
from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from parity import assert_codes, assert_scales

pytestmark = pytest.mark.gpu


def gpu_pack(ops, X, G):
    Q, s = ops.convrot_pack_activations(dev(X), G)
    return host(Q), host(s)


def check(ops, X, G, exact=False):
    Q, s = gpu_pack(ops, X, G)
    Qo, so = oracle.pack(X, G)
    assert_scales(s, so)
    n = assert_codes(Q, Qo)
    if exact:
        assert n == 0
    return n


def test_tiny_workload(ops):
    case = workloads.make_case(workloads.get("tiny"))
    check(ops, case.X, 256, exact=True)   # 1e-4 of 4096 codes rounds to zero mismatches


@pytest.mark.parametrize("G", [4, 16, 64, 256, 1024])
def test_pack_sweep_full_size(ops, G):
    """4096 x 3072 fp32 with 0.5% channel outliers x30, every group size."""
    case = workloads.make_case(workloads.get("pack_sweep"))
    check(ops, case.X, G)


def test_unet_fp16_input(ops):
    case = workloads.make_case(workloads.get("unet"))
    assert case.X.dtype == np.float16
    check(ops, case.X, 256)


def test_dit_input(ops):
    case = workloads.make_case(workloads.get("dit_qkv"))
    check(ops, case.X, 256)


@pytest.mark.parametrize("G", [1, 4, 16, 64, 256, 1024])
@pytest.mark.parametrize("M,Kmul", [(1, 1), (3, 2), (37, 3), (130, 5)])
def test_ragged_shapes(ops, G, M, Kmul):
    K = max(G, 16) * Kmul if G >= 16 else 16 * Kmul + (16 if G < 16 else 0)
    rng = workloads.rng_for(G * 1000 + M * 10 + Kmul)
    X = workloads.activations(rng, M, K, outlier_frac=0.02, outlier_mult=40.0)
    check(ops, X, G)


@pytest.mark.parametrize("K,G", [(16, 1), (48, 4), (80, 16), (1280, 256), (12288, 256),
                                 (12288, 1024), (32768, 1024), (32768, 64)])
def test_row_lengths(ops, K, G):
    rng = workloads.rng_for(K + G)
    X = workloads.activations(rng, 9, K, outlier_frac=0.01, outlier_mult=30.0)
    check(ops, X, G)


@pytest.mark.parametrize("G", [4, 16, 64, 256, 1024])
def test_one_hot_rows(ops, G):
    """x = c e_j: the closed form gives +-127 over the group, 0 elsewhere."""
    K = 2048
    X = np.zeros((4, K), np.float32)
    X[0, 0] = 3.0
    X[1, G + 5] = -40.0
    X[2, K - 1] = 1000.0
    X[3, 17] = 1e-20
    Q, s = gpu_pack(ops, X, G)
    Qo, so = oracle.pack(X, G)
    np.testing.assert_array_equal(Q, Qo)
    np.testing.assert_array_equal(s, so)


def test_zero_and_constant_rows(ops):
    K = 1024
    X = np.zeros((5, K), np.float32)
    X[1] = 2.5
    X[2, ::2] = -1.0
    X[4, 3] = 7.0
    for G in (1, 4, 16, 64, 256, 1024):
        Q, s = gpu_pack(ops, X, G)
        Qo, so = oracle.pack(X, G)
        np.testing.assert_array_equal(Q, Qo)
        np.testing.assert_array_equal(s, so)
        assert s[0] == 0 and s[3] == 0 and not Q[0].any() and not Q[3].any()


def test_prepare_weight(ops):
    case = workloads.make_case(workloads.get("unet"))
    W = case.Ws[0]
    Qw, s_w, Qw16 = ops.convrot_prepare_weight(dev(W), 256)
    Qw, s_w, Qw16 = host(Qw), host(s_w), host(Qw16)
    Qo, so = oracle.prepare_weight(W, 256)
    assert_scales(s_w, so)
    assert_codes(Qw, Qo)
    np.testing.assert_array_equal(Qw16.astype(np.int32), Qw.astype(np.int32))


def test_empty_batch(ops):
    X = torch.zeros((0, 256), dtype=torch.float32, device="cuda")
    Q, s = ops.convrot_pack_activations(X, 256)
    assert Q.shape == (0, 256) and s.shape == (0,)


def test_argument_errors_on_gpu(ops):
    X = torch.zeros((4, 96), dtype=torch.float32, device="cuda")
    with pytest.raises(ops.ConvrotError) as e:
        ops.convrot_pack_activations(X, 64)
    assert e.value.status == ops.ERR_GROUP


def test_rounding_ties_and_neighbours(ops):
    """Quotients exactly at k + 1/2 (round half to even) and one ulp either
    side, plus quotients that land within a few ulp of a half-integer after
    an inexact scale: the quantizer must take the IEEE-division decision."""
    K = 256
    rows = []
    # s = 1 exactly (row max 127): x / s = x
    base = np.zeros(K, np.float32)
    base[0] = 127.0
    ks = np.arange(-60, 60, dtype=np.float32)
    ties = ks + np.float32(0.5)
    r = base.copy(); r[1:1 + len(ties)] = ties; rows.append(r)
    r = base.copy(); r[1:1 + len(ties)] = np.nextafter(ties, np.float32(np.inf)); rows.append(r)
    r = base.copy(); r[1:1 + len(ties)] = np.nextafter(ties, np.float32(-np.inf)); rows.append(r)
    # inexact scales: x = (k + 1/2) * s rounded to fp32, for several row maxima
    for amax in (100.0, 3.3, 0.07, 12345.678):
        s = np.float32(np.float32(amax) / np.float32(127))
        r = np.zeros(K, np.float32)
        r[0] = np.float32(amax)
        vals = (ks + np.float32(0.5)) * s
        r[1:1 + len(vals)] = vals
        r[1 + len(vals):1 + 2 * len(vals)] = np.nextafter(vals, np.float32(np.inf))
        rows.append(r)
    X = np.stack(rows).astype(np.float32)
    Q, s = gpu_pack(ops, X, 1)
    Qo, so = oracle.pack(X, 1)
    np.testing.assert_array_equal(s, so)
    np.testing.assert_array_equal(Q, Qo)
    # the same rows through a rotation (G = 4): still identical decisions
    # whenever the rotated values agree bit for bit
    Q4, s4 = gpu_pack(ops, X, 4)
    Qo4, so4 = oracle.pack(X, 4)
    assert_scales(s4, so4)
    assert_codes(Q4, Qo4)


@pytest.mark.parametrize("M,K,G", [(37, 1024, 1024), (130, 2048, 64), (5, 12288, 256),
                                   (3, 96, 16), (9, 16384, 4), (1000, 1280, 256)])
def test_fp16_input_shapes(ops, M, K, G):
    """fp16 activations: rows of whole 128-byte lines (streamed by tensor
    copies, including a partial last block and rows split over several boxes)
    and a row length that is not (K = 96)."""
    rng = workloads.rng_for(M * 7 + K + G)
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=20.0, dtype="f16")
    check(ops, X, G)


@pytest.mark.parametrize("M,K,G,dtype", [(300, 3072, 256, "f32"), (7, 16384, 1024, "f32"),
                                         (50, 12288, 256, "f32"), (77, 1280, 64, "f16"),
                                         (3, 48, 4, "f32")])
def test_binary16_code_output(ops, M, K, G, dtype):
    """The pack that feeds the tensor-core GEMM writes the same codes as
    binary16 integers."""
    rng = workloads.rng_for(M + K * 3 + G)
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=40.0, dtype=dtype)
    Q16, s = ops.convrot_pack_activations_f16(dev(X), G)
    Q16, s = host(Q16), host(s)
    Qo, so = oracle.pack(X, G)
    assert_scales(s, so)
    assert np.array_equal(Q16, np.rint(Q16)) and np.abs(Q16).max() <= 127
    assert_codes(Q16.astype(np.int32), Qo)


@pytest.mark.parametrize("G", [1, 4, 16, 64, 256, 1024])
def test_rows_with_subnormal_scales(ops, G):
    """Rows whose rotated maximum lies below about 127 * 2^-126, so that
    s = max|X_rot| / 127 is a subnormal float with few significant bits:
    quotients can then exceed 127 and must clamp, and 1 / (s 2^n) can
    overflow. The values are small integers times a power of two, so every
    sum of the rotation is exact in fp32 and the GPU must match the oracle
    exactly; the smallest rows round to s = 0 (a zero row)."""
    K = 2048
    rng = workloads.rng_for(7100 + G)
    rows = []
    for e in (-120, -126, -128, -133, -138, -141, -145, -149):
        k = rng.integers(-50, 51, size=K).astype(np.float64)
        k[rng.integers(0, K)] = 50.0
        rows.append(k * 2.0 ** e)
    # +-1 and 0 times 2^-149: max |X_rot| <= 2^(n-149) <= 32 * 2^-149, so s rounds to 0
    rows.append(rng.integers(-1, 2, size=K).astype(np.float64) * 2.0 ** -149)
    X = np.array(rows).astype(np.float32)
    assert np.array_equal(X.astype(np.float64), np.array(rows))   # exactly representable
    for dtype_out in ("i8", "f16"):
        if dtype_out == "i8":
            Q, s = gpu_pack(ops, X, G)
        else:
            Q16, s16 = ops.convrot_pack_activations_f16(dev(X), G)
            Q, s = host(Q16).astype(np.int32), host(s16)
        Qo, so = oracle.pack(X, G)
        np.testing.assert_array_equal(s, so)
        np.testing.assert_array_equal(np.asarray(Q, np.int32), Qo.astype(np.int32))
        assert np.any((so > 0) & (so < np.float32(2.0 ** -126)))        # some scales are subnormal
        assert np.any(so == 0)                                          # and the smallest rows are zero rows


def test_rows_of_tiny_random_values(ops):
    """Random rows of magnitudes 1e-37 down to 1e-44 (subnormal inputs
    included): codes stay in [-127, 127]; where the GPU's scale equals the
    oracle's (the rotation sums round differently in fp32, which can move a
    subnormal scale by one unit), the codes agree within the usual bar."""
    K, G = 3072, 256
    rng = workloads.rng_for(7200)
    mags = np.repeat([1e-37, 1e-38, 1e-39, 1e-40, 1e-41, 1e-42, 1e-43, 1e-44], 4)
    X = (rng.standard_normal((len(mags), K)) * mags[:, None]).astype(np.float32)
    Q, s = gpu_pack(ops, X, G)
    Qo, so = oracle.pack(X, G)
    assert np.isfinite(s).all() and np.abs(Q.astype(np.int32)).max() <= 127
    same = s == so
    assert same.sum() >= 0.75 * len(s)
    assert_codes(Q[same], Qo[same])
    ulp = np.float32(2.0 ** -149)
    assert np.all(np.abs(s.astype(np.float64) - so) <= np.maximum(1e-6 * so, ulp))
