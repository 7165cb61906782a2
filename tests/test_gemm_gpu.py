"""GPU parity of the tensor-core INT8 GEMM (through the C ABI) against the oracle.

The int32 product must be bit-exact: the same codes go to both sides.
"""
import numpy as np
import pytest
import torch

import oracle
from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from parity import assert_y

pytestmark = pytest.mark.gpu


def run_s32(ops, Qx, Qw, use_w16=True):
    qx = dev(Qx)
    if use_w16:
        A = ops.int8_gemm_s32(qx, Q_w16=dev(Qw.astype(np.float16)))
    else:
        A = ops.int8_gemm_s32(qx, Q_w=dev(Qw))
    return host(A)


def test_structured_permutation(ops):
    """Q_w a signed permutation: each output column is one input column, so a
    layout mistake (swizzle, K offset, lane mapping) shows up as a misplaced
    value rather than a near miss."""
    M, K, N = 256, 256, 128
    rng = workloads.rng_for(100)
    Qx = workloads.random_codes(rng, M, K)
    perm = rng.permutation(K)[:N]
    sign = rng.choice([-1, 1], size=N)
    Qw = np.zeros((N, K), np.int8)
    Qw[np.arange(N), perm] = sign
    A = run_s32(ops, Qx, Qw)
    np.testing.assert_array_equal(A, Qx[:, perm].astype(np.int32) * sign[None, :])


def test_one_hot_products(ops):
    """A[r,o] = r-th row code at column o: places every (row, column) pair."""
    M, K, N = 300, 64, 200
    Qx = np.zeros((M, K), np.int8)
    Qw = np.zeros((N, K), np.int8)
    Qx[np.arange(M), np.arange(M) % K] = ((np.arange(M) % 127) + 1).astype(np.int8)
    Qw[np.arange(N), np.arange(N) % K] = 1
    A = run_s32(ops, Qx, Qw)
    np.testing.assert_array_equal(A, oracle.gemm_s32(Qx, Qw))


@pytest.mark.parametrize("M,N,K", [
    (16, 128, 256), (1, 1, 16), (7, 9, 48), (128, 128, 64), (256, 256, 1024),
    (300, 129, 80), (257, 385, 1040), (513, 300, 3072), (130, 260, 2064),
])
def test_random_codes_bit_exact(ops, M, N, K):
    rng = workloads.rng_for(M * 7 + N * 13 + K)
    Qx = workloads.random_codes(rng, M, K)
    Qw = workloads.random_codes(rng, N, K)
    np.testing.assert_array_equal(run_s32(ops, Qx, Qw), oracle.gemm_s32(Qx, Qw))


@pytest.mark.parametrize("K", [1024, 1040, 2048, 4096, 12288])
def test_extreme_codes_bit_exact(ops, K):
    """All codes +-127: every fp32 chunk partial sum reaches 1024*127^2,
    just under 2^24, where an inexact accumulator would first lose bits."""
    M, N = 256, 128
    rng = workloads.rng_for(K)
    Qx = np.full((M, K), 127, np.int8)
    Qw = np.where(rng.random((N, K)) < 0.5, 127, -127).astype(np.int8)
    Qw[0] = 127
    Qw[1] = -127
    Qx[1::2] = -127
    np.testing.assert_array_equal(run_s32(ops, Qx, Qw), oracle.gemm_s32(Qx, Qw))


def test_largest_k(ops):
    """K = 133120 (the largest multiple of 16 under the int32 bound)."""
    K = 133120
    M, N = 130, 129
    rng = workloads.rng_for(5)
    Qx = np.full((M, K), 127, np.int8)
    Qw = np.full((N, K), 127, np.int8)
    Qw[1::2] = -127
    Qx[5] = workloads.random_codes(rng, 1, K)
    np.testing.assert_array_equal(run_s32(ops, Qx, Qw), oracle.gemm_s32(Qx, Qw))


def test_int8_weight_widened_in_workspace(ops):
    rng = workloads.rng_for(6)
    Qx = workloads.random_codes(rng, 100, 320)
    Qw = workloads.random_codes(rng, 70, 320)
    np.testing.assert_array_equal(run_s32(ops, Qx, Qw, use_w16=False), oracle.gemm_s32(Qx, Qw))


@pytest.mark.parametrize("with_scale,with_bias", [(True, True), (True, False), (False, True), (False, False)])
def test_int8_linear_reconstruction_exact(ops, with_scale, with_bias):
    """Same codes and scales on both sides: Y is the same ordered fp32
    arithmetic, so it must agree bit for bit."""
    case = workloads.make_case(workloads.get("tiny"))
    G = 256
    Qx, s_x = oracle.pack(case.X, G)
    Qw, s_w = oracle.prepare_weight(case.Ws[0], G)
    b = case.bs[0]
    Y = ops.int8_linear(dev(Qx), dev(s_x), Q_w16=dev(Qw.astype(np.float16)),
                        s_w=dev(s_w) if with_scale else None, bias=dev(b) if with_bias else None)
    ref = oracle.reconstruct(oracle.gemm_s32(Qx, Qw), s_x, s_w if with_scale else None,
                             b if with_bias else None)
    np.testing.assert_array_equal(host(Y), ref)


def test_int8_linear_full_dit_codes(ops):
    """DiT-shaped GEMM (M=4608, K=3072, N=3072) on the oracle's own codes."""
    w = workloads.get("dit_qkv")
    case = workloads.make_case(w)
    Qx, s_x = oracle.pack(case.X, w.G)
    Qw, s_w = oracle.prepare_weight(case.Ws[0], w.G)
    Y = ops.int8_linear(dev(Qx), dev(s_x), Q_w16=dev(Qw.astype(np.float16)), s_w=dev(s_w), bias=dev(case.bs[0]))
    ref = oracle.reconstruct(oracle.gemm_s32(Qx, Qw), s_x, s_w, case.bs[0])
    np.testing.assert_array_equal(host(Y), ref)
    assert ops.convrot_device_status() == ops.OK


def test_empty_shapes(ops):
    Qx = torch.zeros((0, 64), dtype=torch.int8, device="cuda")
    Qw16 = torch.zeros((8, 64), dtype=torch.float16, device="cuda")
    A = ops.int8_gemm_s32(Qx, Q_w16=Qw16)
    assert A.shape == (0, 8)
    Qx = torch.zeros((4, 64), dtype=torch.int8, device="cuda")
    A = ops.int8_gemm_s32(Qx, Q_w16=torch.zeros((0, 64), dtype=torch.float16, device="cuda"))
    assert A.shape == (4, 0)


def test_bench_probes_run(ops):
    """The benchmark's own kernels (libconvrot_bench.so): the probe of the
    legacy s8 tensor instruction reports a positive, finite rate, and the
    size-matched copy writes every output byte."""
    import math
    import bench
    tops = bench.int8_mma_rate(2000)
    assert math.isfinite(tops) and tops > 0.0
    X = torch.arange(12 * 64, dtype=torch.float32, device="cuda").reshape(12, 64) % 100
    out = torch.full((12, 64), 0xEE, dtype=torch.uint8, device="cuda")
    sc = torch.full((12,), 1.0, dtype=torch.float32, device="cuda")
    st = bench.bench_lib().bench_copy_ceiling(X.data_ptr(), 12, 64, 1, out.data_ptr(), sc.data_ptr(), 1,
                                              torch.cuda.current_stream().cuda_stream)
    assert st == 0
    np.testing.assert_array_equal(host(out), host(X).astype(np.int64).astype(np.uint8))
    assert not host(sc).any()
