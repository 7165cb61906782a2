"""The packed INT4 convrot weight format on the GPU: the unpack into the
GEMM's codes against the oracle, and a W4A4 linear (INT8 convrot activations
x signed 4-bit weights with per-output scales) against the oracle."""
import numpy as np
import pytest

import oracle
from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from parity import assert_y

pytestmark = pytest.mark.gpu


def packed_weights(seed, N, K):
    return workloads.packed_int4(workloads.rng_for(seed), N, K)


@pytest.mark.parametrize("N,K", [(1, 16), (3, 48), (300, 3072), (129, 1280)])  # (1, 16), (3, 48): odd pack counts
def test_w4_expand_matches_unpack(ops, N, K):
    P = packed_weights(N + K, N, K)
    q8, q16 = ops.convrot_w4_expand(dev(P), K)
    ref = oracle.unpack_w4(P)
    np.testing.assert_array_equal(host(q8), ref)
    np.testing.assert_array_equal(host(q16).astype(np.int32), ref.astype(np.int32))


def test_w4a4_linear(ops):
    w = workloads.get("dit_qkv")
    case = workloads.make_case(w, M=513)
    N, K, G = 1536, w.K, w.G
    P = packed_weights(9, N, K)
    rng = workloads.rng_for(10)
    s_w = (0.001 + 0.01 * rng.random(N)).astype(np.float32)
    b = workloads.biases(rng, N)
    q8, q16 = ops.convrot_w4_expand(dev(P), K)
    plan = ops.convrot_weight_chunks(q8)
    assert (host(plan) == K // 64).all()   # |q_w| <= 8: every row runs all of K in one exact chunk
    (Y,) = ops.convrot_linear(dev(case.X), G, [q16], [dev(s_w)], [dev(b)], kchunks=[plan])
    Qw = oracle.unpack_w4(P)
    assert_y(host(Y), oracle.linear(case.X, Qw, s_w, b, G))
    Qx, _ = ops.convrot_pack_activations(dev(case.X), G)
    A = ops.int8_gemm_s32(Qx, Q_w16=q16, kchunk=plan)
    np.testing.assert_array_equal(host(A), oracle.gemm_s32(host(Qx), Qw))
