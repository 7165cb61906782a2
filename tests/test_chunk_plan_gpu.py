"""The GEMM's exact-chunk plan (convrot_weight_chunks) and the GEMM run with it:
the plan follows the stated rule, never breaks the fp32 exactness bound, and
the int32 product stays bit-exact with it on codes chosen to need short,
medium and whole-K runs."""
import numpy as np
import pytest

import oracle
from int8_hadamard_rotated_gb300 import workloads
from chunk_plan_ref import plan, plan_is_safe
from gpu_common import dev, host
from parity import assert_y

pytestmark = pytest.mark.gpu


def codes(seed, rows, cols, amp):
    rng = workloads.rng_for(seed)
    return workloads.random_codes(rng, rows, cols, -amp, amp)


CASES = [
    # name, M, N, K, weight code amplitude
    ("uniform", 300, 384, 4096, 127),      # mean |q| 63.5: runs of 2048
    ("extreme", 256, 256, 3072, 127),      # replaced by +-127 below: runs of 1024
    ("small", 200, 260, 12288, 3),         # whole-K run
    ("medium", 257, 128, 12288, 40),       # runs of 4096 or 8192
]


@pytest.mark.parametrize("name,M,N,K,amp", CASES)
def test_plan_rule_and_exact_gemm(ops, name, M, N, K, amp):
    Qw = codes(K + N, N, K, amp)
    if name == "extreme":
        Qw = np.where(Qw >= 0, 127, -127).astype(np.int8)
    Qx = codes(M + K, M, K, 127)
    if name == "extreme":
        Qx = np.where(Qx >= 0, 127, -127).astype(np.int8)
    kc = host(ops.convrot_weight_chunks(dev(Qw)))
    np.testing.assert_array_equal(kc, plan(Qw))
    assert plan_is_safe(Qw, kc)
    A = host(ops.int8_gemm_s32(dev(Qx), Q_w16=dev(Qw.astype(np.float16)), kchunk=dev(kc)))
    np.testing.assert_array_equal(A, oracle.gemm_s32(Qx, Qw))


def test_plan_values_on_the_dit_weights(ops):
    """Rotated, per-row quantized N(0, 0.02) weights at K = 3072 run the whole K
    as one exact chunk; at K = 12288 in runs of 4096 or longer."""
    w = workloads.get("dit_mlp")
    case = workloads.make_case(w, M=4)
    for W, whole in ((case.Ws[0], True), (case.Ws[1], False)):
        Qw, _, _ = ops.convrot_prepare_weight(dev(W), 256)
        kc = host(ops.convrot_weight_chunks(Qw))
        Qw = host(Qw)
        np.testing.assert_array_equal(kc, plan(Qw))
        num_kb = W.shape[1] // 64
        if whole:
            assert (kc == num_kb).all()
        else:
            assert (kc >= 64).all()


def test_linear_with_plans_matches_without(ops):
    """The plan changes only how the exact int32 sum is split: Y is identical."""
    w = workloads.get("dit_qkv")
    case = workloads.make_case(w, M=512)
    preps = [ops.convrot_prepare_weight(dev(W), w.G) for W in case.Ws]
    q16s, scales, biases = [p[2] for p in preps], [p[1] for p in preps], [dev(b) for b in case.bs]
    plans = [ops.convrot_weight_chunks(p[0]) for p in preps]
    X = dev(case.X)
    Y0 = [host(y) for y in ops.convrot_linear(X, w.G, q16s, scales, biases)]
    Y1 = [host(y) for y in ops.convrot_linear(X, w.G, q16s, scales, biases, kchunks=plans)]
    for a, b in zip(Y0, Y1):
        np.testing.assert_array_equal(a, b)
    Qw, s_w = host(preps[0][0]), host(preps[0][1])
    assert_y(Y1[0], oracle.linear(case.X, Qw, s_w, case.bs[0], w.G))
