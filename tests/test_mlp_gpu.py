"""convrot_mlp: up linear, GELU applied as the down linear's pack loads the up
output, down linear, all on the device (the DiT MLP shapes), against the
oracle stage by stage."""
import numpy as np
import pytest
import torch

import oracle
from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from parity import assert_y, y_rel_err

pytestmark = pytest.mark.gpu


def prepared(ops, W, G):
    q8, s_w, q16 = ops.convrot_prepare_weight(dev(W), G)
    return q8, s_w, q16, ops.convrot_weight_chunks(q8)


@pytest.mark.parametrize("M", [600, 37])
def test_dit_mlp_on_device(ops, M):
    w = workloads.get("dit_mlp")
    case = workloads.make_case(w, M=M)
    G = w.G
    qu, su, hu, ku = prepared(ops, case.Ws[0], G)
    qd, sd, hd, kd = prepared(ops, case.Ws[1], G)
    bu, bd = dev(case.bs[0]), dev(case.bs[1])
    Y_up = torch.empty((M, w.Ns[0]), dtype=torch.float32, device="cuda")
    Y = ops.convrot_mlp(dev(case.X), G, (hu, su, bu, ku), ops.ACT_GELU, G, (hd, sd, bd, kd), H=Y_up)
    Y_up, Y = host(Y_up), host(Y)
    assert ops.convrot_device_status() == ops.OK
    # stage 1: the up linear, against the oracle with the same weight codes
    Qu, su_h = host(qu), host(su)
    Y_up_ref = oracle.linear(case.X, Qu, su_h, case.bs[0], G)
    assert_y(Y_up, Y_up_ref, "Y_up")
    # stage 2: GELU (applied as the pack loads Y_up) and the down linear, on the GPU's own Y_up
    Qd, sd_h = host(qd), host(sd)
    assert_y(Y, oracle.linear(oracle.gelu(Y_up), Qd, sd_h, case.bs[1], G), "GELU + down on the same Y_up")
    # the whole chain against the oracle chain (informative bar: the two
    # quantized stages compound, so the per-stage 1e-3 does not carry over)
    assert y_rel_err(Y, oracle.linear(oracle.gelu(Y_up_ref), Qd, sd_h, case.bs[1], G)) < 1e-2


def test_mlp_without_activation_is_two_linears(ops):
    """With no activation the chain is convrot_linear twice, bit for bit."""
    rng = workloads.rng_for(77)
    M, K, N1, N2, G1, G2 = 300, 1024, 768, 512, 256, 64
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=30.0)
    W1, W2 = workloads.weights(rng, N1, K), workloads.weights(rng, N2, N1)
    b1, b2 = workloads.biases(rng, N1), workloads.biases(rng, N2)
    _, s1, h1, k1 = prepared(ops, W1, G1)
    _, s2, h2, k2 = prepared(ops, W2, G2)
    Y = host(ops.convrot_mlp(dev(X), G1, (h1, s1, dev(b1), k1), ops.ACT_NONE, G2, (h2, s2, dev(b2), k2)))
    (Y1,) = ops.convrot_linear(dev(X), G1, [h1], [s1], [dev(b1)])
    (Y2,) = ops.convrot_linear(Y1, G2, [h2], [s2], [dev(b2)])
    np.testing.assert_array_equal(Y, host(Y2))
