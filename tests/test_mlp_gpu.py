"""convrot_mlp and convrot_linear_swiglu on the device (the DiT MLP shapes),
against the oracle stage by stage.

The up GEMM applies the activation in its epilogue and writes H: GELU
elementwise, or split SwiGLU h = silu(gate) * up of a gate and an up weight
sharing the input ("ggml operator extensions", sd.cpp integration). On the
GPU's own codes the reconstruction is exact, so H is compared with the oracle's
activation of the exact reconstruction: the device evaluates GELU with the
Abramowitz & Stegun 7.1.28 erf (within 5e-7 |y| of the exact GELU) and SiLU
with the hardware exponential, the oracle both in fp64. The down linear is then
checked on the GPU's own H. The GELU repack (convrot_pack_gelu_f16, the other
place the activation can go) is checked against the oracle's pack of GELU(X).
"""
import numpy as np
import pytest
import torch

import oracle
from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from parity import assert_y, y_rel_err

pytestmark = pytest.mark.gpu

ACT_REL = 1e-5  # fp32 activation against its fp64 definition, relative to max |H|


def prepared(ops, W, G):
    q8, s_w, q16 = ops.convrot_prepare_weight(dev(W), G)
    return q8, s_w, q16, ops.convrot_weight_chunks(q8)


def assert_act(Hg, Href, what):
    err = float(np.max(np.abs(Hg.astype(np.float64) - Href)) / np.max(np.abs(Href)))
    assert err <= ACT_REL, f"{what}: max rel err {err:.2e}"


@pytest.mark.parametrize("M", [600, 37])
def test_dit_mlp_gelu_on_device(ops, M):
    w = workloads.get("dit_mlp")
    case = workloads.make_case(w, M=M)
    G = w.G
    qu, su, hu, ku = prepared(ops, case.Ws[0], G)
    qd, sd, hd, kd = prepared(ops, case.Ws[1], G)
    bu, bd = dev(case.bs[0]), dev(case.bs[1])
    H = torch.empty((M, w.Ns[0]), dtype=torch.float32, device="cuda")
    Y = ops.convrot_mlp(dev(case.X), G, (hu, su, bu, ku), ops.ACT_GELU, G, (hd, sd, bd, kd), H=H)
    H, Y = host(H), host(Y)
    assert ops.convrot_device_status() == ops.OK
    # stage 1: the up linear and its GELU, on the GPU's codes of X
    Qx, s_x = ops.convrot_pack_activations(dev(case.X), G)
    Qu, su_h = host(qu), host(su)
    Y_up = oracle.reconstruct(oracle.gemm_s32(host(Qx), Qu), host(s_x), su_h, case.bs[0])
    assert_act(H, oracle.gelu(Y_up), "GELU(Y_up)")
    # and against the oracle's own pack
    Y_up_ref = oracle.linear(case.X, Qu, su_h, case.bs[0], G)
    assert_y(H, oracle.gelu(Y_up_ref), "H")
    # stage 2: the down linear on the GPU's own H
    Qd, sd_h = host(qd), host(sd)
    assert_y(Y, oracle.linear(H, Qd, sd_h, case.bs[1], G), "down on the same H")
    # the whole chain against the oracle chain (informative bar: the two
    # quantized stages compound, so the per-stage 1e-3 does not carry over)
    assert y_rel_err(Y, oracle.linear(oracle.gelu(Y_up_ref), Qd, sd_h, case.bs[1], G)) < 1e-2


@pytest.mark.parametrize("M,K,G", [(600, 12288, 256), (37, 3072, 64)])
def test_gelu_repack(ops, M, K, G):
    """The repack's GELU prologue: the codes and scales of GELU(X) within the
    pack bars (the device's GELU is within 3e-7 |x| of the exact one, so a
    code can move by one where the quotient is that close to a half)."""
    from parity import assert_codes, assert_scales
    rng = workloads.rng_for(M + K)
    X = (workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=10.0) * 2.0).astype(np.float32)
    Q16, s = ops.convrot_pack_gelu_f16(dev(X), G)
    Qo, so = oracle.pack(oracle.gelu(X), G)
    assert_scales(host(s), so)
    assert_codes(host(Q16).astype(np.int32), Qo)


def test_gelu_epilogue(ops):
    """GELU in the GEMM's epilogue (convrot_linear_packed_act) on the DiT MLP's
    up linear: a shape whose last wave splits (4608 rows x 12288 features = 864
    tiles of 256 x 256 over 76 pairs), exact reconstruction on the GPU's codes,
    then the device GELU against the fp64 definition."""
    w = workloads.get("dit_mlp")
    case = workloads.make_case(w)
    G = w.G
    qu, su, hu, ku = prepared(ops, case.Ws[0], G)
    Q16, s16 = ops.convrot_pack_activations_f16(dev(case.X), G)
    (H,) = ops.convrot_linear_packed_act(Q16, s16, [hu], [su], [dev(case.bs[0])], ops.ACT_GELU, kchunks=[ku])
    Qx, s_x = ops.convrot_pack_activations(dev(case.X), G)
    rows = slice(0, 512)
    Y_up = oracle.reconstruct(oracle.gemm_s32(host(Qx)[rows], host(qu)), host(s_x)[rows], host(su), case.bs[0])
    assert_act(host(H)[rows], oracle.gelu(Y_up), "GELU(Y_up) in the epilogue with split waves")
    assert ops.convrot_device_status() == ops.OK


@pytest.mark.parametrize("M,K,N,G", [(600, 3072, 2048, 256), (37, 1280, 1284, 64), (4608, 3072, 3072, 256)])
def test_linear_swiglu(ops, M, K, N, G):
    """h = silu(gate) * up from one pack and one GEMM: the exact reconstruction
    of both linears on the GPU's codes, then the fp32 SiLU product."""
    rng = workloads.rng_for(M + N)
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=40.0)
    Wg, Wu = workloads.weights(rng, N, K), workloads.weights(rng, N, K)
    bg, bu = workloads.biases(rng, N), workloads.biases(rng, N)
    qg, sg, hg, kg = prepared(ops, Wg, G)
    qu, su, hu, ku = prepared(ops, Wu, G)
    H = host(ops.convrot_linear_swiglu(dev(X), G, (hg, sg, dev(bg), kg), (hu, su, dev(bu), ku)))
    assert ops.convrot_device_status() == ops.OK
    Qx, s_x = ops.convrot_pack_activations(dev(X), G)
    Qx, s_x = host(Qx), host(s_x)
    gate = oracle.reconstruct(oracle.gemm_s32(Qx, host(qg)), s_x, host(sg), bg)
    up = oracle.reconstruct(oracle.gemm_s32(Qx, host(qu)), s_x, host(su), bu)
    assert_act(H, oracle.silu_mul(gate, up), "silu(gate) * up")
    rows = slice(0, min(M, 256))
    assert_y(H[rows], oracle.linear_swiglu(X[rows], host(qg), host(sg), bg, host(qu), host(su), bu, G), "h")


def test_dit_mlp_swiglu_on_device(ops):
    """The MLP pair with split SwiGLU: gate and up [N_up, K] sharing the pack,
    H = silu(gate) * up, then the down linear on the GPU's own H."""
    M, K, N_up, G = 512, 3072, 4096, 256
    rng = workloads.rng_for(91)
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=40.0)
    Wg, Wu, Wd = workloads.weights(rng, N_up, K), workloads.weights(rng, N_up, K), workloads.weights(rng, K, N_up)
    bg, bu, bd = workloads.biases(rng, N_up), workloads.biases(rng, N_up), workloads.biases(rng, K)
    g, u, d = prepared(ops, Wg, G), prepared(ops, Wu, G), prepared(ops, Wd, G)
    H = torch.empty((M, N_up), dtype=torch.float32, device="cuda")
    Y = ops.convrot_mlp(dev(X), G, ((g[2], g[1], dev(bg), g[3]), (u[2], u[1], dev(bu), u[3])), ops.ACT_SWIGLU, G,
                        (d[2], d[1], dev(bd), d[3]), H=H)
    H, Y = host(H), host(Y)
    assert ops.convrot_device_status() == ops.OK
    Qx, s_x = ops.convrot_pack_activations(dev(X), G)
    Qx, s_x = host(Qx), host(s_x)
    gate = oracle.reconstruct(oracle.gemm_s32(Qx, host(g[0])), s_x, host(g[1]), bg)
    up = oracle.reconstruct(oracle.gemm_s32(Qx, host(u[0])), s_x, host(u[1]), bu)
    assert_act(H, oracle.silu_mul(gate, up), "H")
    assert_y(Y, oracle.linear(H, host(d[0]), host(d[1]), bd, G), "down on the same H")


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


@pytest.mark.parametrize("act,M,chunk_rows,x_dtype", [("gelu", 1000, 384, "f32"), ("swiglu", 700, 256, "f32"),
                                                       ("gelu", 4608, 0, "f32"), ("gelu", 520, 256, "f16")])
def test_mlp_host_equals_device_call(ops, act, M, chunk_rows, x_dtype):
    """convrot_mlp_host (host X and Y, row chunks whose copies overlap the
    other chunks' compute; a ragged last chunk in the first two cases, the
    default chunks on the DiT MLP in the last) gives convrot_mlp's output bit
    for bit: the rows are independent and every step is exact or rounds the
    same values in the same order."""
    K, G = 3072, 256
    N_up = 12288 if M == 4608 else 4096
    rng = workloads.rng_for(M + N_up)
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=40.0, dtype=x_dtype)
    Wu, Wd = workloads.weights(rng, N_up, K), workloads.weights(rng, K, N_up)
    bu, bd = workloads.biases(rng, N_up), workloads.biases(rng, K)
    u, d = prepared(ops, Wu, G), prepared(ops, Wd, G)
    up = (u[2], u[1], dev(bu), u[3])
    if act == "swiglu":
        Wg, bg = workloads.weights(rng, N_up, K), workloads.biases(rng, N_up)
        g = prepared(ops, Wg, G)
        up = ((g[2], g[1], dev(bg), g[3]), up)
    a = ops.ACT_SWIGLU if act == "swiglu" else ops.ACT_GELU
    down = (d[2], d[1], dev(bd), d[3])
    Y_dev = host(ops.convrot_mlp(dev(X), G, up, a, G, down))
    Xh = torch.from_numpy(X).pin_memory()
    copy_in, copy_out = torch.cuda.Stream(), torch.cuda.Stream()
    Y_host = ops.convrot_mlp_host(Xh, G, up, a, G, down, chunk_rows=chunk_rows, copy_in_stream=copy_in,
                                  copy_out_stream=copy_out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(Y_host.numpy(), Y_dev)
    assert ops.convrot_device_status() == ops.OK
