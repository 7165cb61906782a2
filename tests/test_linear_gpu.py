"""GPU parity of the fused convrot linear (one pack, one grouped GEMM) against
the oracle on the seeded workloads, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from parity import assert_y, y_rel_err

pytestmark = pytest.mark.gpu


def prepared(ops, W, G):
    Qw, s_w, Qw16 = ops.convrot_prepare_weight(dev(W), G)
    return Qw, s_w, Qw16


def run_linear(ops, X, Ws, bs, G):
    preps = [prepared(ops, W, G) for W in Ws]
    Ys = ops.convrot_linear(dev(X), G, [p[2] for p in preps], [p[1] for p in preps], [dev(b) for b in bs])
    return [host(y) for y in Ys], [(host(p[0]), host(p[1])) for p in preps]


def oracle_linear(X, Ws, bs, G, gpu_weights=None):
    """Oracle Y. With gpu_weights, the oracle uses the GPU's weight codes so
    that only the activation path is compared."""
    out = []
    for j, (W, b) in enumerate(zip(Ws, bs)):
        if gpu_weights is None:
            Qw, s_w = oracle.prepare_weight(W, G)
        else:
            Qw, s_w = gpu_weights[j]
        out.append(oracle.linear(X, Qw, s_w, b, G))
    return out


def check_workload(ops, name):
    w = workloads.get(name)
    case = workloads.make_case(w)
    Ys, gw = run_linear(ops, case.X, case.Ws, case.bs, w.G)
    refs = oracle_linear(case.X, case.Ws, case.bs, w.G)
    errs = [assert_y(y, r, f"{name} Y{j}") for j, (y, r) in enumerate(zip(Ys, refs))]
    # with the GPU's own weight codes the only remaining difference is the
    # rare +-1 activation code
    refs2 = oracle_linear(case.X, case.Ws, case.bs, w.G, gpu_weights=gw)
    for y, r in zip(Ys, refs2):
        assert_y(y, r)
    assert ops.convrot_device_status() == ops.OK
    return errs


def test_tiny(ops):
    check_workload(ops, "tiny")


def test_unet_fp16(ops):
    check_workload(ops, "unet")


def test_dit_qkv_shared_pack(ops):
    check_workload(ops, "dit_qkv")


def test_dit_mlp_pair(ops):
    """Up linear, host GELU, repack, down linear. Stage-wise parity: the down
    stage gets the same host GELU(Y_up_oracle) array on both sides."""
    w = workloads.get("dit_mlp")
    case = workloads.make_case(w)
    G = w.G
    (Y_up,), _ = run_linear(ops, case.X, case.Ws[:1], case.bs[:1], G)
    Qw_up, sw_up = oracle.prepare_weight(case.Ws[0], G)
    Y_up_ref = oracle.linear(case.X, Qw_up, sw_up, case.bs[0], G)
    assert_y(Y_up, Y_up_ref, "mlp up")
    H = oracle.gelu(Y_up_ref)
    (Y_dn,), _ = run_linear(ops, H, case.Ws[1:], case.bs[1:], G)
    Qw_dn, sw_dn = oracle.prepare_weight(case.Ws[1], G)
    Y_dn_ref = oracle.linear(H, Qw_dn, sw_dn, case.bs[1], G)
    assert_y(Y_dn, Y_dn_ref, "mlp down")
    # end-to-end chain (informative): GPU up -> host GELU of the GPU output -> GPU down
    (Y_chain,), _ = run_linear(ops, oracle.gelu(Y_up), case.Ws[1:], case.bs[1:], G)
    assert y_rel_err(Y_chain, Y_dn_ref) < 1e-2


@pytest.mark.parametrize("M,K,Ns,G", [
    (1, 64, (1,), 64), (5, 256, (129, 7), 16), (300, 1024, (256, 130, 385), 1024),
    (257, 1280, (64,), 4), (100, 48, (33,), 1),
])
def test_ragged_grouped(ops, M, K, Ns, G):
    rng = workloads.rng_for(M + K + G)
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=30.0)
    Ws = [workloads.weights(rng, n, K) for n in Ns]
    bs = [workloads.biases(rng, n) for n in Ns]
    Ys, gw = run_linear(ops, X, Ws, bs, G)
    refs = oracle_linear(X, Ws, bs, G, gpu_weights=gw)
    for y, r in zip(Ys, refs):
        assert_y(y, r)


def test_optional_scale_and_bias(ops):
    rng = workloads.rng_for(77)
    X = workloads.activations(rng, 64, 256)
    W = workloads.weights(rng, 96, 256)
    Qw, s_w, Qw16 = prepared(ops, W, 256)
    Y0, Y1 = ops.convrot_linear(dev(X), 256, [Qw16, Qw16], [None, s_w], [None, None])
    Qx, s_x = oracle.pack(X, 256)
    A = oracle.gemm_s32(Qx, host(Qw))
    assert_y(host(Y0), oracle.reconstruct(A, s_x))
    assert_y(host(Y1), oracle.reconstruct(A, s_x, host(s_w)))


def test_alias_rejected(ops):
    X = torch.randn(64, 256, device="cuda")
    W = torch.randn(64, 256, device="cuda")
    _, s_w, Qw16 = ops.convrot_prepare_weight(W, 256)
    with pytest.raises(ops.ConvrotError) as e:
        ops.convrot_linear(X, 256, [Qw16], [s_w], [None], Ys=[X.view(64, 256)])
    assert e.value.status == ops.ERR_ALIAS


def test_packed_entry_points_match_fused_call(ops):
    """convrot_pack_activations_f16 writes the int8 pack's codes as fp16, and
    convrot_linear_packed on them equals the one-call convrot_linear."""
    w = workloads.get("unet")
    case = workloads.make_case(w)
    X = dev(case.X)
    Q8, s8 = ops.convrot_pack_activations(X, w.G)
    Q16, s16 = ops.convrot_pack_activations_f16(X, w.G)
    np.testing.assert_array_equal(host(Q16).astype(np.int32), host(Q8).astype(np.int32))
    np.testing.assert_array_equal(host(s16), host(s8))
    _, s_w, Qw16 = ops.convrot_prepare_weight(dev(case.Ws[0]), w.G)
    b = dev(case.bs[0])
    (Ya,) = ops.convrot_linear(X, w.G, [Qw16], [s_w], [b])
    (Yb,) = ops.convrot_linear_packed(Q16, s16, [Qw16], [s_w], [b])
    np.testing.assert_array_equal(host(Ya), host(Yb))
    # and the packed GEMM equals int8_linear on the int8 codes
    Yc = ops.int8_linear(Q8, s8, Q_w16=Qw16, s_w=s_w, bias=b)
    np.testing.assert_array_equal(host(Yc), host(Ya))


@pytest.mark.parametrize("M,K,Ns,G,xd,chunk,streams", [
    (1000, 1280, (1280,), 256, "f16", 256, True),       # ragged last chunk
    (4608, 3072, (3072, 3072, 3072), 256, "f32", 0, True),  # the DiT projections, default chunks
    (300, 512, (256, 96), 64, "f32", 1024, True),        # one chunk larger than M
    (513, 256, (128,), 4, "f32", 128, False),           # no copy streams: serialized
])
def test_host_pipeline_matches_device_call(ops, M, K, Ns, G, xd, chunk, streams):
    """convrot_linear_host (host X and Y, chunked, overlapped transfers) gives
    exactly convrot_linear's outputs."""
    rng = workloads.rng_for(M + K + sum(Ns))
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=40.0, dtype=xd)
    Ws = [workloads.weights(rng, n, K) for n in Ns]
    bs = [workloads.biases(rng, n) for n in Ns]
    preps = [ops.convrot_prepare_weight(dev(W), G) for W in Ws]
    q16s, scales, biases = [p[2] for p in preps], [p[1] for p in preps], [dev(b) for b in bs]
    Y_ref = [host(y) for y in ops.convrot_linear(dev(X), G, q16s, scales, biases)]
    Xh = torch.from_numpy(X).pin_memory()
    kw = {}
    if streams:
        kw = dict(copy_in_stream=torch.cuda.Stream(), copy_out_stream=torch.cuda.Stream())
    Ys = ops.convrot_linear_host(Xh, G, q16s, scales, biases, chunk_rows=chunk, **kw)
    torch.cuda.current_stream().synchronize()
    assert ops.convrot_device_status() == ops.OK
    for y, r in zip(Ys, Y_ref):
        np.testing.assert_array_equal(y.numpy(), r)


@pytest.mark.parametrize("a", [1.0, 0.25, 3.0, 0.37])
def test_input_scale(ops, a):
    """convrot_linear_scaled against the oracle's scaled linear; power-of-two
    scales give exactly the unscaled output (the oracle pins why)."""
    w = workloads.get("unet")
    case = workloads.make_case(w, M=333)
    G = w.G
    Qw, s_w, Qw16 = ops.convrot_prepare_weight(dev(case.Ws[0]), G)
    (Y,) = ops.convrot_linear_scaled(dev(case.X), G, a, [Qw16], [s_w], [dev(case.bs[0])])
    Y = host(Y)
    ref = oracle.linear_scaled(case.X, host(Qw), host(s_w), case.bs[0], G, a)
    assert_y(Y, ref)
    if a in (1.0, 0.25):
        (Y1,) = ops.convrot_linear(dev(case.X), G, [Qw16], [s_w], [dev(case.bs[0])])
        np.testing.assert_array_equal(Y, host(Y1))


def test_input_scale_epilogue_bit_exact(ops):
    """The scaled linear on the DiT projections (staged Y stores, split
    waves) equals, bit for bit, the reconstruction formed on the host in fp32
    from the raw int32 product of the codes it packed:
    ((float(A) * s_x) * s_w) / a + b, one rounding per operation, in that
    order."""
    w = workloads.get("dit_qkv")
    case = workloads.make_case(w)
    M, K, G, a = w.M, w.K, w.G, np.float32(0.37)
    preps = [ops.convrot_prepare_weight(dev(W), G) for W in case.Ws]
    q16s, scales = [p[2] for p in preps], [p[1] for p in preps]
    biases = [dev(b) for b in case.bs]
    ws = torch.empty((ops.convrot_linear_workspace_size(M, K),), dtype=torch.uint8, device="cuda")
    Ys = ops.convrot_linear_scaled(dev(case.X), G, float(a), q16s, scales, biases, workspace=ws)
    Q8 = ws[: M * K * 2].view(torch.float16).view(M, K).to(torch.int8)
    off = (M * K * 2 + 255) // 256 * 256
    s_x = host(ws[off: off + 4 * M].view(torch.float32))
    for j in range(3):
        A = host(ops.int8_gemm_s32(Q8, Q_w16=q16s[j]))
        ref = (A.astype(np.float32) * s_x[:, None]) * host(scales[j])[None, :]
        ref = ref / a + case.bs[j][None, :]
        np.testing.assert_array_equal(host(Ys[j]), ref)
    assert ops.convrot_device_status() == ops.OK


def _sweep_divisors():
    """Divisors for the unscaling sweep: every significand pattern class that
    matters to a reciprocal (1, just above 1, just below 2, all ones, thirds,
    tenths), the scales the tests use, and seeded random significands, at
    exponents across the step's range [2^-20, 2^20]."""
    rng = np.random.default_rng(20241)
    sig = [1.0, 1.0 + 2.0 ** -23, 1.0 + 2.0 ** -22, 2.0 - 2.0 ** -23, 2.0 - 2.0 ** -22, 1.5, 1.25, 1.75,
           4.0 / 3.0, 5.0 / 3.0, 1.1, 1.2, 1.3, 1.4, 1.6, 1.7, 1.8, 1.9, 0.37 * 4, 0.5 * 3]
    sig = [float(np.float32(v)) for v in sig]
    sig += list(1.0 + rng.integers(0, 1 << 23, size=4096 - len(sig)) * 2.0 ** -23)
    exps = rng.integers(-20, 20, size=len(sig))
    exps[:len(exps) // 8] = 0
    d = np.ldexp(np.asarray(sig, np.float64), exps).astype(np.float32)
    return d


@pytest.mark.parametrize("y_exp", [0, -98, 97])
def test_unscale_step_equals_ieee_division(ops, y_exp):
    """The epilogue's division by the input scale (Markstein's correction step
    after a correctly rounded reciprocal) against the GPU's IEEE division, for
    4096 divisors and all 2^23 significands of y each (the step's results scale
    exactly with the exponents of y and a inside its range, so the significands
    at the range ends and in the middle cover it)."""
    d = torch.from_numpy(_sweep_divisors()).cuda()
    n, first = ops.convrot_test_unscale_sweep(d, y_exp)
    assert n == 0, f"{n} results differ, the first at divisor {first[0]!r}, y {first[1]!r}"


@pytest.mark.parametrize("a", [np.float32(0.37), np.float32(1.0 / 3.0), np.float32(2.0 - 2.0 ** -22),
                               np.float32(1.0e-7), np.float32(3.0e6)])
def test_input_scale_epilogue_bit_exact_scales(ops, a):
    """The scaled linear on the DiT projections equals, bit for bit, the
    host's fp32 reconstruction ((float(A) * s_x) * s_w) / a + b with the
    IEEE division, for divisors inside the correction step's range and
    outside it (1e-7 and 3e6 take the division), with rows of tiny
    activations (row scales near 1e-36, whose tiles take the division) mixed
    in."""
    w = workloads.get("dit_qkv")
    case = workloads.make_case(w, M=1000)
    X = case.X.copy()
    X[17] *= np.float32(1e-38)
    X[600:603] *= np.float32(1e-35)
    M, K, G = X.shape[0], w.K, w.G
    preps = [ops.convrot_prepare_weight(dev(W), G) for W in case.Ws]
    q16s, scales = [p[2] for p in preps], [p[1] for p in preps]
    biases = [dev(case.bs[0]), None, dev(case.bs[2])]
    ws = torch.empty((ops.convrot_linear_workspace_size(M, K),), dtype=torch.uint8, device="cuda")
    Ys = ops.convrot_linear_scaled(dev(X), G, float(a), q16s, scales, biases, workspace=ws)
    Q8 = ws[: M * K * 2].view(torch.float16).view(M, K).to(torch.int8)
    off = (M * K * 2 + 255) // 256 * 256
    s_x = host(ws[off: off + 4 * M].view(torch.float32))
    assert s_x[17] < 1e-30 * s_x[0] and s_x[601] < 1e-27 * s_x[0]
    for j in range(3):
        A = host(ops.int8_gemm_s32(Q8, Q_w16=q16s[j]))
        ref = (A.astype(np.float32) * s_x[:, None]) * host(scales[j])[None, :]
        ref = ref / a
        if biases[j] is not None:
            ref = ref + case.bs[j][None, :]
        np.testing.assert_array_equal(host(Ys[j]).view(np.uint32), ref.astype(np.float32).view(np.uint32))
    assert ops.convrot_device_status() == ops.OK
