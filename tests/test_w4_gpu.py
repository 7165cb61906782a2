"""The packed INT4 convrot weight format on the GPU ("INT8 Convrot
Safetensors", section "Packed INT4 convrot": signed 4-bit weights, low nibble
first, F32 per-output weight scales, INT8 convrot activations).

The S8 x S4 GEMM reads the packed bytes as they are. Its int32 product must be
bit-exact against the oracle's unpack and integer GEMM, at the DiT sizes and on
ragged shapes. That holds for split waves, for every tile height, and for
extreme codes at the largest K (the whole sum stays exact in fp32). The W4A4
linear (pack, S8 x S4 GEMM, reconstruction) matches the oracle within the Y
bar. On the GPU's own codes and scales it is bit-exact, whether alone, mixed
with binary16-weight linears in one call, or inside the MLP pair. The offline
expansion of the same bytes into int8 / binary16 codes matches the unpack.
"""
import numpy as np
import pytest
import torch

import oracle
from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from parity import assert_y

pytestmark = pytest.mark.gpu


def packed_weights(seed, N, K):
    return workloads.packed_int4(workloads.rng_for(seed), N, K)


def codes(seed, rows, cols, amp=127):
    return workloads.random_codes(workloads.rng_for(seed), rows, cols, -amp, amp)


@pytest.mark.parametrize("N,K", [(1, 16), (3, 48), (300, 3072), (129, 1280)])  # (1, 16), (3, 48): odd pack counts
def test_w4_expand_matches_unpack(ops, N, K):
    P = packed_weights(N + K, N, K)
    q8, q16 = ops.convrot_w4_expand(dev(P), K)
    ref = oracle.unpack_w4(P)
    np.testing.assert_array_equal(host(q8), ref)
    np.testing.assert_array_equal(host(q16).astype(np.int32), ref.astype(np.int32))


@pytest.mark.parametrize("M,N,K", [
    (4608, 3072, 3072),     # one DiT projection: 18 x 12 tiles of 256 x 256
    (4608, 9216, 3072),     # the three projections' rows as one weight: 648 tiles, split waves
    (4608, 3072, 12288),    # the MLP down linear's K
    (1000, 1284, 1280),     # ragged M and N (N % 256 != 0), 192-row tiles
    (37, 260, 64),          # one K block, a partial weight tile, 128-row tiles
    (300, 512, 16384),      # the largest K
])
def test_s8s4_int32_exact(ops, M, N, K):
    Qx = codes(M + 3 * K, M, K)
    P = packed_weights(N + 5 * K, N, K)
    A = host(ops.int8_gemm_s32_w4(dev(Qx), dev(P)))
    np.testing.assert_array_equal(A, oracle.gemm_s32(Qx, oracle.unpack_w4(P)))
    assert ops.convrot_device_status() == ops.OK


def test_s8s4_extremes_at_the_largest_k(ops):
    """+-127 activation codes against -8 / +7 weights over K = 16384: sums of
    magnitude 127 * 8 * 16384 = 16,646,144, just under 2^24."""
    M, N, K = 256, 256, 16384
    Qx = np.full((M, K), 127, np.int8)
    Qx[1::2] = -127
    P = np.full((N, K // 2), 0x88, np.uint8)   # every nibble 8: value -8
    P[1::2] = 0x77                             # value 7
    A = host(ops.int8_gemm_s32_w4(dev(Qx), dev(P)))
    ref = oracle.gemm_s32(Qx, oracle.unpack_w4(P))
    assert np.abs(ref).max() == 127 * 8 * K
    np.testing.assert_array_equal(A, ref)


def _w4_linears(seed, Ns, K):
    rng = workloads.rng_for(seed)
    Ps = [workloads.packed_int4(rng, n, K) for n in Ns]
    s_ws = [(0.001 + 0.01 * rng.random(n)).astype(np.float32) for n in Ns]
    bs = [workloads.biases(rng, n) for n in Ns]
    return Ps, s_ws, bs


def test_w4a4_dit_projections(ops):
    """The DiT attention input with three W4A4 projections sharing one pack:
    within the Y bar of the oracle chain, and bit-exact on the GPU's own codes."""
    w = workloads.get("dit_qkv")
    case = workloads.make_case(w)
    K, G = w.K, w.G
    Ps, s_ws, bs = _w4_linears(20, w.Ns, K)
    Xd = dev(case.X)
    Ys = ops.convrot_linear(Xd, G, [dev(P) for P in Ps], [dev(s) for s in s_ws], [dev(b) for b in bs])
    Qx, s_x = ops.convrot_pack_activations(Xd, G)
    Qx, s_x = host(Qx), host(s_x)
    Qo, so = oracle.pack(case.X[:512], G)
    for j, P in enumerate(Ps):
        Qw = oracle.unpack_w4(P)
        Yg = host(Ys[j])
        # bit-exact: the oracle's integer GEMM and reconstruction on the GPU's codes and scales
        np.testing.assert_array_equal(Yg, oracle.reconstruct(oracle.gemm_s32(Qx, Qw), s_x, s_ws[j], bs[j]))
        # the oracle's own pack on a row sample
        assert_y(Yg[:512], oracle.reconstruct(oracle.gemm_s32(Qo, Qw), so, s_ws[j], bs[j]))
    assert ops.convrot_device_status() == ops.OK


@pytest.mark.parametrize("M", [1, 130, 1000, 4352])
def test_w4a4_mixed_with_binary16_weights(ops, M):
    """One call with a W4A4 linear, a binary16-weight linear and another W4A4
    linear (ragged M): each output equals the oracle's on the GPU's codes."""
    rng = workloads.rng_for(M + 77)
    K, G = 1280, 64
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=20.0)
    Ps, s_ws, bs = _w4_linears(M + 78, (512, 768), K)
    W8 = workloads.weights(rng, 640, K)
    b8 = workloads.biases(rng, 640)
    q8, s8, q16 = ops.convrot_prepare_weight(dev(W8), G)
    qs = [dev(Ps[0]), q16, dev(Ps[1])]
    Ys = ops.convrot_linear(dev(X), G, qs, [dev(s_ws[0]), s8, dev(s_ws[1])], [dev(bs[0]), dev(b8), dev(bs[1])])
    Qx, s_x = ops.convrot_pack_activations(dev(X), G)
    Qx, s_x = host(Qx), host(s_x)
    refs = [oracle.reconstruct(oracle.gemm_s32(Qx, oracle.unpack_w4(Ps[0])), s_x, s_ws[0], bs[0]),
            oracle.reconstruct(oracle.gemm_s32(Qx, host(q8)), s_x, host(s8), b8),
            oracle.reconstruct(oracle.gemm_s32(Qx, oracle.unpack_w4(Ps[1])), s_x, s_ws[1], bs[1])]
    for y, r in zip(Ys, refs):
        np.testing.assert_array_equal(host(y), r)
    assert ops.convrot_device_status() == ops.OK


def test_w4a4_split_equals_whole_tiles_and_input_scale(ops):
    """648 tiles of 256 x 256: the split last waves give the same Y as whole
    tiles; an input scale (the unscaling kernel) matches the oracle."""
    w = workloads.get("dit_qkv")
    case = workloads.make_case(w)
    K, G = w.K, w.G
    Ps, s_ws, bs = _w4_linears(21, w.Ns, K)
    qs, ss, bb = [dev(P) for P in Ps], [dev(s) for s in s_ws], [dev(b) for b in bs]
    Q16, s16 = ops.convrot_pack_activations_f16(dev(case.X), G)
    whole = [host(y) for y in ops.convrot_linear_packed(Q16, s16, qs, ss, bb, split_tail=False)]
    split = [host(y) for y in ops.convrot_linear_packed(Q16, s16, qs, ss, bb)]
    for a, b in zip(whole, split):
        np.testing.assert_array_equal(a, b)
    a = 0.37
    Ys = ops.convrot_linear_scaled(dev(case.X), G, a, qs, ss, bb)
    for j in range(3):
        ref = oracle.linear_scaled(case.X[:256], oracle.unpack_w4(Ps[j]), s_ws[j], bs[j], G, a)
        assert_y(host(Ys[j])[:256], ref)
    assert ops.convrot_device_status() == ops.OK


def test_w4a4_mlp_pair(ops):
    """The MLP pair with W4A4 up and down linears: H = GELU of the up output
    (exact on the GPU's codes, then the device GELU in the S8 x S4 GEMM's
    epilogue), then the down linear on the GPU's own H within the Y bar."""
    M, K, N_up, G = 512, 1024, 2048, 256
    rng = workloads.rng_for(31)
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=40.0)
    (Pu,), (su,), (bu,) = _w4_linears(32, (N_up,), K)
    (Pd,), (sd,), (bd,) = _w4_linears(33, (K,), N_up)
    H = torch.empty((M, N_up), dtype=torch.float32, device="cuda")
    Y = ops.convrot_mlp(dev(X), G, (dev(Pu), dev(su), dev(bu), None), ops.ACT_GELU, G,
                        (dev(Pd), dev(sd), dev(bd), None), H=H)
    Qx, s_x = ops.convrot_pack_activations(dev(X), G)
    Hg = host(H)
    # H = GELU(Y_up) from the S8 x S4 GEMM's epilogue: the exact reconstruction, then the device GELU
    Y_up = oracle.reconstruct(oracle.gemm_s32(host(Qx), oracle.unpack_w4(Pu)), host(s_x), su, bu)
    Href = oracle.gelu(Y_up).astype(np.float64)
    assert np.max(np.abs(Hg - Href)) <= 1e-5 * np.max(np.abs(Href))
    ref = oracle.linear(Hg, oracle.unpack_w4(Pd), sd, bd, G)
    assert_y(host(Y), ref)
    assert ops.convrot_device_status() == ops.OK


def test_w4_argument_rules(ops):
    """K % 64, K <= CONVROT_W4_MAX_K and N % 4 are checked before any launch."""
    X = torch.zeros((4, 96), dtype=torch.float32, device="cuda")
    P = torch.zeros((8, 48), dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.ConvrotError) as e:
        ops.convrot_linear(X, 16, [P], [None], [None])
    assert e.value.status == ops.ERR_ALIGN
    X = torch.zeros((4, 128), dtype=torch.float32, device="cuda")
    P = torch.zeros((6, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.ConvrotError) as e:
        ops.convrot_linear(X, 16, [P], [None], [None])
    assert e.value.status == ops.ERR_ALIGN
    Qx = torch.zeros((4, 16384 + 64), dtype=torch.int8, device="cuda")
    P = torch.zeros((8, (16384 + 64) // 2), dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.ConvrotError) as e:
        ops.int8_gemm_s32_w4(Qx, P)
    assert e.value.status == ops.ERR_UNSUPPORTED
