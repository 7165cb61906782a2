"""GPU checks of the GEMM's work distribution: split waves (the K-split whose
partial int32 sums pass between CTA pairs through the tile's output and a
hand-over word). The int32 product stays bit-exact against the oracle on
ragged shapes that take this path (odd band counts included), results are identical with and
without the split, the hand-over words are left zero after use, and a
CUDA-graph replay (the same launch, hence the same hand-over value, again and
again) stays correct."""
import numpy as np
import pytest
import torch

import oracle
from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from split_tail_ref import plan_split

pytestmark = pytest.mark.gpu


def codes(seed, rows, cols, amp=127):
    rng = workloads.rng_for(seed)
    return workloads.random_codes(rng, rows, cols, -amp, amp)


@pytest.mark.parametrize("M,N,K,use_plan", [
    (2597, 2148, 4160, True),    # 11 x 9 tiles of 256 x 256: 99 tiles over the pairs, ragged edges
    (2597, 2148, 4160, False),   # the same with the fixed 1024-product chunks
    (768, 9216, 3072, True),     # a host-pipeline chunk of the DiT projections: 108 tiles
    (300, 20000, 1040, False),   # 2 x 79 tiles, K not a multiple of 1024
    (1024, 9472, 3072, True),    # 148 tiles: under two waves, whole tiles
    (4608, 3072, 12288, True),   # 216 tiles, K = 12288 in runs of >= 4096
])
def test_exact_int32_with_split_tiles(ops, M, N, K, use_plan):
    Qx = codes(M + K, M, K)
    Qw = codes(N + K, N, K)
    kc = ops.convrot_weight_chunks(dev(Qw)) if use_plan else None
    A = host(ops.int8_gemm_s32(dev(Qx), Q_w16=dev(Qw.astype(np.float16)), kchunk=kc))
    np.testing.assert_array_equal(A, oracle.gemm_s32(Qx, Qw))
    assert ops.convrot_device_status() == ops.OK


def _packed_case(name, M=None):
    w = workloads.get(name)
    case = workloads.make_case(w, M=M) if M else workloads.make_case(w)
    return w, case


@pytest.mark.parametrize("name,M,which", [
    ("dit_qkv", None, slice(0, 3)),    # 648 tiles: 7 whole waves, then 116 tiles split
    ("dit_mlp", None, slice(1, 2)),    # the down linear, K = 12288 in exact runs of >= 4096
    ("dit_qkv", 4352, slice(0, 3)),    # 17 bands: 612 tiles
    ("unet", None, slice(0, 1)),       # 80 tiles, every one split in two
])
def test_split_equals_whole_tiles(ops, name, M, which):
    w, case = _packed_case(name, M)
    Ws, bs = case.Ws[which], case.bs[which]
    K = Ws[0].shape[1]
    X = case.X if K == case.X.shape[1] else workloads.activations(workloads.rng_for(9), case.X.shape[0], K)
    Q16, s16 = ops.convrot_pack_activations_f16(dev(X), w.G)
    preps = [ops.convrot_prepare_weight(dev(W), w.G) for W in Ws]
    q16s, scales, biases = [p[2] for p in preps], [p[1] for p in preps], [dev(b) for b in bs]
    plans = [ops.convrot_weight_chunks(p[0]) for p in preps]
    Y_whole = [host(y) for y in ops.convrot_linear_packed(Q16, s16, q16s, scales, biases, kchunks=plans,
                                                          split_tail=False)]
    Y_split = [host(y) for y in ops.convrot_linear_packed(Q16, s16, q16s, scales, biases, kchunks=plans)]
    for a, b in zip(Y_whole, Y_split):
        np.testing.assert_array_equal(a, b)
    assert ops.convrot_device_status() == ops.OK


def test_handover_words_left_zero_and_reusable(ops):
    """Scratch that starts as garbage: after each call every word is either
    untouched or zero, some were used, and repeated calls on one workspace
    give the same Y as whole tiles."""
    w, case = _packed_case("dit_qkv", 2560)    # 10 bands x 36 weight tiles = 360 tiles
    Q16, s16 = ops.convrot_pack_activations_f16(dev(case.X), w.G)
    preps = [ops.convrot_prepare_weight(dev(W), w.G) for W in case.Ws]
    q16s, scales, biases = [p[2] for p in preps], [p[1] for p in preps], [dev(b) for b in case.bs]
    ref = [host(y) for y in ops.convrot_linear_packed(Q16, s16, q16s, scales, biases, split_tail=False)]
    ws = torch.full((ops.GEMM_SYNC_BYTES,), 0x5A, dtype=torch.uint8, device="cuda")
    garbage = np.full(8, 0x5A, dtype=np.uint8).view(np.uint64)[0]
    used = False
    for _ in range(3):
        Ys = ops.convrot_linear_packed(Q16, s16, q16s, scales, biases, workspace=ws)
        for a, b in zip(Ys, ref):
            np.testing.assert_array_equal(host(a), b)
        words = host(ws).view(np.uint64)
        assert np.all((words == garbage) | (words == 0))
        used |= bool(np.any(words == 0))
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    if plan_split(360, pairs):
        assert used
    assert ops.convrot_device_status() == ops.OK


def test_graph_replay_of_a_split_gemm(ops):
    """A captured GEMM replays with the hand-over value fixed at capture: the
    words it consumed are zero again after each replay, so every replay on
    new inputs matches an eager call."""
    w, case = _packed_case("dit_qkv", 2560)
    preps = [ops.convrot_prepare_weight(dev(W), w.G) for W in case.Ws]
    q16s, scales, biases = [p[2] for p in preps], [p[1] for p in preps], [dev(b) for b in case.bs]
    Q16 = torch.empty((2560, w.K), dtype=torch.float16, device="cuda")
    s16 = torch.empty((2560,), dtype=torch.float32, device="cuda")
    Ys = [torch.empty((2560, q.shape[0]), dtype=torch.float32, device="cuda") for q in q16s]
    ws = torch.zeros((ops.GEMM_SYNC_BYTES,), dtype=torch.uint8, device="cuda")
    weights = ops.make_weights(q16s, scales, biases, Ys)
    Xs = [dev(workloads.activations(workloads.rng_for(100 + i), 2560, w.K)) for i in range(3)]
    q, s = ops.convrot_pack_activations_f16(Xs[0], w.G)
    Q16.copy_(q)
    s16.copy_(s)
    ops.convrot_linear_packed(Q16, s16, q16s, scales, biases, Ys=Ys, weights=weights, workspace=ws)  # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ops.convrot_linear_packed(Q16, s16, q16s, scales, biases, Ys=Ys, weights=weights, workspace=ws)
    for X in Xs:
        q, s = ops.convrot_pack_activations_f16(X, w.G)
        Q16.copy_(q)
        s16.copy_(s)
        g.replay()
        got = [host(y) for y in Ys]
        want = [host(y) for y in ops.convrot_linear_packed(q, s, q16s, scales, biases, split_tail=False)]
        for a, b in zip(got, want):
            np.testing.assert_array_equal(a, b)
    assert ops.convrot_device_status() == ops.OK


def test_split_with_direct_stores_and_input_scale(ops):
    """Split waves on the kernels without the staged Y stores: N not a
    multiple of 4 (per-thread stores) and an input scale other than 1 (the
    unscaling variant). Identical to whole tiles; the scaled linear also
    matches the oracle."""
    rng = workloads.rng_for(4608 + 3070)
    M, K, G = 4608, 3072, 256
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=40.0)
    Ws = [workloads.weights(rng, 3070, K) for _ in range(3)]   # 18 bands x 12 weight tiles x 3 = 648 tiles
    bs = [workloads.biases(rng, 3070) for _ in range(3)]
    preps = [ops.convrot_prepare_weight(dev(W), G) for W in Ws]
    q16s, scales, biases = [p[2] for p in preps], [p[1] for p in preps], [dev(b) for b in bs]
    Q16, s16 = ops.convrot_pack_activations_f16(dev(X), G)
    whole = [host(y) for y in ops.convrot_linear_packed(Q16, s16, q16s, scales, biases, split_tail=False)]
    split = [host(y) for y in ops.convrot_linear_packed(Q16, s16, q16s, scales, biases)]
    for a, b in zip(whole, split):
        np.testing.assert_array_equal(a, b)
    a = 0.37   # all three linears: 648 tiles, so the unscaling kernel splits its last waves too
    Ys = ops.convrot_linear_scaled(dev(X), G, a, q16s, scales, biases)
    from parity import assert_y
    for j in range(3):
        ref = oracle.linear_scaled(X[:512], host(preps[j][0]), host(preps[j][1]), bs[j], G, a)
        assert_y(host(Ys[j])[:512], ref)
    assert ops.convrot_device_status() == ops.OK
