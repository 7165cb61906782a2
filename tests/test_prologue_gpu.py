"""The pack's modulation prologue (RMS norm, per-channel weight, modulation)
on the GPU against the oracle: codes and scales of pack(prologue(X)), and the
linear built on it."""
import numpy as np
import pytest
import torch

import oracle
from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from parity import assert_codes, assert_scales, assert_y

pytestmark = pytest.mark.gpu


def vectors(seed, K):
    return workloads.modulation(workloads.rng_for(seed), K)


@pytest.mark.parametrize("M,K,G", [(4608, 3072, 256), (37, 1280, 64), (9, 48, 4), (130, 12288, 1024)])
@pytest.mark.parametrize("rms,use_w,use_sc,use_sh", [
    (True, True, True, True),    # RMSNorm -> Mul(weight) -> Modulate
    (False, False, True, True),  # Modulate
    (False, False, True, False), # scale-only modulation
    (True, False, False, False), # RMS norm alone
])
def test_pack_prologue(ops, M, K, G, rms, use_w, use_sc, use_sh):
    rng = workloads.rng_for(M + K + G)
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=30.0)
    w, sc, sh = vectors(K, K)
    kw = dict(rmsnorm=rms, eps=1e-6, weight=w if use_w else None, scale=sc if use_sc else None,
              shift=sh if use_sh else None)
    Q, s = ops.convrot_pack_prologue(dev(X), G, **{k: (dev(v) if isinstance(v, np.ndarray) else v)
                                                   for k, v in kw.items()})
    Qo, so = oracle.pack(oracle.prologue(X, **kw), G)
    assert_scales(host(s), so)
    assert_codes(host(Q), Qo)


def test_linear_prologue(ops):
    w = workloads.get("dit_qkv")
    case = workloads.make_case(w, M=700)
    g, sc, sh = vectors(1, w.K)
    preps = [ops.convrot_prepare_weight(dev(W), w.G) for W in case.Ws[:2]]
    Ys = ops.convrot_linear_prologue(dev(case.X), w.G, [p[2] for p in preps], [p[1] for p in preps],
                                     [dev(b) for b in case.bs[:2]], rmsnorm=True, eps=1e-6,
                                     weight=dev(g), scale=dev(sc), shift=dev(sh))
    Xp = oracle.prologue(case.X, rmsnorm=True, eps=1e-6, weight=g, scale=sc, shift=sh)
    for y, p, b in zip(Ys, preps, case.bs[:2]):
        assert_y(host(y), oracle.linear(Xp, host(p[0]), host(p[1]), b, w.G))


@pytest.mark.parametrize("M,K", [(4608, 3072), (300, 12288)])
def test_modulated_pack_is_repeatable(ops, M, K):
    """The RMS norm's row sum of squares is added in a fixed order of its lane
    segments, so repeated packs of one input are bit-identical (on the
    TMA-fed kernel, and on the general kernel that long rows take)."""
    rng = workloads.rng_for(M + K + 5)
    X = dev(workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=40.0))
    w, sc, sh = (dev(v) for v in vectors(M + K, K))
    runs = [ops.convrot_pack_prologue(X, 256, rmsnorm=True, weight=w, scale=sc, shift=sh) for _ in range(3)]
    Q0, s0 = host(runs[0][0]), host(runs[0][1])
    for Q, s in runs[1:]:
        np.testing.assert_array_equal(host(Q), Q0)
        np.testing.assert_array_equal(host(s), s0)
    assert ops.convrot_device_status() == ops.OK
