"""convrot_linear_noalloc: the fused convrot linear for callers that cannot
allocate device memory (a plugin handed only its input and output buffers by
a framework that owns every allocation, or a latency-bound loop where
cudaMalloc is not allowed). Instead of a caller workspace it uses one fixed
device array inside the library.

The GPU test calls the entry point through the C ABI twice in a row, with
different shapes, dtypes and group sizes (so the second call runs on an array
still holding the first call's data), and checks each output against
convrot_linear, the workspace-taking entry point, on the same inputs and
weights. This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from parity import assert_y


def _case(seed, M, K, Ns, x_dtype):
    rng = workloads.rng_for(seed)
    X = workloads.activations(rng, M, K, outlier_frac=0.01, outlier_mult=40.0, dtype=x_dtype)
    Ws = [workloads.weights(rng, n, K) for n in Ns]
    bs = [workloads.biases(rng, n) for n in Ns]
    return X, Ws, bs


@pytest.mark.gpu
def test_noalloc_matches_convrot_linear_on_two_calls(ops):
    calls = [
        # seed, M, K, G, output features, activation dtype
        (11, 2304, 3072, 256, (3072, 1024, 640), "f32"),  # 14.2 MB of the 32 MiB array
        (12, 1000, 1280, 64, (1280,), "f16"),             # ragged M, fewer rows
    ]
    for seed, M, K, G, Ns, xd in calls:
        X, Ws, bs = _case(seed, M, K, Ns, xd)
        Xd = dev(X)
        preps = [ops.convrot_prepare_weight(dev(W), G) for W in Ws]
        q16s = [p[2] for p in preps]
        scales = [p[1] for p in preps]
        biases = [dev(b) for b in bs]
        Y_ref = ops.convrot_linear(Xd, G, q16s, scales, biases)
        Y_new = [torch.full_like(y, float("nan")) for y in Y_ref]
        ops.convrot_linear_noalloc(Xd, G, q16s, scales, biases, Ys=Y_new)
        assert ops.convrot_device_status() == ops.OK
        for j, (a, b) in enumerate(zip(Y_new, Y_ref)):
            a, b = host(a), host(b)
            assert np.isfinite(a).all()
            assert_y(a, b, f"noalloc call M={M} Y{j}")
            # same kernels on the same codes: the results are identical
            assert np.array_equal(a, b)


def test_noalloc_rejects_calls_larger_than_its_array():
    """A call whose packed activation exceeds the fixed array fails before any
    device work (fake, never dereferenced addresses)."""
    from int8_hadamard_rotated_gb300 import build, ops
    build.build()
    L = ops.lib()
    A0, A1, A2 = (0x7f0000000000 + i * 0x10000000 for i in range(3))
    W = ops.convrot_weight
    ws = (W * 1)(W(A1, None, None, 64, A2))
    # 4096 x 4096 binary16 codes alone are exactly the 32 MiB; the scales do not fit
    assert L.convrot_linear_noalloc(A0, ops.F32, 4096, 4096, 256, ws, 1, None) == ops.ERR_SCRATCH
    assert b"scratch" in L.convrot_strerror(ops.ERR_SCRATCH)
