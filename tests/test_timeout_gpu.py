"""The GEMM's failure path on the GPU, made to happen without faulting,
trapping or hanging anything: every device-side wait is bounded, and a test
entry point (convrot_test_handover_timeout) shortens the bound to 100 us and
makes the CTA pairs that finish split tiles wait for a hand-over value that
no pair publishes. Those waits must give up, the kernel must record
CONVROT_ERR_TIMEOUT in the device's error word and exit, convrot_device_status
must report it once and clear it, and the next normal call on the same stream
and hand-over words must be correct."""
import numpy as np
import pytest
import torch

from int8_hadamard_rotated_gb300 import workloads
from gpu_common import dev, host
from split_tail_ref import plan_split

pytestmark = pytest.mark.gpu


def test_handover_wait_runs_out_then_the_next_call_is_correct(ops):
    w = workloads.get("dit_qkv")
    case = workloads.make_case(w)
    M, K, G = w.M, w.K, w.G
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    tiles = -(-M // 256) * sum(-(-n // 256) for n in w.Ns)
    assert plan_split(tiles, pairs) > 0, "the shape must split its last wave on this GPU"
    preps = [ops.convrot_prepare_weight(dev(W), G) for W in case.Ws]
    q16s, scales, biases = [p[2] for p in preps], [p[1] for p in preps], [dev(b) for b in case.bs]
    Q16, s16 = ops.convrot_pack_activations_f16(dev(case.X), G)
    ref = [host(y) for y in ops.convrot_linear_packed(Q16, s16, q16s, scales, biases, split_tail=False)]
    assert ops.convrot_device_status() == ops.OK

    ws = torch.zeros((ops.GEMM_SYNC_BYTES,), dtype=torch.uint8, device="cuda")
    Ys = [torch.full((M, n), float("nan"), dtype=torch.float32, device="cuda") for n in w.Ns]
    ops.convrot_test_handover_timeout(Q16, s16, q16s, scales, biases, 100_000, ws, Ys=Ys)
    torch.cuda.synchronize()
    assert ops.convrot_device_status() == ops.ERR_TIMEOUT   # the waits gave up and were reported
    assert ops.convrot_device_status() == ops.OK            # ... once: the word is cleared
    # the split tiles were left unfinished
    assert any(np.isnan(host(y)).any() or not np.array_equal(host(y), r) for y, r in zip(Ys, ref))

    # the device, the stream and the hand-over words stay usable
    Ys = ops.convrot_linear_packed(Q16, s16, q16s, scales, biases, Ys=Ys, workspace=ws)
    for y, r in zip(Ys, ref):
        np.testing.assert_array_equal(host(y), r)
    assert ops.convrot_device_status() == ops.OK
