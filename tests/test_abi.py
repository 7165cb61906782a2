"""CPU checks of the C ABI: the library builds, loads and exports every entry
point that include/convrot.h declares, and the host-side argument checks
reject bad calls with the documented status codes before touching a GPU.
(Fake device addresses are fine here: argument checks never dereference.)
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "convrot.h")


@pytest.fixture(scope="session")
def L():
    from int8_hadamard_rotated_gb300 import build, ops
    build.build()
    return ops.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:int|size_t|const char\s*\*)\s+(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for n in ("convrot_prepare_weight", "convrot_pack_activations", "int8_linear",
              "convrot_linear", "int8_gemm_s32", "convrot_linear_workspace_size",
              "int8_linear_workspace_size", "convrot_device_status", "convrot_strerror",
              "convrot_version", "convrot_last_cuda_error"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    from int8_hadamard_rotated_gb300 import ops
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in ops.SIGNATURES, name


def test_strerror_and_version(L):
    assert L.convrot_version() >= 100
    for code in range(11):
        assert L.convrot_strerror(code)
    assert b"unknown" in L.convrot_strerror(99)


def test_workspace_sizes(L):
    from int8_hadamard_rotated_gb300 import ops
    sync = ops.GEMM_SYNC_BYTES  # the GEMM's hand-over words, one 8-byte word per CTA of up to 256 pairs
    assert sync == 2 * 256 * 8
    assert L.convrot_linear_workspace_size(4608, 3072) == 4608 * 3072 * 2 + ((4608 * 4 + 255) // 256) * 256 + sync
    assert L.int8_linear_workspace_size(16, 128, 256, 1) == 16 * 256 * 2 + sync
    assert L.int8_linear_workspace_size(16, 128, 256, 0) == 16 * 256 * 2 + 128 * 256 * 2 + sync
    m = 4608 * 3072 * 2 + 4608 * 4 + 4608 * 12288 * 4 + 4608 * 12288 * 2 + 4608 * 4
    assert L.convrot_mlp_workspace_size(4608, 3072, 12288) == m + sync


def test_packed_linear_workspace_checks(L):
    """convrot_linear_packed: the hand-over workspace is optional, but when
    given it must be aligned, large enough and apart from every other array
    (checked before any device call)."""
    from int8_hadamard_rotated_gb300 import ops
    W = ops.convrot_weight
    wts = (W * 1)(W(A1, A2, A3, 64, A4, None))
    f = L.convrot_linear_packed
    sync = ops.GEMM_SYNC_BYTES
    assert f(A0, A5, 16, 256, wts, 1, A6 + 8, sync, None) == ops.ERR_ALIGN
    assert f(A0, A5, 16, 256, wts, 1, A6, sync - 1, None) == ops.ERR_WORKSPACE
    assert f(A0, A5, 16, 256, wts, 1, A4, sync, None) == ops.ERR_ALIAS       # on Y
    assert f(A0, A5, 16, 256, wts, 1, A0 + 256, sync, None) == ops.ERR_ALIAS  # inside Q_x16
    assert f(A0, A5, 0, 256, wts, 1, None, 0, None) == ops.OK


# fake, 256-aligned, non-overlapping device addresses
A0, A1, A2, A3, A4, A5, A6 = (0x7f0000000000 + i * 0x10000000 for i in range(7))


def test_pack_argument_checks(L):
    from int8_hadamard_rotated_gb300 import ops
    f = L.convrot_pack_activations
    assert f(A0, ops.F32, 0, 256, 256, A1, A2, None) == ops.OK              # M = 0: no-op
    assert f(None, ops.F32, 4, 256, 256, A1, A2, None) == ops.ERR_ARG
    assert f(A0, 7, 4, 256, 256, A1, A2, None) == ops.ERR_ARG               # dtype
    assert f(A0, ops.F32, -1, 256, 256, A1, A2, None) == ops.ERR_ARG
    for G in (2, 8, 32, 128, 512, 4096, 0):
        assert f(A0, ops.F32, 4, 4096, G, A1, A2, None) == ops.ERR_GROUP
    assert f(A0, ops.F32, 4, 1280, 1024, A1, A2, None) == ops.ERR_GROUP     # 1024 does not divide 1280
    assert f(A0, ops.F32, 4, 40, 4, A1, A2, None) == ops.ERR_ALIGN          # K % 16
    assert f(A0 + 4, ops.F32, 4, 256, 256, A1, A2, None) == ops.ERR_ALIGN
    assert f(A0, ops.F32, 4, 65536, 256, A1, A2, None) == ops.ERR_UNSUPPORTED
    assert f(A0, ops.F32, 4, 256, 256, A0 + 256, A2, None) == ops.ERR_ALIAS  # Q_x inside X
    assert f(A0, ops.F32, 4, 256, 256, A1, A1 + 512, None) == ops.ERR_ALIAS  # s_x inside Q_x


def test_gemm_argument_checks(L):
    from int8_hadamard_rotated_gb300 import ops
    f = L.int8_linear
    big = 1 << 40
    assert f(A0, A1, 0, 256, A2, None, None, None, 128, A3, A4, big, None) == ops.OK
    assert f(None, A1, 4, 256, A2, None, None, None, 128, A3, A4, big, None) == ops.ERR_ARG
    assert f(A0, A1, 4, 256, None, None, None, None, 128, A3, A4, big, None) == ops.ERR_ARG
    assert f(A0, A1, 4, 250, A2, None, None, None, 128, A3, A4, big, None) == ops.ERR_ALIGN
    assert f(A0, A1, 4, 133152, A2, None, None, None, 128, A3, A4, big, None) == ops.ERR_OVERFLOW
    assert f(A0, A1, 4, 256, A2, None, None, None, 128, A3, None, 0, None) == ops.ERR_WORKSPACE
    assert f(A0, A1, 4, 256, A2, None, None, None, 128, A3, A4, 100, None) == ops.ERR_WORKSPACE
    assert f(A0, A1, 4, 256, A2, None, None, None, 128, A0, A4, big, None) == ops.ERR_ALIAS
    assert f(A0, A1, 4, 256, A2, None, None, None, 128, A3, A3 + 256, big, None) == ops.ERR_ALIAS


def test_linear_argument_checks(L):
    from int8_hadamard_rotated_gb300 import ops
    f = L.convrot_linear
    W = ops.convrot_weight
    ws = (W * 2)(W(A1, A2, A3, 64, A4), W(A1 + 0x100000, None, None, 64, A5))
    big = 1 << 40
    assert f(A0, ops.F32, 16, 256, 256, ws, 0, A3 + 0x1000000, big, None) == ops.ERR_ARG
    assert f(A0, ops.F32, 16, 256, 256, ws, 9, A3 + 0x1000000, big, None) == ops.ERR_ARG
    assert f(A0, ops.F32, 16, 256, 128, ws, 2, A3 + 0x1000000, big, None) == ops.ERR_GROUP
    assert f(A0, ops.F32, 16, 256, 256, ws, 2, None, 0, None) == ops.ERR_WORKSPACE
    same = (W * 2)(W(A1, None, None, 64, A4), W(A1, None, None, 64, A4))
    assert f(A0, ops.F32, 16, 256, 256, same, 2, A3 + 0x1000000, big, None) == ops.ERR_ALIAS


def test_valid_call_without_gpu_reports_device(L):
    """A well-formed call on a machine without an sm_103 GPU fails cleanly."""
    import torch
    from int8_hadamard_rotated_gb300 import ops
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert L.convrot_pack_activations(A0, ops.F32, 4, 256, 256, A1, A2, None) == ops.ERR_DEVICE


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from int8_hadamard_rotated_gb300 import ops
    monkeypatch.setattr(ops, "_LIB", None)
    monkeypatch.setattr(ops, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        ops.lib()


def test_host_pipeline_checks(L):
    from int8_hadamard_rotated_gb300 import ops
    ws = L.convrot_linear_host_workspace_size
    # two sets of (input rows, binary16 codes, scales, outputs), each rounded to 256 bytes
    r = 768
    one = (r * 3072 * 4) + (r * 3072 * 2) + ((r * 4 + 255) // 256 * 256) + (r * 9216 * 4)
    assert ws(4608, 3072, ops.F32, 9216, 0) == 2 * one + ops.GEMM_SYNC_BYTES
    assert ws(100, 3072, ops.F32, 9216, 0) == ws(100, 3072, ops.F32, 9216, 100)  # chunk clipped to M
    assert ws(0, 3072, ops.F32, 9216, 0) == 0 and ws(10, 3072, 5, 9216, 0) == 0
    W = ops.convrot_weight
    wts = (W * 1)(W(A1, None, None, 64, A2))
    g = L.convrot_linear_host
    assert g(A0, ops.F32, 16, 256, 128, wts, 1, 0, A3, 1 << 40, None, None, None) == ops.ERR_GROUP
    assert g(A0, ops.F32, 16, 256, 256, wts, 1, 0, None, 0, None, None, None) == ops.ERR_WORKSPACE
    assert g(A0, ops.F32, 16, 256, 256, wts, 1, -1, A3, 1 << 40, None, None, None) == ops.ERR_ARG
    assert g(A0, ops.F32, 0, 256, 256, wts, 1, 0, None, 0, None, None, None) == ops.OK


def test_scaled_linear_rejects_bad_scales(L):
    import ctypes
    from int8_hadamard_rotated_gb300 import ops
    W = ops.convrot_weight
    ws = (W * 1)(W(A1, A2, A3, 64, A4, None))
    f = L.convrot_linear_scaled
    for a in (0.0, -1.0, float("inf"), float("nan")):
        assert f(A0, ops.F32, 16, 256, 256, a, ws, 1, A5, 1 << 40, None) == ops.ERR_ARG


def test_w4_descriptor_checks(L):
    """A weight descriptor holds exactly one kind of weight (binary16 codes or
    packed 4-bit bytes); a packed 4-bit linear needs K % 64 == 0, N % 4 == 0
    and K <= CONVROT_W4_MAX_K. All checked before any device call."""
    from int8_hadamard_rotated_gb300 import ops
    W = ops.convrot_weight
    f = L.convrot_linear
    big = 1 << 40
    both = (W * 1)(W(A1, None, None, 64, A4, None, A2))
    neither = (W * 1)(W(None, None, None, 64, A4, None, None))
    q4 = (W * 1)(W(None, A2, A3, 64, A4, None, A1))
    assert f(A0, ops.F32, 16, 256, 256, both, 1, A5, big, None) == ops.ERR_ARG
    assert f(A0, ops.F32, 16, 256, 256, neither, 1, A5, big, None) == ops.ERR_ARG
    assert f(A0, ops.F32, 16, 96, 16, q4, 1, A5, big, None) == ops.ERR_ALIGN          # K % 64
    odd_n = (W * 1)(W(None, None, None, 66, A4, None, A1))
    assert f(A0, ops.F32, 16, 256, 256, odd_n, 1, A5, big, None) == ops.ERR_ALIGN     # N % 4
    assert f(A0, ops.F32, 16, 16384 + 1024, 1024, q4, 1, A5, big, None) == ops.ERR_UNSUPPORTED
    assert f(A0, ops.F32, 16, 256, 256, (W * 1)(W(None, None, None, 64, A4, None, A1 + 8)), 1, A5, big,
             None) == ops.ERR_ALIGN                                                     # unaligned bytes
    # the packed bytes span N * K / 2: an output placed right after them is fine,
    # one byte earlier overlaps
    after = (W * 1)(W(None, None, None, 64, A1 + 64 * 128, None, A1))
    assert f(A0, ops.F32, 16, 256, 256, after, 1, A5, big, None) == ops.ERR_DEVICE or \
        f(A0, ops.F32, 16, 256, 256, after, 1, A5, big, None) == ops.OK
    inside = (W * 1)(W(None, None, None, 64, A1 + 64 * 128 - 16, None, A1))
    assert f(A0, ops.F32, 16, 256, 256, inside, 1, A5, big, None) == ops.ERR_ALIAS
    g = L.int8_gemm_s32_w4
    assert L.int8_gemm_s32_w4_workspace_size(16, 256) == 16 * 256 * 2 + ops.GEMM_SYNC_BYTES
    assert g(A0, 16, 96, A1, 64, A2, A3, big, None) == ops.ERR_ALIGN
    assert g(A0, 16, 16384 + 64, A1, 64, A2, A3, big, None) == ops.ERR_UNSUPPORTED
    assert g(A0, 16, 256, A1, 64, A2, A3, 100, None) == ops.ERR_WORKSPACE
    assert g(A0, 16, 256, A1, 64, A1 + 64, A3, big, None) == ops.ERR_ALIAS
    assert g(A0, 0, 256, A1, 64, A2, A3, big, None) == ops.OK


def test_timeout_test_entry_checks(L):
    """The timeout-path test entry point checks its arguments like the GEMM."""
    from int8_hadamard_rotated_gb300 import ops
    W = ops.convrot_weight
    wts = (W * 1)(W(A1, A2, A3, 64, A4, None))
    f = L.convrot_test_handover_timeout
    sync = ops.GEMM_SYNC_BYTES
    assert f(A0, A5, 16, 256, wts, 1, A6, sync, 0, None) == ops.ERR_ARG          # no wait limit
    assert f(A0, A5, 16, 256, wts, 1, None, 0, 1000, None) == ops.ERR_ARG        # hand-over words required
    assert f(A0, A5, 16, 256, wts, 1, A6, sync - 8, 1000, None) == ops.ERR_WORKSPACE
    w4 = (W * 1)(W(None, A2, A3, 64, A4, None, A1))
    assert f(A0, A5, 16, 256, w4, 1, A6, sync, 1000, None) == ops.ERR_ARG        # binary16 weights only


def test_unscale_sweep_entry_checks(L):
    """The unscaling sweep (a test of the GEMM epilogue's division step)
    checks its arguments before touching the device."""
    from int8_hadamard_rotated_gb300 import ops
    f = L.convrot_test_unscale_sweep
    assert f(None, 4, 0, A5, A6, None) == ops.ERR_ARG           # no divisors
    assert f(A0, 0, 0, A5, A6, None) == ops.ERR_ARG             # empty
    assert f(A0, 65536, 0, A5, A6, None) == ops.ERR_ARG         # more than a grid's y extent
    assert f(A0, 4, -99, A5, A6, None) == ops.ERR_ARG           # y below the step's range
    assert f(A0, 4, 98, A5, A6, None) == ops.ERR_ARG            # y above it
    assert f(A0, 4, 0, None, A6, None) == ops.ERR_ARG           # no counter
    assert f(A0 + 4, 4, 0, A5, A6, None) == ops.ERR_ALIGN       # divisors not 16-byte aligned


def test_mlp_host_argument_checks(L):
    """convrot_mlp_host checks its arguments before touching the device."""
    from int8_hadamard_rotated_gb300 import ops
    W = ops.convrot_weight
    up = (W * 1)(W(A1, A2, A3, 256, None, None))
    down = (W * 1)(W(A4, A2, A3, 64, None, None))
    f = L.convrot_mlp_host
    need = L.convrot_mlp_host_workspace_size(16, 64, ops.F32, 256, 64, 0)
    assert need > 0
    assert L.convrot_mlp_host_workspace_size(16, 64, 7, 256, 64, 0) == 0          # bad dtype
    assert f(None, ops.F32, 16, 64, 64, up, ops.ACT_GELU, 64, down, A5, 0, A6, need, None, None, None) == ops.ERR_ARG
    assert f(A0, ops.F32, 16, 64, 64, up, ops.ACT_GELU, 64, down, None, 0, A6, need, None, None, None) == ops.ERR_ARG
    assert f(A0, ops.F32, 16, 64, 64, up, 9, 64, down, A5, 0, A6, need, None, None, None) == ops.ERR_ARG
    assert f(A0, 7, 16, 64, 64, up, ops.ACT_GELU, 64, down, A5, 0, A6, need, None, None, None) == ops.ERR_ARG
    assert f(A0, ops.F32, 16, 64, 64, up, ops.ACT_GELU, 64, down, A5, -1, A6, need, None, None, None) == ops.ERR_ARG
    assert f(A0, ops.F32, 16, 64, 64, up, ops.ACT_GELU, 64, down, A5, 0, None, 0, None, None, None) == ops.ERR_WORKSPACE
    assert f(A0, ops.F32, 16, 64, 64, up, ops.ACT_GELU, 64, down, A5, 0, A6, need - 256, None, None,
             None) == ops.ERR_WORKSPACE
    assert f(A0, ops.F32, 16, 64, 64, up, ops.ACT_GELU, 64, down, A5, 0, A6 + 8, need, None, None,
             None) == ops.ERR_ALIGN
