"""Thin Python binding of libconvrot.so (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks dtypes/devices, allocates outputs and
workspace with PyTorch when the caller does not pass them, and hands raw
device pointers plus the current CUDA stream to the library. All compute runs
in the library's sm_103a kernels; if the library is missing this module
raises, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import struct
from typing import List, Optional, Sequence, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libconvrot.so")

# status codes (include/convrot.h)
OK = 0
ERR_ARG = 1
ERR_GROUP = 2
ERR_ALIGN = 3
ERR_OVERFLOW = 4
ERR_ALIAS = 5
ERR_WORKSPACE = 6
ERR_UNSUPPORTED = 7
ERR_TIMEOUT = 8
ERR_CUDA = 9
ERR_DEVICE = 10
ERR_SCRATCH = 11

ACT_NONE = 0
ACT_GELU = 1
ACT_SWIGLU = 2

F32 = 0
F16 = 1
MAX_LINEARS = 8
PACK_MAX_K = 32768
MAX_K = 133144
W4_MAX_K = 16384
CHUNK_ROWS = 128
NOALLOC_SCRATCH_BYTES = 32 << 20
GEMM_SYNC_BYTES = 4096


class ConvrotError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _lib_or_none()
        msg = lib.convrot_strerror(status).decode() if lib else str(status)
        if status == ERR_CUDA and lib:
            msg += f" (cudaError {lib.convrot_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [status {status}]")
        self.status = status


class convrot_prologue(ctypes.Structure):
    _fields_ = [("rmsnorm", ctypes.c_int), ("eps", ctypes.c_float), ("weight", ctypes.c_void_p),
                ("scale", ctypes.c_void_p), ("shift", ctypes.c_void_p)]


class convrot_weight(ctypes.Structure):
    _fields_ = [("q16", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("N", ctypes.c_int64),
                ("Y", ctypes.c_void_p), ("kchunk", ctypes.c_void_p),
                ("q4", ctypes.c_void_p)]


_LIB = None

_VP, _I64, _I, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "convrot_version": (_I, []),
    "convrot_strerror": (ctypes.c_char_p, [_I]),
    "convrot_last_cuda_error": (_I, []),
    "convrot_prepare_weight": (_I, [_VP, _I64, _I64, _I, _VP, _VP, _VP, _VP]),
    "convrot_pack_activations": (_I, [_VP, _I, _I64, _I64, _I, _VP, _VP, _VP]),
    "int8_linear_workspace_size": (_SZ, [_I64, _I64, _I64, _I]),
    "int8_linear": (_I, [_VP, _VP, _I64, _I64, _VP, _VP, _VP, _VP, _I64, _VP, _VP, _SZ, _VP]),
    "convrot_linear_workspace_size": (_SZ, [_I64, _I64]),
    "convrot_linear": (_I, [_VP, _I, _I64, _I64, _I, ctypes.POINTER(convrot_weight), _I, _VP, _SZ, _VP]),
    "convrot_pack_prologue": (_I, [_VP, _I64, _I64, _I, ctypes.POINTER(convrot_prologue), _VP, _VP, _VP]),
    "convrot_linear_prologue": (_I, [_VP, _I64, _I64, _I, ctypes.POINTER(convrot_prologue),
                                     ctypes.POINTER(convrot_weight), _I, _VP, _SZ, _VP]),
    "convrot_linear_scaled": (_I, [_VP, _I, _I64, _I64, _I, ctypes.c_float, ctypes.POINTER(convrot_weight), _I,
                                   _VP, _SZ, _VP]),
    "int8_gemm_s32": (_I, [_VP, _I64, _I64, _VP, _VP, _VP, _I64, _VP, _VP, _SZ, _VP]),
    "int8_gemm_s32_w4_workspace_size": (_SZ, [_I64, _I64]),
    "int8_gemm_s32_w4": (_I, [_VP, _I64, _I64, _VP, _I64, _VP, _VP, _SZ, _VP]),
    "convrot_weight_chunks": (_I, [_VP, _I64, _I64, _VP, _VP]),
    "convrot_w4_expand": (_I, [_VP, _I64, _I64, _VP, _VP, _VP]),
    "convrot_pack_activations_f16": (_I, [_VP, _I, _I64, _I64, _I, _VP, _VP, _VP]),
    "convrot_linear_packed": (_I, [_VP, _VP, _I64, _I64, ctypes.POINTER(convrot_weight), _I, _VP, _SZ, _VP]),
    "convrot_pack_gelu_f16": (_I, [_VP, _I64, _I64, _I, _VP, _VP, _VP]),
    "convrot_linear_packed_act": (_I, [_VP, _VP, _I64, _I64, ctypes.POINTER(convrot_weight), _I, _I, _VP, _SZ,
                                       _VP]),
    "convrot_linear_host_workspace_size": (_SZ, [_I64, _I64, _I, _I64, _I64]),
    "convrot_linear_host": (_I, [_VP, _I, _I64, _I64, _I, ctypes.POINTER(convrot_weight), _I, _I64, _VP, _SZ,
                                 _VP, _VP, _VP]),
    "convrot_mlp_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "convrot_mlp_host_workspace_size": (_SZ, [_I64, _I64, _I, _I64, _I64, _I64]),
    "convrot_mlp_host": (_I, [_VP, _I, _I64, _I64, _I, ctypes.POINTER(convrot_weight), _I, _I,
                              ctypes.POINTER(convrot_weight), _VP, _I64, _VP, _SZ, _VP, _VP, _VP]),
    "convrot_mlp": (_I, [_VP, _I, _I64, _I64, _I, ctypes.POINTER(convrot_weight), _I, _I,
                         ctypes.POINTER(convrot_weight), _VP, _SZ, _VP]),
    "convrot_linear_noalloc": (_I, [_VP, _I, _I64, _I64, _I, ctypes.POINTER(convrot_weight), _I, _VP]),
    "convrot_linear_swiglu": (_I, [_VP, _I, _I64, _I64, _I, ctypes.POINTER(convrot_weight), _VP, _SZ, _VP]),
    "convrot_device_status": (_I, [_VP]),
    "convrot_test_handover_timeout": (_I, [_VP, _VP, _I64, _I64, ctypes.POINTER(convrot_weight), _I, _VP, _SZ,
                                           ctypes.c_uint64, _VP]),
    "convrot_test_unscale_sweep": (_I, [_VP, _I, _I, _VP, _VP, _VP]),
}


def _lib_or_none():
    return _LIB


def lib() -> ctypes.CDLL:
    """Load libconvrot.so (once). Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m int8_hadamard_rotated_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _check(status: int, where: str):
    if status != OK:
        raise ConvrotError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _need(t: torch.Tensor, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _xdtype(X: torch.Tensor) -> int:
    if X.dtype == torch.float32:
        return F32
    if X.dtype == torch.float16:
        return F16
    raise ValueError("X must be float32 or float16")


# ---------------------------------------------------------------------------

def convrot_pack_activations(X: torch.Tensor, G: int, Q_x: Optional[torch.Tensor] = None,
                             s_x: Optional[torch.Tensor] = None, stream=None
                             ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Rotate and quantize the rows of X [M,K] -> (Q_x int8 [M,K], s_x f32 [M])."""
    xd = _xdtype(X)
    _need(X, X.dtype, "X")
    M, K = X.shape
    if Q_x is None:
        Q_x = torch.empty((M, K), dtype=torch.int8, device=X.device)
    if s_x is None:
        s_x = torch.empty((M,), dtype=torch.float32, device=X.device)
    _need(Q_x, torch.int8, "Q_x")
    _need(s_x, torch.float32, "s_x")
    _check(lib().convrot_pack_activations(_ptr(X), xd, M, K, G, _ptr(Q_x), _ptr(s_x), _stream(stream)),
           "convrot_pack_activations")
    return Q_x, s_x


def convrot_prepare_weight(W: torch.Tensor, G: int, with_f16: bool = True, stream=None):
    """Offline weight path: W [N,K] f32 -> (Q_w int8, s_w f32, Q_w16 fp16 codes or None)."""
    _need(W, torch.float32, "W")
    N, K = W.shape
    Q_w = torch.empty((N, K), dtype=torch.int8, device=W.device)
    s_w = torch.empty((N,), dtype=torch.float32, device=W.device)
    Q_w16 = torch.empty((N, K), dtype=torch.float16, device=W.device) if with_f16 else None
    _check(lib().convrot_prepare_weight(_ptr(W), N, K, G, _ptr(Q_w), _ptr(s_w), _ptr(Q_w16), _stream(stream)),
           "convrot_prepare_weight")
    return Q_w, s_w, Q_w16


def int8_linear_workspace_size(M: int, N: int, K: int, have_q_w16: bool) -> int:
    return int(lib().int8_linear_workspace_size(M, N, K, 1 if have_q_w16 else 0))


def convrot_linear_workspace_size(M: int, K: int) -> int:
    return int(lib().convrot_linear_workspace_size(M, K))


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is None:
        return torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError("workspace too small")
    return workspace


def int8_linear(Q_x, s_x, Q_w=None, Q_w16=None, s_w=None, bias=None, Y=None,
                workspace=None, stream=None) -> torch.Tensor:
    """Y = float(Q_x Q_w^T) * s_x * s_w + bias, fp32 [M,N]."""
    _need(Q_x, torch.int8, "Q_x")
    _need(s_x, torch.float32, "s_x")
    ref = Q_w16 if Q_w16 is not None else Q_w
    if ref is None:
        raise ValueError("Q_w or Q_w16 is required")
    M, K = Q_x.shape
    N = ref.shape[0]
    if Q_w is not None:
        _need(Q_w, torch.int8, "Q_w")
    if Q_w16 is not None:
        _need(Q_w16, torch.float16, "Q_w16")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=Q_x.device)
    ws = _workspace(int8_linear_workspace_size(M, N, K, Q_w16 is not None), Q_x.device, workspace)
    _check(lib().int8_linear(_ptr(Q_x), _ptr(s_x), M, K, _ptr(Q_w), _ptr(Q_w16), _ptr(s_w), _ptr(bias),
                             N, _ptr(Y), _ptr(ws), ws.numel(), _stream(stream)), "int8_linear")
    return Y


def convrot_weight_chunks(Q_w: torch.Tensor, kchunk: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Exact-chunk plan of int8 weight codes [N,K]: int32 [ceil(N/128)]."""
    _need(Q_w, torch.int8, "Q_w")
    N, K = Q_w.shape
    if kchunk is None:
        kchunk = torch.empty(((N + CHUNK_ROWS - 1) // CHUNK_ROWS,), dtype=torch.int32, device=Q_w.device)
    _check(lib().convrot_weight_chunks(_ptr(Q_w), N, K, _ptr(kchunk), _stream(stream)), "convrot_weight_chunks")
    return kchunk


def convrot_w4_expand(Q_w4: torch.Tensor, K: int, with_int8: bool = True, stream=None):
    """Packed signed 4-bit weights [N, K/2] (uint8, low nibble first) ->
    (int8 codes or None, binary16 codes) [N, K]."""
    _need(Q_w4, torch.uint8, "Q_w4")
    N = Q_w4.shape[0]
    if Q_w4.shape[1] * 2 != K:
        raise ValueError("Q_w4 must be [N, K/2]")
    q8 = torch.empty((N, K), dtype=torch.int8, device=Q_w4.device) if with_int8 else None
    q16 = torch.empty((N, K), dtype=torch.float16, device=Q_w4.device)
    _check(lib().convrot_w4_expand(_ptr(Q_w4), N, K, _ptr(q8), _ptr(q16), _stream(stream)), "convrot_w4_expand")
    return q8, q16


def int8_gemm_s32(Q_x, Q_w=None, Q_w16=None, A=None, workspace=None, stream=None, kchunk=None) -> torch.Tensor:
    """Raw int32 A = Q_x Q_w^T through the tensor-core GEMM (optionally with
    the weight's exact-chunk plan)."""
    _need(Q_x, torch.int8, "Q_x")
    ref = Q_w16 if Q_w16 is not None else Q_w
    M, K = Q_x.shape
    N = ref.shape[0]
    if A is None:
        A = torch.empty((M, N), dtype=torch.int32, device=Q_x.device)
    ws = _workspace(int8_linear_workspace_size(M, N, K, Q_w16 is not None), Q_x.device, workspace)
    _check(lib().int8_gemm_s32(_ptr(Q_x), M, K, _ptr(Q_w), _ptr(Q_w16), _ptr(kchunk), N, _ptr(A), _ptr(ws),
                               ws.numel(), _stream(stream)), "int8_gemm_s32")
    return A


def int8_gemm_s32_w4(Q_x, Q_w4, A=None, workspace=None, stream=None) -> torch.Tensor:
    """Raw int32 A = Q_x Q_w^T with packed signed 4-bit weights Q_w4 [N, K/2]
    (uint8, low nibble first), through the S8 x S4 GEMM."""
    _need(Q_x, torch.int8, "Q_x")
    _need(Q_w4, torch.uint8, "Q_w4")
    M, K = Q_x.shape
    N = Q_w4.shape[0]
    if Q_w4.shape[1] * 2 != K:
        raise ValueError("Q_w4 must be [N, K/2]")
    if A is None:
        A = torch.empty((M, N), dtype=torch.int32, device=Q_x.device)
    ws = _workspace(int(lib().int8_gemm_s32_w4_workspace_size(M, K)), Q_x.device, workspace)
    _check(lib().int8_gemm_s32_w4(_ptr(Q_x), M, K, _ptr(Q_w4), N, _ptr(A), _ptr(ws), ws.numel(), _stream(stream)),
           "int8_gemm_s32_w4")
    return A


def make_weights(q16s: Sequence[torch.Tensor], scales: Sequence[Optional[torch.Tensor]],
                 biases: Sequence[Optional[torch.Tensor]], Ys: Sequence[torch.Tensor],
                 kchunks: Optional[Sequence[Optional[torch.Tensor]]] = None):
    """The convrot_weight descriptors (kchunks: optional exact-chunk plans).
    Each weight is binary16 codes [N, K] (float16) or packed signed 4-bit
    weights [N, K/2] (uint8, low nibble first), which the S8 x S4 GEMM reads
    as they are."""
    arr = (convrot_weight * len(q16s))()
    if kchunks is None:
        kchunks = [None] * len(q16s)
    for j, (q, s, b, y, kc) in enumerate(zip(q16s, scales, biases, Ys, kchunks)):
        if q.dtype == torch.uint8:
            arr[j] = convrot_weight(None, _ptr(s), _ptr(b), q.shape[0], _ptr(y), None, _ptr(q))
        else:
            arr[j] = convrot_weight(_ptr(q), _ptr(s), _ptr(b), q.shape[0], _ptr(y), _ptr(kc), None)
    return arr


def convrot_linear(X: torch.Tensor, G: int, q16s: Sequence[torch.Tensor],
                   scales: Sequence[Optional[torch.Tensor]], biases: Sequence[Optional[torch.Tensor]],
                   Ys: Optional[List[torch.Tensor]] = None, workspace=None, stream=None,
                   weights=None, kchunks=None) -> List[torch.Tensor]:
    """Pack X once, then every Y_j = float(Q_x Q_wj^T) * s_x * s_wj + b_j."""
    xd = _xdtype(X)
    _need(X, X.dtype, "X")
    M, K = X.shape
    if Ys is None:
        Ys = [torch.empty((M, q.shape[0]), dtype=torch.float32, device=X.device) for q in q16s]
    ws = _workspace(convrot_linear_workspace_size(M, K), X.device, workspace)
    if weights is None:
        weights = make_weights(q16s, scales, biases, Ys, kchunks)
    _check(lib().convrot_linear(_ptr(X), xd, M, K, G, weights, len(q16s), _ptr(ws), ws.numel(),
                                _stream(stream)), "convrot_linear")
    return Ys


def convrot_linear_scaled(X: torch.Tensor, G: int, input_scale: float, q16s: Sequence[torch.Tensor],
                          scales: Sequence[Optional[torch.Tensor]], biases: Sequence[Optional[torch.Tensor]],
                          Ys: Optional[List[torch.Tensor]] = None, workspace=None, stream=None,
                          kchunks=None, weights=None) -> List[torch.Tensor]:
    """convrot_linear with an input scale: X is scaled before the pack and
    every output unscaled before its bias."""
    xd = _xdtype(X)
    _need(X, X.dtype, "X")
    M, K = X.shape
    if Ys is None:
        Ys = [torch.empty((M, q.shape[0]), dtype=torch.float32, device=X.device) for q in q16s]
    ws = _workspace(convrot_linear_workspace_size(M, K), X.device, workspace)
    if weights is None:
        weights = make_weights(q16s, scales, biases, Ys, kchunks)
    _check(lib().convrot_linear_scaled(_ptr(X), xd, M, K, G, float(input_scale), weights, len(q16s), _ptr(ws),
                                       ws.numel(), _stream(stream)), "convrot_linear_scaled")
    return Ys


def _prologue(rmsnorm=False, eps=1e-6, weight=None, scale=None, shift=None):
    for name, t in (("weight", weight), ("scale", scale), ("shift", shift)):
        if t is not None:
            _need(t, torch.float32, name)
    return convrot_prologue(1 if rmsnorm else 0, float(eps), _ptr(weight), _ptr(scale), _ptr(shift))


def convrot_pack_prologue(X: torch.Tensor, G: int, rmsnorm=False, eps=1e-6, weight=None, scale=None, shift=None,
                          Q_x=None, s_x=None, stream=None):
    """Pack of the modulated X (RMS norm, per-channel weight, modulation) into
    int8 codes and row scales, without materializing the modulated X."""
    _need(X, torch.float32, "X")
    M, K = X.shape
    if Q_x is None:
        Q_x = torch.empty((M, K), dtype=torch.int8, device=X.device)
    if s_x is None:
        s_x = torch.empty((M,), dtype=torch.float32, device=X.device)
    pro = _prologue(rmsnorm, eps, weight, scale, shift)
    _check(lib().convrot_pack_prologue(_ptr(X), M, K, G, ctypes.byref(pro), _ptr(Q_x), _ptr(s_x), _stream(stream)),
           "convrot_pack_prologue")
    return Q_x, s_x


def convrot_linear_prologue(X: torch.Tensor, G: int, q16s, scales, biases, rmsnorm=False, eps=1e-6,
                            weight=None, scale=None, shift=None, Ys=None, workspace=None, stream=None,
                            kchunks=None):
    """convrot_linear of the modulated X."""
    _need(X, torch.float32, "X")
    M, K = X.shape
    if Ys is None:
        Ys = [torch.empty((M, q.shape[0]), dtype=torch.float32, device=X.device) for q in q16s]
    ws = _workspace(convrot_linear_workspace_size(M, K), X.device, workspace)
    pro = _prologue(rmsnorm, eps, weight, scale, shift)
    weights = make_weights(q16s, scales, biases, Ys, kchunks)
    _check(lib().convrot_linear_prologue(_ptr(X), M, K, G, ctypes.byref(pro), weights, len(q16s), _ptr(ws),
                                         ws.numel(), _stream(stream)), "convrot_linear_prologue")
    return Ys


def convrot_pack_activations_f16(X: torch.Tensor, G: int, Q_x16: Optional[torch.Tensor] = None,
                                 s_x: Optional[torch.Tensor] = None, stream=None):
    """Pack X into the GEMM operand form: (Q_x16 fp16 codes [M,K], s_x f32 [M])."""
    xd = _xdtype(X)
    _need(X, X.dtype, "X")
    M, K = X.shape
    if Q_x16 is None:
        Q_x16 = torch.empty((M, K), dtype=torch.float16, device=X.device)
    if s_x is None:
        s_x = torch.empty((M,), dtype=torch.float32, device=X.device)
    _need(Q_x16, torch.float16, "Q_x16")
    _need(s_x, torch.float32, "s_x")
    _check(lib().convrot_pack_activations_f16(_ptr(X), xd, M, K, G, _ptr(Q_x16), _ptr(s_x), _stream(stream)),
           "convrot_pack_activations_f16")
    return Q_x16, s_x


def convrot_linear_packed(Q_x16: torch.Tensor, s_x: torch.Tensor, q16s, scales, biases,
                          Ys=None, stream=None, weights=None, kchunks=None, workspace=None,
                          split_tail: bool = True):
    """Grouped GEMM on an already packed activation (fp16 codes + row scales).
    With split_tail (the default) the GEMM gets GEMM_SYNC_BYTES of scratch
    (`workspace`, or a fresh buffer) and may split its last wave of tiles by K;
    split_tail=False passes none (whole tiles only; same results)."""
    _need(Q_x16, torch.float16, "Q_x16")
    _need(s_x, torch.float32, "s_x")
    M, K = Q_x16.shape
    if Ys is None:
        Ys = [torch.empty((M, q.shape[0]), dtype=torch.float32, device=Q_x16.device) for q in q16s]
    if weights is None:
        weights = make_weights(q16s, scales, biases, Ys, kchunks)
    ws_ptr, ws_bytes = None, 0
    if split_tail:
        ws = _workspace(GEMM_SYNC_BYTES, Q_x16.device, workspace)
        ws_ptr, ws_bytes = _ptr(ws), ws.numel() * ws.element_size()
    _check(lib().convrot_linear_packed(_ptr(Q_x16), _ptr(s_x), M, K, weights, len(q16s), ws_ptr, ws_bytes,
                                       _stream(stream)),
           "convrot_linear_packed")
    return Ys


def convrot_linear_packed_act(Q_x16: torch.Tensor, s_x: torch.Tensor, q16s, scales, biases, activation: int,
                              Ys=None, stream=None, kchunks=None, workspace=None):
    """convrot_linear_packed with an activation in the GEMM's epilogue: GELU
    on every output, or split SwiGLU of q16s = [gate, up] (returns [h])."""
    _need(Q_x16, torch.float16, "Q_x16")
    _need(s_x, torch.float32, "s_x")
    M, K = Q_x16.shape
    if Ys is None:
        n_out = 1 if activation == ACT_SWIGLU else len(q16s)
        Ys = [torch.empty((M, q16s[j].shape[0]), dtype=torch.float32, device=Q_x16.device) for j in range(n_out)]
    outs = [Ys[0], Ys[0]] if activation == ACT_SWIGLU else Ys
    weights = make_weights(q16s, scales, biases, outs, kchunks)
    ws = _workspace(GEMM_SYNC_BYTES, Q_x16.device, workspace)
    _check(lib().convrot_linear_packed_act(_ptr(Q_x16), _ptr(s_x), M, K, weights, len(q16s), activation, _ptr(ws),
                                           ws.numel() * ws.element_size(), _stream(stream)),
           "convrot_linear_packed_act")
    return Ys


def convrot_pack_gelu_f16(X: torch.Tensor, G: int, Q_x16: Optional[torch.Tensor] = None,
                          s_x: Optional[torch.Tensor] = None, stream=None):
    """The MLP's repack: GELU applied to fp32 X as it is loaded, then the pack
    into binary16 codes and row scales."""
    _need(X, torch.float32, "X")
    M, K = X.shape
    if Q_x16 is None:
        Q_x16 = torch.empty((M, K), dtype=torch.float16, device=X.device)
    if s_x is None:
        s_x = torch.empty((M,), dtype=torch.float32, device=X.device)
    _check(lib().convrot_pack_gelu_f16(_ptr(X), M, K, G, _ptr(Q_x16), _ptr(s_x), _stream(stream)),
           "convrot_pack_gelu_f16")
    return Q_x16, s_x


def convrot_linear_host_workspace_size(M: int, K: int, x_dtype: int, n_total: int, chunk_rows: int = 0) -> int:
    return int(lib().convrot_linear_host_workspace_size(M, K, x_dtype, n_total, chunk_rows))


def convrot_linear_host(X: torch.Tensor, G: int, q16s: Sequence[torch.Tensor],
                        scales: Sequence[Optional[torch.Tensor]], biases: Sequence[Optional[torch.Tensor]],
                        Ys: Optional[List[torch.Tensor]] = None, chunk_rows: int = 0, workspace=None,
                        stream=None, copy_in_stream=None, copy_out_stream=None, weights=None,
                        kchunks=None) -> List[torch.Tensor]:
    """convrot_linear on host arrays: X [M,K] and the outputs live in (pinned)
    host memory, the weights on the device; transfers of row chunks overlap
    compute on the given copy streams."""
    xd = _xdtype(X)
    if X.is_cuda or not X.is_contiguous():
        raise ValueError("X must be a contiguous host tensor")
    M, K = X.shape
    dev = q16s[0].device
    if Ys is None:
        Ys = [torch.empty((M, q.shape[0]), dtype=torch.float32, pin_memory=True) for q in q16s]
    for y in Ys:
        if y.is_cuda or y.dtype != torch.float32 or not y.is_contiguous():
            raise ValueError("every Y must be a contiguous float32 host tensor")
    n_total = sum(q.shape[0] for q in q16s)
    ws = _workspace(convrot_linear_host_workspace_size(M, K, xd, n_total, chunk_rows), dev, workspace)
    if weights is None:
        weights = make_weights(q16s, scales, biases, Ys, kchunks)
    _check(lib().convrot_linear_host(X.data_ptr(), xd, M, K, G, weights, len(q16s), chunk_rows, _ptr(ws),
                                     ws.numel(), _stream(stream), _stream(copy_in_stream) if copy_in_stream else None,
                                     _stream(copy_out_stream) if copy_out_stream else None),
           "convrot_linear_host")
    return Ys


def convrot_mlp_workspace_size(M: int, K: int, N_up: int) -> int:
    return int(lib().convrot_mlp_workspace_size(M, K, N_up))


def convrot_mlp(X: torch.Tensor, G_up: int, up: Tuple, activation: int, G_down: int, down: Tuple,
                Y: Optional[torch.Tensor] = None, H: Optional[torch.Tensor] = None, workspace=None,
                stream=None) -> torch.Tensor:
    """Up linear, activation, down linear on the device. `up` and `down` are
    (weight codes, scale, bias, kchunk) tuples, the codes binary16 [N, K] or
    packed 4-bit [N, K/2] (uint8); with ACT_SWIGLU `up` is a pair of such
    tuples, (gate, up). H (optional, fp32 [M, N_up]) receives the activated
    up output that the down linear packs (GELU(Y_up), or with ACT_SWIGLU
    h = silu(gate) * up)."""
    xd = _xdtype(X)
    _need(X, X.dtype, "X")
    M, K = X.shape
    ups = list(up) if activation == ACT_SWIGLU else [up]
    dq, ds, db, dk = down
    N_up, N_down = ups[0][0].shape[0], dq.shape[0]
    if Y is None:
        Y = torch.empty((M, N_down), dtype=torch.float32, device=X.device)
    if H is not None:
        _need(H, torch.float32, "H")
    wu = make_weights([u[0] for u in ups], [u[1] for u in ups], [u[2] for u in ups], [H] * len(ups),
                      [u[3] for u in ups])
    wd = make_weights([dq], [ds], [db], [Y], [dk])
    ws = _workspace(convrot_mlp_workspace_size(M, K, N_up), X.device, workspace)
    _check(lib().convrot_mlp(_ptr(X), xd, M, K, G_up, wu, activation, G_down, wd, _ptr(ws), ws.numel(),
                             _stream(stream)), "convrot_mlp")
    return Y


def convrot_mlp_host_workspace_size(M: int, K: int, x_dtype: int, N_up: int, N_down: int,
                                    chunk_rows: int = 0) -> int:
    return int(lib().convrot_mlp_host_workspace_size(M, K, x_dtype, N_up, N_down, chunk_rows))


def convrot_mlp_host(X: torch.Tensor, G_up: int, up: Tuple, activation: int, G_down: int, down: Tuple,
                     Y: Optional[torch.Tensor] = None, chunk_rows: int = 0, workspace=None, stream=None,
                     copy_in_stream=None, copy_out_stream=None) -> torch.Tensor:
    """convrot_mlp on host arrays: X [M,K] and Y [M,N_down] live in (pinned)
    host memory, the weights on the device; row chunks are copied in, run
    and copied out on three streams so that transfers overlap compute. `up`
    and `down` as in convrot_mlp."""
    xd = _xdtype(X)
    if X.is_cuda or not X.is_contiguous():
        raise ValueError("X must be a contiguous host tensor")
    M, K = X.shape
    ups = list(up) if activation == ACT_SWIGLU else [up]
    dq, ds, db, dk = down
    N_up, N_down = ups[0][0].shape[0], dq.shape[0]
    dev = dq.device
    if Y is None:
        Y = torch.empty((M, N_down), dtype=torch.float32, pin_memory=True)
    if Y.is_cuda or Y.dtype != torch.float32 or not Y.is_contiguous():
        raise ValueError("Y must be a contiguous float32 host tensor")
    wu = make_weights([u[0] for u in ups], [u[1] for u in ups], [u[2] for u in ups], [None] * len(ups),
                      [u[3] for u in ups])
    wd = make_weights([dq], [ds], [db], [None], [dk])
    ws = _workspace(convrot_mlp_host_workspace_size(M, K, xd, N_up, N_down, chunk_rows), dev, workspace)
    _check(lib().convrot_mlp_host(X.data_ptr(), xd, M, K, G_up, wu, activation, G_down, wd, Y.data_ptr(),
                                  chunk_rows, _ptr(ws), ws.numel(), _stream(stream),
                                  _stream(copy_in_stream) if copy_in_stream else None,
                                  _stream(copy_out_stream) if copy_out_stream else None), "convrot_mlp_host")
    return Y


def convrot_linear_noalloc(X: torch.Tensor, G: int, q16s: Sequence[torch.Tensor],
                           scales: Sequence[Optional[torch.Tensor]],
                           biases: Sequence[Optional[torch.Tensor]],
                           Ys: Optional[List[torch.Tensor]] = None, stream=None,
                           weights=None, kchunks=None) -> List[torch.Tensor]:
    """convrot_linear without a workspace, for callers that cannot allocate
    device memory: the packed activation lives in the library's fixed device
    array (NOALLOC_SCRATCH_BYTES per GPU). Pass preallocated Ys to make the
    whole call allocation-free; calls that overlap on the GPU race."""
    xd = _xdtype(X)
    _need(X, X.dtype, "X")
    M, K = X.shape
    if Ys is None:
        Ys = [torch.empty((M, q.shape[0]), dtype=torch.float32, device=X.device) for q in q16s]
    if weights is None:
        weights = make_weights(q16s, scales, biases, Ys, kchunks)
    _check(lib().convrot_linear_noalloc(_ptr(X), xd, M, K, G, weights, len(q16s), _stream(stream)),
           "convrot_linear_noalloc")
    return Ys


def convrot_device_status(stream=None) -> int:
    return int(lib().convrot_device_status(_stream(stream)))


def convrot_test_unscale_sweep(divisors: torch.Tensor, y_exp: int, stream=None) -> Tuple[int, Optional[Tuple[float, float]]]:
    """Test-only: the GEMM epilogue's unscaling step against the IEEE division
    for every divisor in `divisors` (fp32, on the device) and all 2^23 values
    y = 1.m * 2^y_exp. Returns (count of results that differ, (divisor, y) of
    the first of them or None)."""
    _need(divisors, torch.float32, "divisors")
    out = torch.tensor([0, -1], dtype=torch.int64, device=divisors.device)  # count, first (~0)
    _check(lib().convrot_test_unscale_sweep(_ptr(divisors), divisors.numel(), int(y_exp), _ptr(out),
                                            out.data_ptr() + 8, _stream(stream)),
           "convrot_test_unscale_sweep")
    n, first = (int(v) for v in out.cpu())
    if n == 0:
        return 0, None
    first &= (1 << 64) - 1
    d = float(divisors[first >> 32].item())
    y = struct.unpack("<f", struct.pack("<I", first & 0xffffffff))[0]
    return n, (d, y)


def convrot_test_handover_timeout(Q_x16: torch.Tensor, s_x: torch.Tensor, q16s, scales, biases, wait_ns: int,
                                  workspace: torch.Tensor, Ys=None, stream=None):
    """Test-only GEMM launch whose split-tile hand-over waits can never be
    satisfied and give up after wait_ns: the kernel records CONVROT_ERR_TIMEOUT
    (read it with convrot_device_status) and exits, leaving those tiles of Ys
    unfinished. Returns Ys."""
    _need(Q_x16, torch.float16, "Q_x16")
    _need(s_x, torch.float32, "s_x")
    M, K = Q_x16.shape
    if Ys is None:
        Ys = [torch.empty((M, q.shape[0]), dtype=torch.float32, device=Q_x16.device) for q in q16s]
    weights = make_weights(q16s, scales, biases, Ys)
    _check(lib().convrot_test_handover_timeout(_ptr(Q_x16), _ptr(s_x), M, K, weights, len(q16s), _ptr(workspace),
                                               workspace.numel() * workspace.element_size(), int(wait_ns),
                                               _stream(stream)),
           "convrot_test_handover_timeout")
    return Ys


def convrot_linear_swiglu(X: torch.Tensor, G: int, gate: Tuple, up: Tuple, H: Optional[torch.Tensor] = None,
                          workspace=None, stream=None) -> torch.Tensor:
    """Split SwiGLU of two linears sharing X: h = silu(gate) * up, where gate
    and up are (q16, scale, bias, kchunk) tuples with the same N; one pack and
    one GEMM whose epilogue writes only h (fp32 [M, N])."""
    xd = _xdtype(X)
    _need(X, X.dtype, "X")
    M, K = X.shape
    N = gate[0].shape[0]
    if H is None:
        H = torch.empty((M, N), dtype=torch.float32, device=X.device)
    _need(H, torch.float32, "H")
    w = make_weights([gate[0], up[0]], [gate[1], up[1]], [gate[2], up[2]], [H, H], [gate[3], up[3]])
    ws = _workspace(convrot_linear_workspace_size(M, K), X.device, workspace)
    _check(lib().convrot_linear_swiglu(_ptr(X), xd, M, K, G, w, _ptr(ws), ws.numel(), _stream(stream)),
           "convrot_linear_swiglu")
    return H

