"""Python binding of libqgemm.so (include/qgemm.h): argument marshalling only.

Every function here has the name of a C entry point, takes torch tensors that
live on the current CUDA device, passes their data pointers and sizes through
ctypes and raises ``QGError`` when the library returns a non-zero status.  All
arithmetic runs in the library's CUDA kernels; there is no fallback.  If the
library has not been built, importing the binding works but the first call
raises ``QGLibraryMissing`` (build it with ``gemm_blockwise_dequant_gb300.build``).

PyTorch provides device memory and streams only.  Workspaces the library asks
for are allocated here, by torch, when the caller does not pass one.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "QG_OK", "QG_ERR_INVALID_ARG", "QG_ERR_UNSUPPORTED", "QG_ERR_CUDA", "QG_ERR_WORKSPACE_TOO_SMALL",
    "QG_F32", "QG_F16", "QG_BF16", "QGError", "QGLibraryMissing", "lib", "library_path",
    "qgemm_nbits", "qgemm_nbits_uniform_zp", "qgemm_codebook4", "qgemm_workspace_bytes",
    "qmoe_decode_fused", "qmoe_decode_fused_dp4a", "qmoe_decode_fused_noalloc", "qmoe_decode_workspace_bytes", "QG_QMOE_NOALLOC_SCRATCH_BYTES",
    "qg_fp16_uniform_value", "qg_dequant_nbits",
    "qg_dequant_nbits_uniform_zp", "qg_dequant_codebook4", "qg_read_device_fault", "qg_status_string",
    "qgemm_codebook4_nested", "qgemm_codebook4_nested_workspace_bytes", "qmoe_ragged_mm",
    "qmoe_ragged_mm_workspace_bytes", "qg_gather_block_quantized", "QG_WF_U2", "QG_WF_U4", "QG_WF_U8", "QG_WF_E4M3",
    "qgemm_nbits_packed_zp", "qgemm_nbits_packed_zp_workspace_bytes", "qg_test_bounded_wait",
    "qg_test_gemv_plan", "qmoe_ragged_mm_device_offsets", "qmoe_ragged_mm_device_offsets_workspace_bytes",
]

QG_OK, QG_ERR_INVALID_ARG, QG_ERR_UNSUPPORTED, QG_ERR_CUDA, QG_ERR_WORKSPACE_TOO_SMALL = 0, 1, 2, 3, 4
QG_F32, QG_F16, QG_BF16 = 0, 1, 2
QG_QMOE_NOALLOC_SCRATCH_BYTES = 1 << 20
QG_WF_U2, QG_WF_U4, QG_WF_U8, QG_WF_E4M3 = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libqgemm.so")
_lib = None
_lock = threading.Lock()


class QGError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s returned %s" % (where, _status_name(status)))


class QGLibraryMissing(ImportError):
    pass


def _status_name(s):
    return {0: "QG_OK", 1: "QG_ERR_INVALID_ARG", 2: "QG_ERR_UNSUPPORTED", 3: "QG_ERR_CUDA",
            4: "QG_ERR_WORKSPACE_TOO_SMALL"}.get(s, "status %d" % s)


_P, _I, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_SIGS = {
    "qgemm_nbits": ([_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P], _I),
    "qgemm_nbits_uniform_zp": ([_P, _I, _P, _P, _F, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P], _I),
    "qgemm_codebook4": ([_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P], _I),
    "qgemm_workspace_bytes": ([_I, _I, _I, _I, _I, _I], _SZ),
    "qmoe_decode_fused": ([_P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _SZ,
                           _P], _I),
    "qmoe_decode_fused_dp4a": ([_P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P,
                                _SZ, _P], _I),
    "qmoe_decode_workspace_bytes": ([_I, _I, _I], _SZ),
    "qmoe_decode_fused_noalloc": ([_P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P,
                                   _P], _I),
    "qg_fp16_uniform_value": ([_P, _SZ, _P, _P, _P, _SZ, _P], _I),
    "qg_dequant_nbits": ([_P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "qg_dequant_nbits_uniform_zp": ([_P, _P, _F, _P, _I, _I, _I, _I, _P], _I),
    "qg_dequant_codebook4": ([_P, _P, _P, _P, _I, _I, _I, _P], _I),
    "qg_gather_block_quantized": ([_P, ctypes.c_int64, _P, _I, _P, _P, ctypes.c_int64, _I, _I, _P, _I, _P, _P], _I),
    "qgemm_codebook4_nested": ([_P, _I, _P, _P, _P, _P, _P, _F, _I, _P, _I, _I, _I, _I, _I, _P, _SZ, _P], _I),
    "qgemm_codebook4_nested_workspace_bytes": ([_I, _I, _I, _I, _I], _SZ),
    "qgemm_nbits_packed_zp": ([_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P], _I),
    "qgemm_nbits_packed_zp_workspace_bytes": ([_I, _I, _I, _I, _I, _I], _SZ),
    "qmoe_ragged_mm": ([_P, _I, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P], _I),
    "qmoe_ragged_mm_workspace_bytes": ([_I, _P, _I, _I, _I, _I, _I], _SZ),
    "qmoe_ragged_mm_device_offsets": ([_P, _I, _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P, _P], _I),
    "qmoe_ragged_mm_device_offsets_workspace_bytes": ([_I], _SZ),
    "qg_read_device_fault": ([_P], _I),
    "qg_test_bounded_wait": ([_I, ctypes.c_uint, _P, _P], _I),
    "qg_test_gemv_plan": ([_I, _I, _I, _I, _I, _P], _I),
    "qg_status_string": ([_I], ctypes.c_char_p),
}


def lib():
    """The loaded libqgemm.so (raises QGLibraryMissing if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise QGLibraryMissing("libqgemm.so not built; run gemm_blockwise_dequant_gb300.build.build()")
            L = ctypes.CDLL(library_path)
            for name, (args, res) in _SIGS.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


# ---------------------------------------------------------------- marshalling
def _torch():
    import torch

    return torch


_DTYPE_CODES = None


def _dtype_code(t):
    global _DTYPE_CODES
    if _DTYPE_CODES is None:
        torch = _torch()
        _DTYPE_CODES = {torch.float32: QG_F32, torch.float16: QG_F16, torch.bfloat16: QG_BF16}
    return _DTYPE_CODES[t.dtype]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, where):
    if status != QG_OK:
        raise QGError(status, where)
    return status


def _workspace(need, workspace, device):
    """(workspace, its size in bytes): the caller's, else a new one of need()
    bytes (None when the call needs none); the library checks the size."""
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    nbytes = need()
    if nbytes == 0:
        return None, 0
    return _torch().empty(nbytes, dtype=_torch().uint8, device=device), nbytes


def qgemm_workspace_bytes(a_dtype: int, M: int, N: int, K: int, bits: int, block_size: int) -> int:
    return lib().qgemm_workspace_bytes(a_dtype, M, N, K, bits, block_size)


def qgemm_nbits(A, W, scales, zero_points, Y, *, bits, block_size, workspace=None, stream=None, raw=False):
    """Y[M,N] = A[M,K] . dequant(W)^T with fp16 scales and fp16 zero points (or None).

    A: [M, K] float32/float16/bfloat16; W: [N, K*bits/8] uint8; scales and
    zero_points: [N, K/block_size] float16; Y: [M, N] float32/float16/bfloat16.
    """
    M, K = A.shape
    N = W.shape[0]
    ws, wsb = _workspace(lambda: qgemm_workspace_bytes(_dtype_code(A), M, N, K, bits, block_size), workspace, A.device)
    s = lib().qgemm_nbits(_ptr(A), _dtype_code(A), _ptr(W), _ptr(scales), _ptr(zero_points), _ptr(Y),
                          _dtype_code(Y), M, N, K, bits, block_size, _ptr(ws), wsb, _stream(stream))
    return s if raw else _check(s, "qgemm_nbits")


def qgemm_nbits_uniform_zp(A, W, scales, uniform_zp, Y, *, bits, block_size, workspace=None, stream=None,
                           raw=False):
    """As qgemm_nbits with every zero point equal to the scalar uniform_zp."""
    M, K = A.shape
    N = W.shape[0]
    ws, wsb = _workspace(lambda: qgemm_workspace_bytes(_dtype_code(A), M, N, K, bits, block_size), workspace, A.device)
    s = lib().qgemm_nbits_uniform_zp(_ptr(A), _dtype_code(A), _ptr(W), _ptr(scales), float(uniform_zp), _ptr(Y),
                                     _dtype_code(Y), M, N, K, bits, block_size, _ptr(ws), wsb, _stream(stream))
    return s if raw else _check(s, "qgemm_nbits_uniform_zp")


def qgemm_codebook4(A, W, codebook, absmax, Y, *, block_size, workspace=None, stream=None, raw=False):
    """Y = A . (codebook[q] * absmax)^T; codebook [16] float32, absmax [N, K/block_size] float32."""
    M, K = A.shape
    N = W.shape[0]
    ws, wsb = _workspace(lambda: qgemm_workspace_bytes(_dtype_code(A), M, N, K, 4, block_size), workspace, A.device)
    s = lib().qgemm_codebook4(_ptr(A), _dtype_code(A), _ptr(W), _ptr(codebook), _ptr(absmax), _ptr(Y),
                              _dtype_code(Y), M, N, K, block_size, _ptr(ws), wsb, _stream(stream))
    return s if raw else _check(s, "qgemm_codebook4")


def qmoe_decode_workspace_bytes(k: int, hidden: int, inter: int) -> int:
    return lib().qmoe_decode_workspace_bytes(k, hidden, inter)


def qmoe_decode_fused(x, expert_ids, expert_weights, *, num_experts, fc1_w, fc1_scales, fc1_zp, fc1_bias, fc2_w,
                      fc2_scales, fc2_zp, fc2_bias, bits, block_size, y, swiglu_interleaved=0, status=None,
                      workspace=None, stream=None, raw=False):
    """One-token fused QMoE decode (fc1 -> SwiGLU -> fc2, weighted over the k slots); y [hidden] float16."""
    hidden = x.shape[-1]
    inter = fc2_w.shape[-1] * 8 // bits
    k = expert_ids.numel()
    ws, wsb = _workspace(lambda: qmoe_decode_workspace_bytes(k, hidden, inter), workspace, x.device)
    s = lib().qmoe_decode_fused(_ptr(x), _ptr(expert_ids), _ptr(expert_weights), k, num_experts, _ptr(fc1_w),
                                _ptr(fc1_scales), _ptr(fc1_zp), _ptr(fc1_bias), _ptr(fc2_w), _ptr(fc2_scales),
                                _ptr(fc2_zp), _ptr(fc2_bias), hidden, inter, bits, block_size,
                                int(swiglu_interleaved), _ptr(y), _ptr(status), _ptr(ws), wsb, _stream(stream))
    return s if raw else _check(s, "qmoe_decode_fused")


def qmoe_decode_fused_dp4a(x, expert_ids, expert_weights, *, num_experts, fc1_w, fc1_scales, fc1_zp, fc1_bias,
                           fc2_w, fc2_scales, fc2_zp, fc2_bias, bits, block_size, y, swiglu_interleaved=0,
                           status=None, workspace=None, stream=None, raw=False):
    """qmoe_decode_fused with int8 activations (per-block symmetric quantization, dp4a dot products)."""
    hidden = x.shape[-1]
    inter = fc2_w.shape[-1] * 8 // bits
    k = expert_ids.numel()
    ws, wsb = _workspace(lambda: qmoe_decode_workspace_bytes(k, hidden, inter), workspace, x.device)
    s = lib().qmoe_decode_fused_dp4a(_ptr(x), _ptr(expert_ids), _ptr(expert_weights), k, num_experts, _ptr(fc1_w),
                                     _ptr(fc1_scales), _ptr(fc1_zp), _ptr(fc1_bias), _ptr(fc2_w), _ptr(fc2_scales),
                                     _ptr(fc2_zp), _ptr(fc2_bias), hidden, inter, bits, block_size,
                                     int(swiglu_interleaved), _ptr(y), _ptr(status), _ptr(ws), wsb, _stream(stream))
    return s if raw else _check(s, "qmoe_decode_fused_dp4a")


def qmoe_decode_fused_noalloc(x, expert_ids, expert_weights, *, num_experts, fc1_w, fc1_scales, fc1_zp, fc1_bias,
                              fc2_w, fc2_scales, fc2_zp, fc2_bias, bits, block_size, y, swiglu_interleaved=0,
                              status=None, stream=None, raw=False):
    """qmoe_decode_fused without a workspace: the library's fixed device scratch is used
    (callers that cannot allocate; shapes beyond QG_QMOE_NOALLOC_SCRATCH_BYTES are refused)."""
    hidden = x.shape[-1]
    inter = fc2_w.shape[-1] * 8 // bits
    k = expert_ids.numel()
    s = lib().qmoe_decode_fused_noalloc(_ptr(x), _ptr(expert_ids), _ptr(expert_weights), k, num_experts,
                                        _ptr(fc1_w), _ptr(fc1_scales), _ptr(fc1_zp), _ptr(fc1_bias), _ptr(fc2_w),
                                        _ptr(fc2_scales), _ptr(fc2_zp), _ptr(fc2_bias), hidden, inter, bits,
                                        block_size, int(swiglu_interleaved), _ptr(y), _ptr(status), _stream(stream))
    return s if raw else _check(s, "qmoe_decode_fused_noalloc")


def qg_fp16_uniform_value(t, workspace=None, stream=None):
    """(is_uniform, value) for an fp16 tensor (bitwise equality of all elements)."""
    torch = _torch()
    if workspace is None:
        workspace = torch.empty(16, dtype=torch.uint8, device=t.device)
    u = ctypes.c_int(0)
    v = ctypes.c_float(0.0)
    _check(lib().qg_fp16_uniform_value(_ptr(t), t.numel(), ctypes.byref(u), ctypes.byref(v), _ptr(workspace),
                                       workspace.numel(), _stream(stream)), "qg_fp16_uniform_value")
    return bool(u.value), (float(v.value) if u.value else None)


def qg_dequant_nbits(W, scales, zero_points, out, *, bits, block_size, stream=None, raw=False):
    N, K = out.shape
    s = lib().qg_dequant_nbits(_ptr(W), _ptr(scales), _ptr(zero_points), _ptr(out), N, K, bits, block_size,
                               _stream(stream))
    return s if raw else _check(s, "qg_dequant_nbits")


def qg_dequant_nbits_uniform_zp(W, scales, uniform_zp, out, *, bits, block_size, stream=None, raw=False):
    N, K = out.shape
    s = lib().qg_dequant_nbits_uniform_zp(_ptr(W), _ptr(scales), float(uniform_zp), _ptr(out), N, K, bits,
                                          block_size, _stream(stream))
    return s if raw else _check(s, "qg_dequant_nbits_uniform_zp")


def qg_dequant_codebook4(W, codebook, absmax, out, *, block_size, stream=None, raw=False):
    N, K = out.shape
    s = lib().qg_dequant_codebook4(_ptr(W), _ptr(codebook), _ptr(absmax), _ptr(out), N, K, block_size,
                                   _stream(stream))
    return s if raw else _check(s, "qg_dequant_codebook4")


def qgemm_codebook4_nested_workspace_bytes(a_dtype: int, M: int, N: int, K: int, block_size: int) -> int:
    return lib().qgemm_codebook4_nested_workspace_bytes(a_dtype, M, N, K, block_size)


def qgemm_codebook4_nested(A, W, codebook, absmax_q, absmax_table, absmax2, absmax_offset, Y, *, block_size,
                           nested_block=256, workspace=None, stream=None, raw=False):
    """qgemm_codebook4 with a nested absmax: absmax = table[absmax_q] * absmax2[i // nested_block] + offset
    (absmax_q [N, K/block_size] uint8, absmax_table [256] float32, absmax2 float32)."""
    M, K = A.shape
    N = W.shape[0]
    ws, wsb = _workspace(lambda: qgemm_codebook4_nested_workspace_bytes(_dtype_code(A), M, N, K, block_size), workspace,
                         A.device)
    s = lib().qgemm_codebook4_nested(_ptr(A), _dtype_code(A), _ptr(W), _ptr(codebook), _ptr(absmax_q),
                                     _ptr(absmax_table), _ptr(absmax2), float(absmax_offset), nested_block, _ptr(Y),
                                     _dtype_code(Y), M, N, K, block_size, _ptr(ws), wsb, _stream(stream))
    return s if raw else _check(s, "qgemm_codebook4_nested")


def qgemm_nbits_packed_zp_workspace_bytes(a_dtype: int, M: int, N: int, K: int, bits: int, block_size: int) -> int:
    return lib().qgemm_nbits_packed_zp_workspace_bytes(a_dtype, M, N, K, bits, block_size)


def qgemm_nbits_packed_zp(A, W, scales, zero_points_packed, Y, *, bits, block_size, workspace=None, stream=None,
                          raw=False):
    """qgemm_nbits with unsigned integer zero points packed like the codes:
    zero_points_packed [N, ceil((K/block_size)*bits/8)] uint8, field b of a row
    at bit b*bits, least significant bit first."""
    M, K = A.shape
    N = W.shape[0]
    ws, wsb = _workspace(lambda: qgemm_nbits_packed_zp_workspace_bytes(_dtype_code(A), M, N, K, bits, block_size),
                         workspace, A.device)
    s = lib().qgemm_nbits_packed_zp(_ptr(A), _dtype_code(A), _ptr(W), _ptr(scales), _ptr(zero_points_packed),
                                    _ptr(Y), _dtype_code(Y), M, N, K, bits, block_size, _ptr(ws), wsb,
                                    _stream(stream))
    return s if raw else _check(s, "qgemm_nbits_packed_zp")


def _host_offsets(offsets):
    import numpy as np

    off = np.ascontiguousarray(np.asarray(offsets.cpu() if hasattr(offsets, "cpu") else offsets, dtype=np.int64))
    return off, off.ctypes.data_as(ctypes.c_void_p)


def qmoe_ragged_mm_workspace_bytes(x_dtype: int, offsets, N: int, K: int, bits: int, block_size: int) -> int:
    off, p = _host_offsets(offsets)
    return lib().qmoe_ragged_mm_workspace_bytes(x_dtype, p, off.size - 1, N, K, bits, block_size)


def qmoe_ragged_mm(X, offsets, W, scales, zero_points, Y, *, bits, block_size, workspace=None, stream=None,
                   raw=False):
    """Y[r] = X[r] . dequant(W[e])^T for the rows r of expert e (offsets[e] <= r < offsets[e+1]).

    X: [T, K] float32/float16/bfloat16; offsets: host sequence (or CPU tensor) of E+1 ints;
    W: [E, N, K*bits/8] uint8; scales / zero_points: [E, N, K/block_size] float16 (zero_points None
    for the midpoint); Y: [T, N] float32/float16/bfloat16.
    """
    off, p = _host_offsets(offsets)
    E, N = W.shape[0], W.shape[1]
    K = X.shape[1]
    ws, wsb = _workspace(lambda: lib().qmoe_ragged_mm_workspace_bytes(_dtype_code(X), p, E, N, K, bits, block_size),
                         workspace, X.device)
    s = lib().qmoe_ragged_mm(_ptr(X), _dtype_code(X), p, E, _ptr(W), _ptr(scales), _ptr(zero_points), _ptr(Y),
                             _dtype_code(Y), N, K, bits, block_size, _ptr(ws), wsb, _stream(stream))
    return s if raw else _check(s, "qmoe_ragged_mm")


def qmoe_ragged_mm_device_offsets_workspace_bytes(num_experts: int) -> int:
    return lib().qmoe_ragged_mm_device_offsets_workspace_bytes(int(num_experts))


def qmoe_ragged_mm_device_offsets(X, offsets_dev, W, scales, zero_points, Y, *, bits, block_size, status=None,
                                  workspace=None, stream=None, raw=False):
    """qmoe_ragged_mm with the E+1 expert offsets in a device int64 tensor (no host copy).

    X: [max_rows, K] float16/bfloat16 (max_rows >= offsets[E]); Y: [max_rows, N]; rows of Y at or
    past offsets[E] are left untouched; status: a device int32 set to 1 for refused offsets, or None.
    """
    E, N = W.shape[0], W.shape[1]
    max_rows, K = X.shape
    ws, wsb = _workspace(lambda: lib().qmoe_ragged_mm_device_offsets_workspace_bytes(E), workspace, X.device)
    s = lib().qmoe_ragged_mm_device_offsets(_ptr(X), _dtype_code(X), _ptr(offsets_dev), E, max_rows, _ptr(W),
                                            _ptr(scales), _ptr(zero_points), _ptr(Y), _dtype_code(Y), N, K, bits,
                                            block_size, _ptr(ws), wsb, _ptr(status), _stream(stream))
    return s if raw else _check(s, "qmoe_ragged_mm_device_offsets")


def qg_gather_block_quantized(indices, W, scales, zero_points, Y, *, w_format, block_size, status=None, stream=None,
                              raw=False):
    """Y[i] = dequant(table row indices[i]) for a block-quantized [vocab, D] table.

    indices: int64 (any shape; Y is [indices.numel(), D]); W: [vocab, D*bits/8] uint8 codes or
    [vocab, D] E4M3 bytes; scales / zero_points: [vocab, D/block_size] float16 (zero_points None
    for the midpoint, and for E4M3); Y: float32/float16/bfloat16; status: a device int32 or None.
    """
    n, D = Y.shape
    s = lib().qg_gather_block_quantized(_ptr(indices), n, _ptr(W), int(w_format), _ptr(scales), _ptr(zero_points),
                                        W.shape[0], D, block_size, _ptr(Y), _dtype_code(Y), _ptr(status),
                                        _stream(stream))
    return s if raw else _check(s, "qg_gather_block_quantized")


def qg_read_device_fault() -> int:
    v = ctypes.c_uint(0)
    _check(lib().qg_read_device_fault(ctypes.byref(v)), "qg_read_device_fault")
    return int(v.value)


def qg_test_bounded_wait(fill: bool, limit_us: int, out, stream=None, raw=False):
    """Test hook (include/qgemm_testing.h): the library's bounded pipeline wait
    in a one-CTA kernel whose producer fills the stage only if `fill`; out is a
    device int32 tensor of 3 (1: that consumer warp's wait completed, 0: it
    gave up)."""
    s = lib().qg_test_bounded_wait(1 if fill else 0, int(limit_us), _ptr(out), _stream(stream))
    return s if raw else _check(s, "qg_test_bounded_wait")


def qg_test_gemv_plan(M: int, N: int, K: int, a_dtype: int = QG_F32, zp_mode: int = 2):
    """Test hook (include/qgemm_testing.h): the launch plan of the 2-bit
    tensor-core GEMV for this shape -- a dict of rows_per_tile, warps (consumer
    warps), ctas, stages -- or None when the shape takes another path."""
    out = (ctypes.c_int * 4)()
    s = lib().qg_test_gemv_plan(int(M), int(N), int(K), int(a_dtype), int(zp_mode), ctypes.cast(out, ctypes.c_void_p))
    if s == QG_ERR_UNSUPPORTED:
        return None
    _check(s, "qg_test_gemv_plan")
    return dict(zip(("rows_per_tile", "warps", "ctas", "stages"), list(out)))


def qg_status_string(status: int) -> str:
    return lib().qg_status_string(status).decode()
