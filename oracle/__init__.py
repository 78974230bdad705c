"""CPU oracle for blockwise low-bit dequantize + GEMM and the fused QMoE decode.

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The GPU library never
imports, links or runs anything here, and this package shares no code with it.

The arithmetic lives in ``qgemm_oracle.c`` (plain loops, fp32 dequantization,
fp64 accumulation); this module compiles it with gcc and wraps it with ctypes.
Every function is pinned by ``tests/test_oracle_pins.py``.

Sources: hip-ep pull requests #1318 (2-bit MatMulNBits, section "What",
Commit 1; the kernel test table's gather_block_quantized leaves) and #1328 (fused QMoE decode, sections "Summary" and "What"), and
bitsandbytes pull request #1979 ("[ROCm] Fused 4-bit SIMT GEMM", section
"Summary").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qgemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16, F64 = 0, 1, 2, 3
ZP_NONE, ZP_TENSOR, ZP_UNIFORM = 0, 1, 2
# table formats of the embedding gather
W_U2, W_U4, W_U8, W_E4M3 = 0, 1, 2, 3
W_BITS = {W_U2: 2, W_U4: 4, W_U8: 8, W_E4M3: 8}


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into a shared library (gcc, no FP contraction)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-std=c11",
               "-shared", "-fPIC", src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library and declare its signatures."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        P, I64, I, F, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = D
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = D
        lib.oracle_code.argtypes = [P, I64, I64, I64, I]
        lib.oracle_code.restype = I
        lib.oracle_dequant_nbits.argtypes = [P, P, P, I, F, I64, I64, I, I, P]
        lib.oracle_dequant_nbits.restype = None
        lib.oracle_dequant_codebook4.argtypes = [P, P, P, I64, I64, I, P]
        lib.oracle_dequant_codebook4.restype = None
        lib.oracle_qgemm_nbits.argtypes = [P, I, P, P, P, I, F, I64, I64, I64, I, I, P, I64, P]
        lib.oracle_qgemm_nbits.restype = None
        lib.oracle_qgemm_codebook4.argtypes = [P, I, P, P, P, I64, I64, I64, I, P, I64, P]
        lib.oracle_qgemm_codebook4.restype = None
        lib.oracle_fp16_uniform_value.argtypes = [P, I64, P]
        lib.oracle_fp16_uniform_value.restype = I
        lib.oracle_qmoe_decode.argtypes = [P, P, P, I, I, P, P, P, P, P, P, P, P, I64, I64, I, I, I, P, P, P]
        lib.oracle_qmoe_decode.restype = I
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = D
        lib.oracle_gather_block_quantized.argtypes = [P, I64, P, I, P, P, I64, I64, I, P]
        lib.oracle_gather_block_quantized.restype = I64
        lib.oracle_quantize_i8_blocks.argtypes = [P, I64, I, P, P]
        lib.oracle_quantize_i8_blocks.restype = None
        lib.oracle_qmoe_decode_dp4a.argtypes = [P, P, P, I, I, P, P, P, P, P, P, P, P, I64, I64, I, I, I, P, P, P,
                                                P, P]
        lib.oracle_qmoe_decode_dp4a.restype = I
        lib.oracle_qmoe_ragged_mm.argtypes = [P, I, P, I, P, P, P, I64, I64, I, I, P]
        lib.oracle_qmoe_ragged_mm.restype = I
        lib.oracle_nested_absmax.argtypes = [P, P, P, F, I, I64, P]
        lib.oracle_nested_absmax.restype = None
        lib.oracle_unpack_zero_points.argtypes = [P, I64, I64, I, P]
        lib.oracle_unpack_zero_points.restype = None
        if path is None:
            _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError("expected %s, got %s" % (np.dtype(dtype), a.dtype))
    return a


def _a_dtype(A):
    if A.dtype == np.float32:
        return F32
    if A.dtype == np.float64:
        return F64
    raise TypeError("A must be float32, float64, or uint16 with an explicit a_dtype")


def half_to_double(bits: int, lib=None) -> float:
    return (lib or load()).oracle_half_to_double(int(bits))


def bf16_to_double(bits: int, lib=None) -> float:
    return (lib or load()).oracle_bf16_to_double(int(bits))


def code(W, K, n, k, bits, lib=None) -> int:
    W = _c(W, np.uint8)
    return (lib or load()).oracle_code(_ptr(W), K, n, k, bits)


def dequant_nbits(W, scales, zero_points=None, *, N, K, bits, block_size, uniform_zp=None, lib=None):
    """fp32 [N, K] dequantized weights (zero points: tensor, scalar or absent)."""
    W = _c(W, np.uint8)
    scales = _c(scales, np.uint16)
    zp = _c(zero_points, np.uint16)
    mode = ZP_UNIFORM if uniform_zp is not None else (ZP_TENSOR if zp is not None else ZP_NONE)
    out = np.empty((N, K), dtype=np.float32)
    (lib or load()).oracle_dequant_nbits(_ptr(W), _ptr(scales), _ptr(zp), mode,
                                         float(uniform_zp or 0.0), N, K, bits, block_size, _ptr(out))
    return out


def dequant_codebook4(W, codebook, absmax, *, N, K, block_size, lib=None):
    W = _c(W, np.uint8)
    codebook = _c(codebook, np.float32)
    absmax = _c(absmax, np.float32)
    out = np.empty((N, K), dtype=np.float32)
    (lib or load()).oracle_dequant_codebook4(_ptr(W), _ptr(codebook), _ptr(absmax), N, K, block_size,
                                             _ptr(out))
    return out


def qgemm_nbits(A, W, scales, zero_points=None, *, M, N, K, bits, block_size, uniform_zp=None,
                a_dtype=None, rows=None, lib=None):
    """Unrounded fp64 Y[M, len(rows)] = A . dequant(W)[rows].T  (rows=None: all N)."""
    if a_dtype is None:
        a_dtype = _a_dtype(A)
    A = np.ascontiguousarray(A)
    W = _c(W, np.uint8)
    scales = _c(scales, np.uint16)
    zp = _c(zero_points, np.uint16)
    mode = ZP_UNIFORM if uniform_zp is not None else (ZP_TENSOR if zp is not None else ZP_NONE)
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n_rows = N if rows_a is None else rows_a.size
    Y = np.empty((M, n_rows), dtype=np.float64)
    (lib or load()).oracle_qgemm_nbits(_ptr(A), a_dtype, _ptr(W), _ptr(scales), _ptr(zp), mode,
                                       float(uniform_zp or 0.0), M, N, K, bits, block_size,
                                       _ptr(rows_a), n_rows, _ptr(Y))
    return Y


def zp_packed_row_bytes(nb: int, bits: int) -> int:
    """Bytes per row of packed integer zero points (rows padded to whole bytes)."""
    return (nb * bits + 7) // 8


def unpack_zero_points(zp_packed, *, N, nb, bits, lib=None):
    """int32 [N, nb] zero points from their packed form [N, ceil(nb*bits/8)] uint8."""
    zp = _c(zp_packed, np.uint8)
    assert zp.size == N * zp_packed_row_bytes(nb, bits)
    out = np.empty((N, nb), dtype=np.int32)
    (lib or load()).oracle_unpack_zero_points(_ptr(zp), N, nb, bits, _ptr(out))
    return out


def qgemm_nbits_packed_zp(A, W, scales, zp_packed, *, M, N, K, bits, block_size, a_dtype=None, rows=None,
                          lib=None):
    """qgemm_nbits with packed integer zero points: the unpacked integers (exact
    in fp16) serve as the zero-point tensor."""
    z = unpack_zero_points(zp_packed, N=N, nb=K // block_size, bits=bits, lib=lib)
    z16 = z.astype(np.float16).view(np.uint16)
    return qgemm_nbits(A, W, scales, z16, M=M, N=N, K=K, bits=bits, block_size=block_size, a_dtype=a_dtype,
                       rows=rows, lib=lib)


def qgemm_codebook4(A, W, codebook, absmax, *, M, N, K, block_size, a_dtype=None, rows=None, lib=None):
    if a_dtype is None:
        a_dtype = _a_dtype(A)
    A = np.ascontiguousarray(A)
    W = _c(W, np.uint8)
    codebook = _c(codebook, np.float32)
    absmax = _c(absmax, np.float32)
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n_rows = N if rows_a is None else rows_a.size
    Y = np.empty((M, n_rows), dtype=np.float64)
    (lib or load()).oracle_qgemm_codebook4(_ptr(A), a_dtype, _ptr(W), _ptr(codebook), _ptr(absmax),
                                           M, N, K, block_size, _ptr(rows_a), n_rows, _ptr(Y))
    return Y


def nested_absmax(qa, table256, absmax2, offset, nested_block, lib=None):
    """Expand a nested (double-quantized) absmax: fp32 array of qa's shape."""
    qa = _c(qa, np.uint8)
    table256 = _c(table256, np.float32)
    absmax2 = _c(absmax2, np.float32)
    out = np.empty(qa.shape, dtype=np.float32)
    (lib or load()).oracle_nested_absmax(_ptr(qa), _ptr(table256), _ptr(absmax2), float(offset), nested_block,
                                         qa.size, _ptr(out))
    return out


def qgemm_codebook4_nested(A, W, codebook, qa, table256, absmax2, offset, *, M, N, K, block_size, nested_block,
                           a_dtype=None, rows=None, lib=None):
    """The codebook GEMM with a nested absmax: the expansion above, then the plain codebook GEMM."""
    absmax = nested_absmax(qa, table256, absmax2, offset, nested_block, lib=lib)
    return qgemm_codebook4(A, W, codebook, absmax, M=M, N=N, K=K, block_size=block_size, a_dtype=a_dtype,
                           rows=rows, lib=lib)


def fp16_uniform_value(t, lib=None):
    """(is_uniform, value) for a uint16 array of fp16 bit patterns."""
    t = _c(np.asarray(t).reshape(-1), np.uint16)
    v = ctypes.c_float(0.0)
    r = (lib or load()).oracle_fp16_uniform_value(_ptr(t), t.size, ctypes.addressof(v))
    return bool(r), (float(v.value) if r else None)


def qmoe_decode(x_f16, ids, weights, *, num_experts, fc1_w, fc1_scales, fc1_zp, fc1_bias, fc2_w,
                fc2_scales, fc2_zp, fc2_bias, hidden, inter, bits, block_size, swiglu_interleaved=0,
                lib=None):
    """Unrounded fp64 y[hidden]; also returns the number of out-of-range expert slots."""
    x_f16 = _c(x_f16, np.uint16)
    ids = _c(ids, np.int32)
    weights = _c(weights, np.float32)
    fc1_w, fc2_w = _c(fc1_w, np.uint8), _c(fc2_w, np.uint8)
    fc1_scales, fc2_scales = _c(fc1_scales, np.uint16), _c(fc2_scales, np.uint16)
    fc1_zp, fc2_zp = _c(fc1_zp, np.uint16), _c(fc2_zp, np.uint16)
    fc1_bias, fc2_bias = _c(fc1_bias, np.uint16), _c(fc2_bias, np.uint16)
    g = np.empty(2 * inter, dtype=np.float64)
    h = np.empty(inter, dtype=np.float64)
    y = np.empty(hidden, dtype=np.float64)
    bad = (lib or load()).oracle_qmoe_decode(
        _ptr(x_f16), _ptr(ids), _ptr(weights), ids.size, num_experts, _ptr(fc1_w), _ptr(fc1_scales),
        _ptr(fc1_zp), _ptr(fc1_bias), _ptr(fc2_w), _ptr(fc2_scales), _ptr(fc2_zp), _ptr(fc2_bias),
        hidden, inter, bits, block_size, int(swiglu_interleaved), _ptr(g), _ptr(h), _ptr(y))
    return y, bad


def quantize_i8_blocks(v, block_size, lib=None):
    """Per-block symmetric int8 quantization of an fp32 vector (dp4a QMoE activations).

    Returns (q8 int8 [n], sx float32 [n / block_size]).
    """
    v = _c(np.asarray(v, dtype=np.float32).reshape(-1), np.float32)
    q8 = np.empty(v.size, dtype=np.int8)
    sx = np.empty(v.size // block_size, dtype=np.float32)
    (lib or load()).oracle_quantize_i8_blocks(_ptr(v), v.size, block_size, _ptr(q8), _ptr(sx))
    return q8, sx


def qmoe_decode_dp4a(x_f16, ids, weights, *, num_experts, fc1_w, fc1_scales, fc1_zp, fc1_bias, fc2_w,
                     fc2_scales, fc2_zp, fc2_bias, hidden, inter, bits, block_size, swiglu_interleaved=0,
                     lib=None, return_g=False):
    """The int8-activation decode: unrounded fp64 y[hidden] and the number of out-of-range slots
    (and, with return_g, the fc1 output g[2*inter] of the last valid slot)."""
    x_f16 = _c(x_f16, np.uint16)
    ids = _c(ids, np.int32)
    weights = _c(weights, np.float32)
    fc1_w, fc2_w = _c(fc1_w, np.uint8), _c(fc2_w, np.uint8)
    fc1_scales, fc2_scales = _c(fc1_scales, np.uint16), _c(fc2_scales, np.uint16)
    fc1_zp, fc2_zp = _c(fc1_zp, np.uint16), _c(fc2_zp, np.uint16)
    fc1_bias, fc2_bias = _c(fc1_bias, np.uint16), _c(fc2_bias, np.uint16)
    n = max(hidden, inter)
    g = np.empty(2 * inter, dtype=np.float64)
    h = np.empty(n, dtype=np.float32)
    q8 = np.empty(n, dtype=np.int8)
    sx = np.empty(n // block_size, dtype=np.float32)
    y = np.empty(hidden, dtype=np.float64)
    bad = (lib or load()).oracle_qmoe_decode_dp4a(
        _ptr(x_f16), _ptr(ids), _ptr(weights), ids.size, num_experts, _ptr(fc1_w), _ptr(fc1_scales),
        _ptr(fc1_zp), _ptr(fc1_bias), _ptr(fc2_w), _ptr(fc2_scales), _ptr(fc2_zp), _ptr(fc2_bias),
        hidden, inter, bits, block_size, int(swiglu_interleaved), _ptr(g), _ptr(h), _ptr(q8), _ptr(sx), _ptr(y))
    return (y, bad, g) if return_g else (y, bad)


def qmoe_ragged_mm(X, offsets, W, scales, zero_points=None, *, N, K, bits, block_size, x_dtype=None, lib=None):
    """Ragged expert GEMM: rows offsets[e] .. offsets[e+1]-1 of X use expert e's weight.

    X: [T, K] float32 / float64, or uint16 fp16 / bf16 bit patterns with x_dtype;
    W: [E, N, K*bits/8]; scales / zero_points: [E, N, K/block_size] fp16 bits.
    Returns fp64 Y [T, N] (unrounded).  Raises ValueError for offsets that do not
    start at 0 or decrease.
    """
    lib = lib or load()
    X = np.ascontiguousarray(X)
    if x_dtype is None:
        x_dtype = _a_dtype(X)
    off = _c(np.asarray(offsets, dtype=np.int64), np.int64)
    E = off.size - 1
    W = _c(W, np.uint8)
    scales = _c(scales, np.uint16)
    zero_points = _c(zero_points, np.uint16)
    T = int(off[-1])
    Y = np.zeros((T, N), dtype=np.float64)
    if lib.oracle_qmoe_ragged_mm(_ptr(X), x_dtype, _ptr(off), E, _ptr(W), _ptr(scales), _ptr(zero_points), N, K,
                                 bits, block_size, _ptr(Y)) != 0:
        raise ValueError("offsets must start at 0 and not decrease")
    return Y


def e4m3_to_double(bits: int, lib=None) -> float:
    return (lib or load()).oracle_e4m3_to_double(bits)


def gather_block_quantized(indices, W, scales, zero_points=None, *, V, D, fmt, block_size, lib=None):
    """Gather rows of a block-quantized [V][D] table (kernel test table, gather_block_quantized).

    Returns (out fp32 [n][D] exact dequantized values, number of indices outside [-V, V)).
    Rounding to an output type is the caller's step (numpy float16 / torch bfloat16, RN-even).
    """
    lib = lib or load()
    idx = _c(np.asarray(indices, dtype=np.int64).reshape(-1), np.int64)
    W = _c(W, np.uint8)
    scales = _c(scales, np.uint16)
    zero_points = _c(zero_points, np.uint16)
    if fmt == W_E4M3 and zero_points is not None:
        raise ValueError("E4M3 tables have no zero points")
    n = idx.shape[0]
    out = np.empty((n, D), dtype=np.float32)
    bad = lib.oracle_gather_block_quantized(_ptr(idx), n, _ptr(W), fmt, _ptr(scales), _ptr(zero_points), V, D,
                                            block_size, _ptr(out))
    return out, int(bad)


def max_rel_l2(Y, Yref) -> float:
    """max over rows m of ||Y[m] - Yref[m]||_2 / ||Yref[m]||_2 (metric of the parity bar)."""
    Y = np.asarray(Y, dtype=np.float64).reshape(np.asarray(Yref).shape[0] if np.ndim(Yref) > 1 else 1, -1)
    R = np.asarray(Yref, dtype=np.float64).reshape(Y.shape)
    num = np.linalg.norm(Y - R, axis=1)
    den = np.linalg.norm(R, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(den > 0, num / np.where(den > 0, den, 1.0), np.where(num > 0, np.inf, 0.0))
    return float(np.max(r)) if r.size else 0.0
