"""Host-side argument checks of the C ABI, on the CPU.

Every refusal below is decided on the host before the library touches the
device (the header documents that refusals come first), so these calls run
without a GPU and exercise the validation logic of the entry points added for
the 3-bit / 8-bit codes, the int8 QMoE decode, the ragged expert GEMM, the nested
absmax and the embedding gather.  Pointers are fake but never dereferenced.
"""
import ctypes

import numpy as np
import pytest

qg = pytest.importorskip("gemm_blockwise_dequant_gb300")


@pytest.fixture(scope="module")
def L():
    from gemm_blockwise_dequant_gb300 import build

    build.build()
    return qg.lib()


P16 = ctypes.c_void_p(4096)  # a 16-byte aligned, never dereferenced address


def _off(values):
    a = np.ascontiguousarray(np.asarray(values, dtype=np.int64))
    return a, a.ctypes.data_as(ctypes.c_void_p)


def test_ragged_refuses_bad_offsets_widths_and_alignment(L):
    call = lambda off, E, N=64, K=64, bits=4, bs=32, x=1, y=1: L.qmoe_ragged_mm(
        P16, x, off, E, P16, P16, None, P16, y, N, K, bits, bs, None, 0, None)
    keep = []
    a, p = _off([1, 2, 3]); keep.append(a)
    assert call(p, 2) == qg.QG_ERR_INVALID_ARG          # does not start at 0
    a, p = _off([0, 3, 2, 5]); keep.append(a)
    assert call(p, 3) == qg.QG_ERR_INVALID_ARG          # decreases
    assert call(None, 3) == qg.QG_ERR_INVALID_ARG       # no offsets
    a, p = _off([0, 2, 2, 5]); keep.append(a)
    assert call(p, 0) == qg.QG_ERR_INVALID_ARG          # no experts
    assert call(p, 3, bits=3) == qg.QG_ERR_UNSUPPORTED  # 3-bit codes: not for the stacked layout
    assert call(p, 3, bs=16) == qg.QG_ERR_UNSUPPORTED
    assert call(p, 3, K=80) == qg.QG_ERR_INVALID_ARG    # K % block_size
    assert call(p, 3, x=7) == qg.QG_ERR_INVALID_ARG     # activation type
    # u2, K = 32, N odd: one expert's codes are 8 * N bytes, not a multiple of 16
    assert call(p, 3, N=63, K=32, bits=2) == qg.QG_ERR_UNSUPPORTED
    a, p = _off([0, 0, 0]); keep.append(a)
    assert call(p, 2) == qg.QG_OK                       # no rows: nothing to do
    a, p = _off([2, 3])
    assert L.qmoe_ragged_mm_workspace_bytes(1, p, 1, 64, 64, 4, 32) == 0


def test_ragged_device_offsets_needs_no_workspace(L):
    """The device-offset launch numbers its tiles inside the kernel: no
    workspace at any expert count, and a NULL workspace passes the host
    checks (refusals here come from the other arguments)."""
    for E in (1, 2, 128, 256, 257):
        assert L.qmoe_ragged_mm_device_offsets_workspace_bytes(E) == 0
    call = lambda E=4, x=1, bits=4, bs=32, K=64, off=P16: L.qmoe_ragged_mm_device_offsets(
        P16, x, off, E, 64, P16, P16, None, P16, 1, 64, K, bits, bs, None, 0, None, None)
    assert call(x=0) == qg.QG_ERR_UNSUPPORTED     # fp32 activations: not on the grouped launch
    assert call(E=257) == qg.QG_ERR_UNSUPPORTED
    assert call(bits=3) == qg.QG_ERR_UNSUPPORTED
    assert call(K=80) == qg.QG_ERR_INVALID_ARG    # K % block_size
    assert call(off=ctypes.c_void_p(4100)) == qg.QG_ERR_INVALID_ARG  # offsets not 8-byte aligned
    assert call(off=None) == qg.QG_ERR_INVALID_ARG


def test_gather_refusals(L):
    call = lambda n=4, fmt=qg.QG_WF_U4, zp=None, V=100, D=64, bs=32, y=1: L.qg_gather_block_quantized(
        P16, n, P16, fmt, P16, zp, V, D, bs, P16, y, None, None)
    assert call(n=-1) == qg.QG_ERR_INVALID_ARG
    assert call(V=-1) == qg.QG_ERR_INVALID_ARG
    assert call(fmt=7) == qg.QG_ERR_UNSUPPORTED
    assert call(fmt=-1) == qg.QG_ERR_UNSUPPORTED
    assert call(y=5) == qg.QG_ERR_UNSUPPORTED
    assert call(bs=16) == qg.QG_ERR_UNSUPPORTED
    assert call(D=80) == qg.QG_ERR_INVALID_ARG
    assert call(fmt=qg.QG_WF_E4M3, zp=P16) == qg.QG_ERR_INVALID_ARG  # E4M3 tables have no zero point
    assert call(n=0) == qg.QG_OK
    assert call(D=0) == qg.QG_OK


def test_nested_codebook_refusals(L):
    call = lambda nb=256, off=0.06, M=1, bs=64, a=2: L.qgemm_codebook4_nested(
        P16, a, P16, P16, P16, P16, P16, off, nb, P16, 2, M, 64, 256, bs, None, 0, None)
    assert call(nb=0) == qg.QG_ERR_INVALID_ARG
    assert call(off=float("nan")) == qg.QG_ERR_INVALID_ARG
    assert call(bs=48) == qg.QG_ERR_UNSUPPORTED
    assert call(a=9) == qg.QG_ERR_INVALID_ARG
    assert call(M=0) == qg.QG_OK
    assert L.qgemm_codebook4_nested_workspace_bytes(2, 1, 64, 256, 48) == 0


def test_dp4a_decode_size_limit_and_widths(L):
    call = lambda hidden=256, inter=256, bits=4, bs=32: L.qmoe_decode_fused_dp4a(
        P16, P16, P16, 2, 4, P16, P16, None, None, P16, P16, None, None, hidden, inter, bits, bs, 0, P16, None,
        P16, 1 << 20, None)
    assert call(hidden=70016) == qg.QG_ERR_UNSUPPORTED  # the quantized vector must fit in shared memory
    assert call(bits=3) == qg.QG_ERR_UNSUPPORTED
    assert call(bs=16) == qg.QG_ERR_UNSUPPORTED
    assert call(hidden=272) == qg.QG_ERR_INVALID_ARG    # hidden % block_size


def test_three_bit_codes_are_accepted_widths(L):
    # bits 5 is refused, 3 passes the width check (and then fails on the zero-sized problem as OK)
    assert L.qgemm_nbits(P16, 0, P16, P16, None, P16, 0, 1, 64, 64, 5, 32, None, 0, None) == qg.QG_ERR_UNSUPPORTED
    assert L.qgemm_nbits(P16, 0, P16, P16, None, P16, 0, 0, 64, 64, 3, 32, None, 0, None) == qg.QG_OK


def test_packed_zp_refusals(L):
    call = lambda zp=P16, M=1, K=256, bits=4, bs=64, a=0, y=0, ws=None, wsb=0: L.qgemm_nbits_packed_zp(
        P16, a, P16, P16, zp, P16, y, M, 64, K, bits, bs, ws, wsb, None)
    assert call(a=9) == qg.QG_ERR_INVALID_ARG
    assert call(y=7) == qg.QG_ERR_INVALID_ARG
    assert call(M=-1) == qg.QG_ERR_INVALID_ARG
    assert call(bits=5) == qg.QG_ERR_UNSUPPORTED
    assert call(bs=48) == qg.QG_ERR_UNSUPPORTED
    assert call(K=250, bs=32) == qg.QG_ERR_INVALID_ARG  # K % block_size
    assert call(zp=None) == qg.QG_ERR_INVALID_ARG
    assert call(ws=None, wsb=0) == qg.QG_ERR_WORKSPACE_TOO_SMALL
    assert call(M=0) == qg.QG_OK
    assert L.qgemm_nbits_packed_zp_workspace_bytes(0, 1, 64, 256, 4, 48) == 0
    assert L.qgemm_nbits_packed_zp_workspace_bytes(0, 1, 64, 256, 5, 64) == 0
