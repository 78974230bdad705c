"""GPU parity of MatMulNBits with packed unsigned-integer zero points.

Zero point b of a row is the bits-wide field at bit b*bits of the row's bit
string, rows padded to whole bytes (the codes' packing rule; the layout is
the library's reading of the hip-ep #1318 kernel test table, whose MatMulNBits
leaves the pages do not spell out).  Checked: parity with the oracle on the
SIMT and tensor-core paths for 2-, 3-, 4- and 8-bit codes, odd field counts
whose fields straddle bytes, bit-identity with qgemm_nbits given the same
integers as an fp16 zero-point tensor, sampled rows of a phi4-sized shape,
repeat calls, a workspace with garbage contents and the refusals.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import act_tensor, dev, to64, torch, y_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    t = torch()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_blockwise_dequant_gb300 as qg
    from gemm_blockwise_dequant_gb300 import build

    build.build()
    qg.lib()
    return qg


def _dev(d):
    t = torch()
    return act_tensor(d["A"], d["a_dtype"]), dev(d["W"]), dev(d["scales"], t.float16), dev(d["zp_packed"])


def _run(qg, d, y_dtype=None, workspace=None):
    A, W, S, Z = _dev(d)
    Y = y_tensor(d["M"], d["N"], d["a_dtype"] if y_dtype is None else y_dtype)
    qg.qgemm_nbits_packed_zp(A, W, S, Z, Y, bits=d["bits"], block_size=d["block_size"], workspace=workspace)
    torch().cuda.synchronize()
    return Y


def _oracle(d, rows=None):
    return O.qgemm_nbits_packed_zp(d["A"], d["W"], d["scales"], d["zp_packed"], M=d["M"], N=d["N"], K=d["K"],
                                   bits=d["bits"], block_size=d["block_size"], a_dtype=d["a_dtype"], rows=rows)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("M,a_dtype", [(1, 0), (4, 0), (1, 1), (16, 1), (64, 2)])
@pytest.mark.parametrize("bs", [32, 128])
def test_packed_zp_parity(qg, bits, M, a_dtype, bs):
    d = WL.packed_zp(300, 1024, M=M, bits=bits, block_size=bs, a_dtype=a_dtype, seed=bits * 7 + M + bs)
    Y = _run(qg, d)
    tol = 1e-4 if a_dtype == 0 else 5e-3
    assert O.max_rel_l2(to64(Y), _oracle(d)) <= tol


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("M,a_dtype", [(1, 0), (16, 1)])
def test_packed_zp_equals_fp16_tensor_path(qg, bits, M, a_dtype):
    """nb = 7 blocks per row (fields straddle bytes for 3 bits, rows end in pad
    bits): the result is bit-identical to qgemm_nbits with the oracle's unpacked
    integers as fp16 zero points."""
    t = torch()
    d = WL.packed_zp(333, 224, M=M, bits=bits, block_size=32, a_dtype=a_dtype, seed=60 + bits)
    Y = _run(qg, d)
    z = O.unpack_zero_points(d["zp_packed"], N=d["N"], nb=7, bits=bits).astype(np.float16).view(np.uint16)
    A, W, S, _ = _dev(d)
    Y2 = y_tensor(d["M"], d["N"], d["a_dtype"])
    qg.qgemm_nbits(A, W, S, dev(z, t.float16), Y2, bits=bits, block_size=32)
    t.cuda.synchronize()
    assert t.equal(Y, Y2)
    tol = 1e-4 if a_dtype == 0 else 5e-3
    assert O.max_rel_l2(to64(Y), _oracle(d)) <= tol


def test_packed_zp_phi4_qkv_u4_sampled_rows_and_repeats(qg):
    """qkv-shaped (7680 x 5120) u4 block 32 decode, M = 1: sampled rows against
    the oracle, then 129 calls bit-identical, also with a garbage workspace."""
    t = torch()
    d = WL.packed_zp(7680, 5120, M=1, bits=4, block_size=32, seed=5)
    Y0 = _run(qg, d)
    rows = np.random.default_rng(0).choice(d["N"], 256, replace=False)
    assert O.max_rel_l2(to64(Y0)[:, rows], _oracle(d, rows=rows)) <= 1e-4
    A, W, S, Z = _dev(d)
    nbytes = qg.qgemm_nbits_packed_zp_workspace_bytes(0, 1, d["N"], d["K"], 4, 32)
    ws = t.full((nbytes,), 0xA5, dtype=t.uint8, device="cuda")
    Y = y_tensor(1, d["N"], 0)
    for i in range(129):
        qg.qgemm_nbits_packed_zp(A, W, S, Z, Y, bits=4, block_size=32, workspace=ws if i % 2 else None)
        t.cuda.synchronize()
        assert t.equal(Y, Y0), i


def test_packed_zp_16bit_output(qg):
    d = WL.packed_zp(200, 512, M=2, bits=4, block_size=64, a_dtype=0, seed=9)
    Y = _run(qg, d, y_dtype=1)
    assert O.max_rel_l2(to64(Y), _oracle(d)) <= 5e-3


def test_packed_zp_refusals(qg):
    t = torch()
    d = WL.packed_zp(64, 256, M=1, bits=4, block_size=64, seed=2)
    A, W, S, Z = _dev(d)
    Y = y_tensor(1, 64, 0)
    f = lambda z=Z, bits=4, ws=None: qg.qgemm_nbits_packed_zp(A, W, S, z, Y, bits=bits, block_size=64, raw=True,
                                                             workspace=ws)
    assert f() == qg.QG_OK
    assert f(z=None) == qg.QG_ERR_INVALID_ARG
    assert f(bits=5) == qg.QG_ERR_UNSUPPORTED
    small = t.zeros(16, dtype=t.uint8, device="cuda")
    assert f(ws=small) == qg.QG_ERR_WORKSPACE_TOO_SMALL
    t.cuda.synchronize()


@pytest.mark.parametrize("bits,bs,K", [(4, 32, 17920), (3, 32, 8960), (2, 128, 17920), (8, 64, 4096)])
def test_packed_zp_long_rows(qg, bits, bs, K):
    """Rows long enough that the SIMT kernel splits K across CTAs: each slice
    reads its blocks' fields out of the whole staged row of packed bytes."""
    d = WL.packed_zp(96, K, M=1, bits=bits, block_size=bs, a_dtype=0, seed=K + bits)
    Y = _run(qg, d)
    assert O.max_rel_l2(to64(Y), _oracle(d)) <= 1e-4


@pytest.mark.parametrize("bits,bs,M,N,K,widened", [
    (4, 32, 1, 640, 1024, False),   # SIMT kernel: packed bytes staged with the codes
    (3, 32, 2, 333, 224, False),
    (8, 128, 4, 256, 2048, False),
    (2, 64, 1, 640, 1024, True),    # tensor-pipe GEMV: an fp16 copy first
    (4, 32, 16, 256, 1024, True),   # tensor cores (16-bit activations)
])
def test_packed_zp_widened_copy_only_off_simt(qg, bits, bs, M, N, K, widened):
    """The fp16 copy of the zero points (the workspace's first N * nb * 2
    bytes) is written only for requests that another kernel than the SIMT
    one takes; a SIMT request leaves those bytes as they were."""
    t = torch()
    a_dtype = 1 if M >= 16 else 0
    d = WL.packed_zp(N, K, M=M, bits=bits, block_size=bs, a_dtype=a_dtype, seed=N + K + bits)
    A, W, S, Z = _dev(d)
    nbytes = qg.qgemm_nbits_packed_zp_workspace_bytes(a_dtype, M, N, K, bits, bs)
    ws = t.full((nbytes,), 0xA5, dtype=t.uint8, device="cuda")
    Y = y_tensor(M, N, a_dtype)
    qg.qgemm_nbits_packed_zp(A, W, S, Z, Y, bits=bits, block_size=bs, workspace=ws)
    t.cuda.synchronize()
    expanded = N * (K // bs) * 2
    untouched = bool((ws[:expanded] == 0xA5).all().item())
    assert untouched != widened
    tol = 1e-4 if a_dtype == 0 else 5e-3
    assert O.max_rel_l2(to64(Y), _oracle(d)) <= tol


@pytest.mark.parametrize("bits,nb_rows", [(4, 32), (3, 7)])
def test_packed_zp_unaligned_pointer(qg, bits, nb_rows):
    """Packed zero points at an odd address (any byte offset is allowed): the
    SIMT kernel copies them byte by byte instead of with bulk copies."""
    t = torch()
    K = 32 * nb_rows
    d = WL.packed_zp(203, K, M=1, bits=bits, block_size=32, a_dtype=0, seed=77 + bits)
    A, W, S, Z = _dev(d)
    buf = t.zeros(Z.numel() + 1, dtype=t.uint8, device="cuda")
    buf[1:] = Z.flatten()
    Zodd = buf[1:].view(Z.shape)
    Y = y_tensor(1, d["N"], 0)
    qg.qgemm_nbits_packed_zp(A, W, S, Zodd, Y, bits=bits, block_size=32)
    t.cuda.synchronize()
    assert O.max_rel_l2(to64(Y), _oracle(d)) <= 1e-4
