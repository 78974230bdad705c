"""GPU parity of the block-quantized embedding gather against the CPU oracle.

The gather moves bytes only and every dequantized value is computed with the
same fp32 operations on both sides, then rounded to nearest-even into the
output type (numpy's float16 and torch's bfloat16 conversions on the oracle's
side), so outputs are compared bit for bit, NaN positions included.  Covers
the kernel test table's leaves (u4, u8 and fp8 tables with int64 indices and
fp16 output; hip-ep #1318), u2 tables, fp32 / bf16 outputs, every block size,
negative and out-of-range indices, empty inputs, refusals and phi4-14B's
embedding table looked up for a 2048-token prompt.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import dev, torch

pytestmark = pytest.mark.gpu

FMTS = {"u2": O.W_U2, "u4": O.W_U4, "u8": O.W_U8, "e4m3": O.W_E4M3}


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


def _expected_bits(out32: np.ndarray, y: str) -> np.ndarray:
    """The oracle's exact fp32 values rounded (RN-even) to the output type, as bit patterns."""
    t = torch()
    if y == "f32":
        return out32.astype(np.float32).view(np.uint32)
    if y == "f16":
        return out32.astype(np.float16).view(np.uint16)
    return t.from_numpy(out32).to(t.bfloat16).view(t.int16).numpy().view(np.uint16)


def _got_bits(Y, y: str) -> np.ndarray:
    t = torch()
    if y == "f32":
        return Y.cpu().numpy().view(np.uint32)
    return Y.view(t.int16).cpu().numpy().view(np.uint16)


def _isnan_bits(bits, y):
    if y == "f32":
        return np.isnan(bits.view(np.float32))
    if y == "f16":
        return np.isnan(bits.view(np.float16))
    return _bf_isnan(bits)


def _assert_same(got, want, y):
    """Bit-identical outputs; NaN positions must agree (NaN payloads may differ)."""
    nan_w, nan_g = _isnan_bits(want, y), _isnan_bits(got, y)
    assert np.array_equal(nan_w, nan_g)
    diff = np.argwhere((got != want) & ~nan_w)
    assert diff.size == 0, "first mismatches at %s" % diff[:5].tolist()


def _bf_isnan(bits):
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


def _ydt(y):
    t = torch()
    return {"f32": t.float32, "f16": t.float16, "bf16": t.bfloat16}[y]


def _run(qg, d, y, status=None, indices=None):
    t = torch()
    idx = d["indices"] if indices is None else indices
    zp = None if d["zero_points"] is None else dev(d["zero_points"], t.float16)
    Y = t.full((len(idx), d["D"]), float("nan"), dtype=_ydt(y), device="cuda")
    qg.qg_gather_block_quantized(dev(np.asarray(idx, dtype=np.int64)), dev(d["W"]), dev(d["scales"], t.float16), zp,
                                 Y, w_format=d["fmt"], block_size=d["block_size"], status=status)
    t.cuda.synchronize()
    return Y


def _oracle(d, indices=None):
    return O.gather_block_quantized(d["indices"] if indices is None else indices, d["W"], d["scales"],
                                    d["zero_points"], V=d["V"], D=d["D"], fmt=d["fmt"], block_size=d["block_size"])


def _case(fmt, bs, zp, V=300, D=512, n=257, seed=5, nan_patterns=False):
    d = WL.embedding(fmt, V=V, D=D, n=n, block_size=bs, zero_points=zp, seed=seed)
    g = np.random.default_rng(seed + 1)
    # indices from the whole valid range, negative ones included, and repeats
    d["indices"] = g.integers(-V, V, size=n, dtype=np.int64)
    d["indices"][:3] = [0, V - 1, -V]
    if nan_patterns and fmt == O.W_E4M3:
        d["W"][0, :4] = [0x7F, 0xFF, 0x80, 0x00]
        d["indices"][3] = 0
    return d


@pytest.mark.parametrize("fmt", sorted(FMTS))
@pytest.mark.parametrize("bs", [32, 64, 128, 256])
@pytest.mark.parametrize("y", ["f16", "f32", "bf16"])
def test_gather_matches_oracle_bit_for_bit(qg, fmt, bs, y):
    f = FMTS[fmt]
    for zp in ([True, False] if f != O.W_E4M3 else [False]):
        d = _case(f, bs, zp, nan_patterns=True)
        status = torch().full((1,), -1, dtype=torch().int32, device="cuda")
        Y = _run(qg, d, y, status=status)
        out, bad = _oracle(d)
        assert bad == 0 and int(status.item()) == 0
        _assert_same(_got_bits(Y, y), _expected_bits(out, y), y)


@pytest.mark.parametrize("fmt", ["u4", "e4m3"])
def test_out_of_range_indices_give_zero_rows_and_status(qg, fmt):
    f = FMTS[fmt]
    d = _case(f, 64, f != O.W_E4M3, V=100, D=256, n=12)
    idx = np.array([0, 99, -1, -100, 100, -101, 2**40, -(2**62), 7, 7, 50, -50], dtype=np.int64)
    t = torch()
    status = t.full((1,), -1, dtype=t.int32, device="cuda")
    Y = _run(qg, d, "f16", status=status, indices=idx)
    out, bad = _oracle(d, indices=idx)
    assert bad == 4 and int(status.item()) == 1
    _assert_same(_got_bits(Y, "f16"), _expected_bits(out, "f16"), "f16")
    assert not Y[4:8].any()


def test_empty_and_zero_vocab(qg):
    t = torch()
    d = _case(O.W_U4, 32, True, V=64, D=128, n=4)
    status = t.full((1,), -1, dtype=t.int32, device="cuda")
    Y = t.empty((0, 128), dtype=t.float16, device="cuda")
    qg.qg_gather_block_quantized(t.empty(0, dtype=t.int64, device="cuda"), dev(d["W"]),
                                 dev(d["scales"], t.float16), None, Y, w_format=qg.QG_WF_U4, block_size=32,
                                 status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    # a table with no rows: every index is out of range
    Y = t.full((3, 128), float("nan"), dtype=t.float16, device="cuda")
    W0 = t.empty((0, 64), dtype=t.uint8, device="cuda")
    S0 = t.empty((0, 4), dtype=t.float16, device="cuda")
    qg.qg_gather_block_quantized(dev(np.array([0, 1, -1], dtype=np.int64)), W0, S0, None, Y,
                                 w_format=qg.QG_WF_U4, block_size=32, status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 1
    assert not Y.any()


def test_refusals(qg):
    t = torch()
    d = _case(O.W_U4, 32, True, V=64, D=128, n=4)
    idx = dev(d["indices"])
    W = dev(d["W"])
    S = dev(d["scales"], t.float16)
    Z = dev(d["zero_points"], t.float16)
    Y = t.zeros((4, 128), dtype=t.float16, device="cuda")
    L = qg.lib()
    call = lambda **kw: qg.qg_gather_block_quantized(kw.get("idx", idx), kw.get("W", W), kw.get("S", S),
                                                     kw.get("Z", None), kw.get("Y", Y),
                                                     w_format=kw.get("fmt", qg.QG_WF_U4),
                                                     block_size=kw.get("bs", 32), raw=True)
    assert call() == qg.QG_OK
    assert call(bs=16) == qg.QG_ERR_UNSUPPORTED
    assert call(bs=48) == qg.QG_ERR_UNSUPPORTED
    assert call(fmt=7) == qg.QG_ERR_UNSUPPORTED
    assert call(fmt=qg.QG_WF_E4M3, Z=Z) == qg.QG_ERR_INVALID_ARG  # E4M3 has no zero point
    Yodd = t.zeros(4 * 128 + 8, dtype=t.float16, device="cuda")[1:1 + 4 * 128].view(4, 128)
    assert call(Y=Yodd) == qg.QG_ERR_INVALID_ARG
    s = L.qg_gather_block_quantized(idx.data_ptr(), 4, W.data_ptr(), 1, S.data_ptr(), None, 64, 100, 32,
                                    Y.data_ptr(), 1, None, t.cuda.current_stream().cuda_stream)
    assert s == qg.QG_ERR_INVALID_ARG  # D % block_size != 0
    s = L.qg_gather_block_quantized(idx.data_ptr(), 4, W.data_ptr(), 1, S.data_ptr(), None, 64, 128, 32,
                                    Y.data_ptr(), 5, None, t.cuda.current_stream().cuda_stream)
    assert s == qg.QG_ERR_UNSUPPORTED  # output type
    t.cuda.synchronize()


@pytest.mark.parametrize("fmt", ["u4", "u8", "e4m3"])
def test_phi4_embedding_prompt_full_size(qg, fmt):
    """phi4-14B embedding table (100352 x 5120, block 32) looked up for 2048 tokens, fp16 out;
    every output element checked."""
    f = FMTS[fmt]
    d = WL.embedding(f, block_size=32, zero_points=(f != O.W_E4M3))
    Y = _run(qg, d, "f16")
    out, bad = _oracle(d)
    assert bad == 0
    _assert_same(_got_bits(Y, "f16"), _expected_bits(out, "f16"), "f16")
