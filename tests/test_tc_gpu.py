"""GPU parity of the tensor-core path (M >= 9, fp16 / bf16 activations).

The weight is rounded to the activation's 16-bit type before the MMA, so the
bar is 5e-3 max relative L2 against the oracle's exact fp64 result.  One-hot
tests pin the operand layout and its rounding exactly: with A = e_k every
output is one dequantized weight rounded once to fp16 (fp16 activations) or
to bf16 (bf16 activations).
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import BF16, F16, F32, act_tensor, dev, nbits_case, oracle_nbits, sample_rows, to64, torch, y_tensor

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


def _rand(seed, M, N, K, bits, bs, a_dtype, zp_mode):
    g = WL.rng(seed)
    d = dict(M=M, N=N, K=K, bits=bits, block_size=bs, a_dtype=a_dtype)
    d["W"] = WL.packed_codes(g, N, K, bits)
    d["scales"] = WL.fp16_uniform(g, (N, K // bs), 0.005, 0.05)
    d["zero_points"] = WL.fp16_uniform_int(g, (N, K // bs), 0, 2 ** bits - 1) if zp_mode == "tensor" else None
    d["uniform_zp"] = 1.5 if zp_mode == "uniform" else None
    d["A"] = WL.activations(g, M, K, a_dtype)
    return d


def _run(qg, d, y_dtype):
    t = nbits_case(d)
    Y = y_tensor(d["M"], d["N"], y_dtype)
    if d.get("uniform_zp") is not None:
        qg.qgemm_nbits_uniform_zp(t["A"], t["W"], t["scales"], d["uniform_zp"], Y, bits=d["bits"],
                                  block_size=d["block_size"])
    else:
        qg.qgemm_nbits(t["A"], t["W"], t["scales"], t["zero_points"], Y, bits=d["bits"], block_size=d["block_size"])
    torch().cuda.synchronize()
    return Y


TC_CASES = [
    # (M, N, K, bits, bs, a_dtype, zp_mode, y_dtype)
    (16, 256, 1024, 2, 64, F16, "uniform", F32),
    (9, 200, 1024, 2, 64, F16, "uniform", F32),
    (130, 333, 1536, 2, 64, F16, "tensor", F32),
    (300, 520, 2048, 2, 128, BF16, "uniform", F32),
    (64, 1000, 4096, 4, 64, F16, "tensor", F32),
    (33, 77, 512, 4, 32, BF16, "none", BF16),
    (128, 384, 4096, 4, 256, F16, "none", F16),
    (16, 96, 8192, 2, 64, F16, "uniform", F32),     # few tiles, long K: split-K
    (260, 1024, 1536, 2, 64, BF16, "tensor", F32),
    (16, 256, 512, 2, 64, F16, "tensor", F32),      # 8 parameter columns: narrower than one parameter box
    (40, 300, 2560, 4, 32, F16, "tensor", F32),     # 40 K steps: code super-stages of 2 steps for 4-bit codes
    (64, 300, 2048, 8, 64, F16, "tensor", F32),     # 8-bit codes: one K step per code super-stage
    (130, 256, 1024, 8, 128, BF16, "uniform", F32),
    (300, 520, 4096, 8, 256, F16, "none", F16),
    # K / bs not a multiple of 8: parameter rows of 180 / 40 / 12 bytes, copied in 4-byte pieces
    (64, 300, 2880, 4, 32, F16, "tensor", F32),
    (300, 520, 2880, 4, 32, BF16, "none", F16),
    (16, 96, 640, 2, 32, F16, "tensor", F32),
    (40, 200, 768, 8, 128, BF16, "uniform", BF16),
    (16, 100, 2080, 4, 32, F16, "tensor", F32),    # 65 blocks (odd): stays on the SIMT path
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: "M%d_N%d_K%d_u%d_bs%d_a%d_%s_y%d" % c)
def test_tc_nbits_parity(qg, case):
    M, N, K, bits, bs, ad, zpm, yd = case
    d = _rand(31, M, N, K, bits, bs, ad, zpm)
    Y = _run(qg, d, yd)
    assert O.max_rel_l2(to64(Y), oracle_nbits(d)) <= 5e-3


@pytest.mark.parametrize("case", [
    (300, 19968, 1024, 2, 64, F16, "uniform", F32),   # 156 tiles of 256 x 256: a full wave plus a K-split tail
    (512, 9984, 2048, 4, 128, BF16, "tensor", F32),   # 78 tiles of 256 x 256 (or 156 of 256 x 128)
])
def test_tc_split_tail_sampled(qg, case):
    """Shapes whose tiles do not fill whole waves: the tiles left over run split
    along K and are summed afterwards; checked on sampled weight rows."""
    M, N, K, bits, bs, ad, zpm, yd = case
    d = _rand(43, M, N, K, bits, bs, ad, zpm)
    Y = _run(qg, d, yd)
    rows = sample_rows(N, 48, seed=3)
    rows = np.unique(np.concatenate([rows, np.arange(N - 300, N, 37)]))  # the last tiles are the split ones
    got = to64(Y)[:, rows]
    assert O.max_rel_l2(got, oracle_nbits(d, rows=rows)) <= 5e-3


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_tc_onehot_layout_exact(qg, bits):
    """A = e_k for 16 rows: Y[i, n] = fp16(w[n, k_i]) exactly (zero point 1.5 and
    power-of-two-free fp16 scales make (q - zp) exact, so the only rounding is
    the single fp16 rounding of the weight)."""
    t = torch()
    M, N, K, bs = 16, 300, 2048, 64
    d = _rand(5, M, N, K, bits, bs, F16, "uniform")
    ks = np.array([0, 1, 7, 8, 63, 64, 65, 127, 511, 777, 1024, 1500, 1999, 2040, 2046, 2047])
    A = np.zeros((M, K), np.float16)
    A[np.arange(M), ks] = 1.0
    d["A"] = A.view(np.uint16)
    Y = _run(qg, d, F32)
    deq = O.dequant_nbits(d["W"], d["scales"], None, N=N, K=K, bits=bits, block_size=bs, uniform_zp=1.5)
    expect = deq[:, ks].T.astype(np.float16).astype(np.float32)
    assert np.array_equal(Y.cpu().numpy(), expect)


def _bf16_rn(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 (round to nearest even, torch's conversion) -> float32."""
    b = WL.bf16_bits_from_f32(np.asarray(x, np.float32)).astype(np.uint32) << 16
    return b.view(np.float32)


def _onehot_bf16(M, K, ks):
    A = np.zeros((M, K), np.float32)
    A[np.arange(M), ks] = 1.0
    return WL.bf16_bits_from_f32(A)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("zp_mode", ["uniform", "tensor", "none"])
def test_tc_onehot_layout_exact_bf16(qg, bits, zp_mode):
    """bf16 activations, A = e_k for 16 rows: Y[i, n] = bf16(w[n, k_i]) exactly,
    where w is the oracle's fp32 dequantized weight -- the tensor-core operand is
    one round-to-nearest of that fp32 value to bf16 (no fp16 step in between)."""
    M, N, K, bs = 16, 300, 2048, 64
    d = _rand(6, M, N, K, bits, bs, BF16, zp_mode)
    ks = np.array([0, 1, 7, 8, 63, 64, 65, 127, 511, 777, 1024, 1500, 1999, 2040, 2046, 2047])
    d["A"] = _onehot_bf16(M, K, ks)
    Y = _run(qg, d, F32)
    if zp_mode == "uniform":
        deq = O.dequant_nbits(d["W"], d["scales"], None, N=N, K=K, bits=bits, block_size=bs, uniform_zp=1.5)
    else:
        deq = O.dequant_nbits(d["W"], d["scales"], d["zero_points"], N=N, K=K, bits=bits, block_size=bs)
    expect = _bf16_rn(deq[:, ks].T)
    assert np.array_equal(Y.cpu().numpy(), expect)


@pytest.mark.parametrize("scale_range", [(30000.0, 65000.0), (1e-7, 5e-6)], ids=["beyond_fp16_max", "fp16_subnormal"])
def test_tc_bf16_weight_range(qg, scale_range):
    """bf16 activations with 8-bit codes and scales chosen so that (q - zp) * s
    lies beyond fp16's largest finite value (up to 127 * 65000) or in fp16's
    subnormal range: bf16 represents both, and the operand must be the single
    bf16 rounding of the fp32 weight (one-hot pin), and the GEMM must match the
    oracle at the 16-bit bar."""
    M, N, K, bs, bits = 16, 256, 1024, 64, 8
    g = WL.rng(9)
    d = dict(M=M, N=N, K=K, bits=bits, block_size=bs, a_dtype=BF16)
    d["W"] = WL.packed_codes(g, N, K, bits)
    d["scales"] = WL.fp16_uniform(g, (N, K // bs), *scale_range)
    d["zero_points"] = None
    d["uniform_zp"] = None
    ks = np.linspace(0, K - 1, M).astype(np.int64)
    d["A"] = _onehot_bf16(M, K, ks)
    Y = _run(qg, d, F32)
    deq = O.dequant_nbits(d["W"], d["scales"], None, N=N, K=K, bits=bits, block_size=bs)
    assert np.isfinite(deq).all() and np.abs(deq).max() > (65504.0 if scale_range[0] > 1 else 0.0)
    assert np.array_equal(Y.cpu().numpy(), _bf16_rn(deq[:, ks].T))
    # a dense GEMM on the same weights
    d["A"] = WL.activations(g, M, K, BF16)
    Y = _run(qg, d, F32)
    assert O.max_rel_l2(to64(Y), oracle_nbits(d)) <= 5e-3


@pytest.mark.parametrize("case", [(16, 700, 4096, 64, BF16), (64, 500, 2048, 32, F16), (130, 256, 1024, 128, BF16)])
def test_tc_codebook_parity(qg, case):
    M, N, K, bs, ad = case
    d = WL.nf4((N, K), M, ad, seed=17)
    if bs != 64:
        d["absmax"] = WL.f32_uniform(WL.rng(18), (N, K // bs), 0.02, 0.1)
    Y = y_tensor(M, N, ad)
    qg.qgemm_codebook4(act_tensor(d["A"], ad), dev(d["W"]), dev(d["codebook"]), dev(d["absmax"]), Y, block_size=bs)
    torch().cuda.synchronize()
    ref = O.qgemm_codebook4(d["A"], d["W"], d["codebook"], d["absmax"], M=M, N=N, K=K, block_size=bs, a_dtype=ad)
    assert O.max_rel_l2(to64(Y), ref) <= 5e-3


def test_tc_repeat_bit_identical(qg):
    d = _rand(41, 64, 512, 4096, 2, 64, F16, "uniform")
    Y0 = _run(qg, d, F32)
    for _ in range(20):
        assert torch().equal(_run(qg, d, F32), Y0)
    assert qg.qg_read_device_fault() == 0
