"""GPU parity of the GEMM / GEMV entry points against the CPU oracle.

Bars (stated by the method's target): dequantization bit-exact; matmul
outputs within max relative L2 error 1e-4 (fp32 activations, fp32 output) or
5e-3 (fp16 / bf16 activations or 16-bit output) of the oracle's unrounded
fp64 result; 129 repeated calls bit-identical.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import BF16, F16, F32, act_tensor, dev, nbits_case, oracle_nbits, sample_rows, to64, tol_for, torch, \
    y_tensor

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


def _rand_nbits(seed, M, N, K, bits, bs, a_dtype, zp_mode):
    g = WL.rng(seed)
    d = dict(M=M, N=N, K=K, bits=bits, block_size=bs, a_dtype=a_dtype)
    d["W"] = WL.packed_codes(g, N, K, bits)
    d["scales"] = WL.fp16_uniform(g, (N, K // bs), 0.005, 0.05)
    d["zero_points"] = WL.fp16_uniform_int(g, (N, K // bs), 0, 2 ** bits - 1) if zp_mode == "tensor" else None
    d["uniform_zp"] = 1.5 if zp_mode == "uniform" else None
    d["A"] = WL.activations(g, M, K, a_dtype)
    return d


def _run_nbits(qg, d, y_dtype=F32, use_uniform=True):
    t = nbits_case(d)
    Y = y_tensor(d["M"], d["N"], y_dtype)
    if use_uniform and d.get("uniform_zp") is not None:
        qg.qgemm_nbits_uniform_zp(t["A"], t["W"], t["scales"], d["uniform_zp"], Y, bits=d["bits"],
                                  block_size=d["block_size"])
    else:
        qg.qgemm_nbits(t["A"], t["W"], t["scales"], t["zero_points"], Y, bits=d["bits"], block_size=d["block_size"])
    torch().cuda.synchronize()
    return Y


# --------------------------------------------------------------- dequant export
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("bs", [32, 64, 128, 256])
@pytest.mark.parametrize("zp_mode", ["tensor", "none", "uniform"])
def test_dequant_nbits_bit_exact(qg, bits, bs, zp_mode):
    d = _rand_nbits(3, 1, 37, 1024, bits, bs, F32, zp_mode)
    t = nbits_case(d)
    out = torch().full((37, 1024), float("nan"), device="cuda")
    if zp_mode == "uniform":
        qg.qg_dequant_nbits_uniform_zp(t["W"], t["scales"], 1.5, out, bits=bits, block_size=bs)
        ref = O.dequant_nbits(d["W"], d["scales"], None, N=37, K=1024, bits=bits, block_size=bs, uniform_zp=1.5)
    else:
        qg.qg_dequant_nbits(t["W"], t["scales"], t["zero_points"], out, bits=bits, block_size=bs)
        ref = O.dequant_nbits(d["W"], d["scales"], d["zero_points"], N=37, K=1024, bits=bits, block_size=bs)
    assert np.array_equal(out.cpu().numpy(), ref)


@pytest.mark.parametrize("bs", [32, 64, 128, 256])
def test_dequant_codebook_bit_exact(qg, bs):
    d = WL.nf4((41, 768), 1, F16)
    g = WL.rng(5)
    absmax = WL.f32_uniform(g, (41, 768 // bs), 0.02, 0.1)
    out = torch().full((41, 768), float("nan"), device="cuda")
    qg.qg_dequant_codebook4(dev(d["W"]), dev(d["codebook"]), dev(absmax), out, block_size=bs)
    ref = O.dequant_codebook4(d["W"], d["codebook"], absmax, N=41, K=768, block_size=bs)
    assert np.array_equal(out.cpu().numpy(), ref)


# ------------------------------------------------------------------ nbits GEMV
NBITS_CASES = [
    # (M, N, K, bits, bs, a_dtype, zp_mode, y_dtype)
    (1, 301, 1536, 2, 64, F32, "uniform", F32),
    (1, 301, 1536, 2, 64, F32, "tensor", F32),
    (1, 301, 1536, 2, 64, F32, "none", F32),
    (1, 130, 1056, 2, 32, F32, "tensor", F32),     # row bytes not a multiple of 16; ragged slice
    (1, 257, 2048, 2, 32, F32, "uniform", F32),    # 64 codes per lane span two blocks
    (1, 200, 4096, 2, 128, F32, "tensor", F32),
    (1, 64, 1024, 2, 256, F32, "uniform", F32),
    (2, 301, 1536, 2, 64, F32, "uniform", F32),
    (3, 150, 1536, 2, 64, F32, "tensor", F32),
    (4, 301, 5120, 2, 64, F32, "uniform", F32),
    (5, 97, 1536, 2, 64, F32, "tensor", F32),
    (8, 97, 1536, 2, 64, F32, "uniform", F32),
    (1, 301, 1536, 4, 64, F32, "tensor", F32),
    (1, 301, 2880, 4, 32, F32, "none", F32),
    (1, 129, 1024, 4, 128, F32, "uniform", F32),
    (2, 301, 1536, 4, 64, F32, "tensor", F32),
    (4, 301, 1536, 4, 64, F32, "tensor", F32),
    (7, 61, 1024, 4, 256, F32, "none", F32),
    (1, 301, 1536, 2, 64, F16, "uniform", F32),
    (1, 301, 1536, 2, 64, BF16, "uniform", F16),
    (4, 301, 1536, 4, 64, BF16, "tensor", BF16),
    (1, 301, 1536, 4, 64, F32, "tensor", F16),
    (4, 70, 8192, 2, 64, F32, "uniform", F32),     # long K: split across CTAs
    (4, 33, 17920, 2, 64, F32, "tensor", F32),     # long K, split-K with a ragged last split
    (12, 50, 1536, 2, 64, F32, "uniform", F32),    # fp32 activations beyond 8 rows
    (1, 40000, 512, 2, 64, F32, "uniform", F32),   # short K, many rows: more row groups than ring stages
    (1, 301, 1536, 3, 64, F32, "tensor", F32),     # 3-bit codes (hip-ep #1318 kernel test table, Wu3 leaves)
    (1, 257, 2048, 3, 32, F32, "uniform", F32),    # 64 codes per lane span two 32-blocks
    (1, 200, 4096, 3, 128, F32, "none", F32),
    (1, 130, 1056, 3, 32, F32, "tensor", F32),     # K % 64 != 0: 12-byte lane groups
    (2, 150, 1024, 3, 256, F32, "uniform", F32),
    (4, 301, 1536, 3, 64, F32, "tensor", F32),     # two 2-row launches
    (5, 33, 17920, 3, 64, F32, "tensor", F32),     # long K: split across CTAs
    (1, 301, 1536, 3, 64, F16, "uniform", F32),
    (16, 300, 2048, 3, 64, F16, "tensor", F32),    # M >= 9 with 16-bit activations stays on SIMT for u3
    (1, 301, 1536, 8, 64, F32, "tensor", F32),     # 8-bit codes (hip-ep #1318 kernel test table, Wi8 leaves)
    (1, 257, 2048, 8, 32, F32, "uniform", F32),
    (1, 200, 4096, 8, 128, F32, "none", F32),
    (2, 150, 1024, 8, 256, F32, "uniform", F32),
    (4, 301, 1536, 8, 64, F32, "tensor", F32),
    (1, 301, 1536, 8, 64, F16, "uniform", F32),
    (3, 97, 5120, 8, 64, BF16, "tensor", BF16),
    (1, 30000, 256, 4, 64, F32, "tensor", F32),
]


@pytest.mark.parametrize("case", NBITS_CASES, ids=lambda c: "M%d_N%d_K%d_u%d_bs%d_a%d_%s_y%d" % c)
def test_qgemm_nbits_parity(qg, case):
    M, N, K, bits, bs, ad, zpm, yd = case
    d = _rand_nbits(7, M, N, K, bits, bs, ad, zpm)
    Y = _run_nbits(qg, d, yd)
    ref = oracle_nbits(d)
    err = O.max_rel_l2(to64(Y), ref)
    assert err <= tol_for(ad, yd), err


@pytest.mark.parametrize("scale_exp", [110, -110])
def test_extreme_activation_magnitudes(qg, scale_exp):
    """Activations near the ends of the fp32 range in part of K (the kernel
    normalises each lane's slice by a power of two; slices past 2^104 take the
    rare post-scaling path) against the oracle."""
    M, N, K, bits, bs = 1, 301, 5120, 2, 64
    d = _rand_nbits(13, M, N, K, bits, bs, F32, "uniform")
    A = d["A"].astype(np.float64)
    A[:, 1024:2048] *= 2.0 ** scale_exp
    d["A"] = A.astype(np.float32)
    Y = _run_nbits(qg, d, F32)
    assert np.all(np.isfinite(Y.cpu().numpy()))
    assert O.max_rel_l2(to64(Y), oracle_nbits(d)) <= 1e-4


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_onehot_recovers_dequantized_column_exactly(qg, bits):
    N, K, bs = 96, 1024, 64
    d = _rand_nbits(9, 1, N, K, bits, bs, F32, "tensor")
    deq = O.dequant_nbits(d["W"], d["scales"], d["zero_points"], N=N, K=K, bits=bits, block_size=bs)
    for k in (0, 1, 15, 16, 511, 777, K - 1):
        d["A"] = np.zeros((1, K), np.float32)
        d["A"][0, k] = 1.0
        Y = _run_nbits(qg, d, F32)
        assert np.array_equal(Y.cpu().numpy()[0], deq[:, k]), k


@pytest.mark.parametrize("bits,zpv", [(2, 1.5), (3, 3.5), (4, 7.0), (8, 127.5)])
def test_uniform_zp_matches_full_tensor_bitwise(qg, bits, zpv):
    d = _rand_nbits(11, 4, 333, 2048, bits, 64, F32, "uniform")
    d["uniform_zp"] = zpv
    Yu = _run_nbits(qg, d, F32, use_uniform=True)
    d2 = dict(d)
    d2["zero_points"] = WL.fp16_const((333, 2048 // 64), zpv)
    d2["uniform_zp"] = None
    Yt = _run_nbits(qg, d2, F32, use_uniform=False)
    assert torch().equal(Yu, Yt)
    assert O.max_rel_l2(to64(Yu), oracle_nbits(d)) <= 1e-4


def test_fp16_uniform_value_detection(qg):
    t = torch()
    z = t.full((5120, 80), 1.5, dtype=t.float16, device="cuda")
    assert qg.qg_fp16_uniform_value(z) == (True, 1.5)
    z[4000, 7] = 2.5
    assert qg.qg_fp16_uniform_value(z) == (False, None)
    zz = t.zeros(1001, dtype=t.float16, device="cuda")
    zz[1000] = -0.0
    assert qg.qg_fp16_uniform_value(zz) == (False, None)
    nan = t.full((64,), float("nan"), dtype=t.float16, device="cuda")
    assert qg.qg_fp16_uniform_value(nan) == (False, None)
    odd = t.full((3,), -3.0, dtype=t.float16, device="cuda")
    assert qg.qg_fp16_uniform_value(odd) == (True, -3.0)
    # agrees with the oracle on a random tensor and on a uniform one
    for arr in (WL.fp16_uniform_int(WL.rng(2), (100, 9), 0, 1), WL.fp16_const((77,), 0.25)):
        assert qg.qg_fp16_uniform_value(dev(arr, t.float16)) == O.fp16_uniform_value(arr)


# -------------------------------------------------------------- codebook GEMM
CODEBOOK_CASES = [
    (1, 301, 1536, 64, F16), (1, 301, 1536, 64, BF16), (2, 130, 1024, 32, BF16), (4, 301, 2048, 128, F16),
    (8, 97, 1536, 64, BF16), (16, 64, 1024, 64, F16), (1, 200, 1536, 64, F32), (4, 90, 8192, 64, BF16),
]


@pytest.mark.parametrize("case", CODEBOOK_CASES, ids=lambda c: "M%d_N%d_K%d_bs%d_a%d" % c)
def test_qgemm_codebook4_parity(qg, case):
    M, N, K, bs, ad = case
    d = WL.nf4((N, K), M, ad, seed=13)
    if bs != 64:
        d["absmax"] = WL.f32_uniform(WL.rng(14), (N, K // bs), 0.02, 0.1)
    Y = y_tensor(M, N, ad)
    qg.qgemm_codebook4(act_tensor(d["A"], ad), dev(d["W"]), dev(d["codebook"]), dev(d["absmax"]), Y, block_size=bs)
    torch().cuda.synchronize()
    ref = O.qgemm_codebook4(d["A"], d["W"], d["codebook"], d["absmax"], M=M, N=N, K=K, block_size=bs, a_dtype=ad)
    assert O.max_rel_l2(to64(Y), ref) <= tol_for(ad, ad)


# ------------------------------------------------------------ determinism
# Every configuration repeats bit-identically: 129 calls on the same inputs,
# each compared with the first, the output refilled with NaN before every call
# (hip-ep #1328, "Test plan": 129 calls, a distinct shape per process).
REPEAT_CASES = ["tiny_u4", "phi4_qkv_M1", "phi4_lm_head_M4", "split_k_M4", "nf4_simt_M1", "nf4_simt_M4",
                "nf4_tc_M16", "nf4_tc_M64", "prefill_gate_up", "prefill_down",
                # the tensor-pipe GEMV's 16-row tiles (down, long K), eight 16-bit activation rows,
                # and fp32 activations at M = 64 (split-precision tensor cores)
                "phi4_down_M1", "phi4_qkv_M8_f16", "phi4_gate_up_M64_f32"]


def _repeat_case(qg, which):
    """(output shape and dtype, call(out)) for one repeat case."""
    if which.startswith("nf4"):
        M = int(which.rsplit("_M", 1)[1])
        ad = BF16 if M in (1, 16) else F16
        shape = {1: (14336, 4096), 4: (4096, 14336), 16: (4096, 4096), 64: (14336, 4096)}[M]
        d = WL.nf4(shape, M, ad, seed=M)
        A, W, C, AM = act_tensor(d["A"], ad), dev(d["W"]), dev(d["codebook"]), dev(d["absmax"])
        return (M, d["N"], ad), lambda out: qg.qgemm_codebook4(A, W, C, AM, out, block_size=64)
    if which == "tiny_u4":
        d = WL.tiny_u4()
    elif which == "phi4_qkv_M1":
        d = WL.phi4_u2("qkv", M=1)
    elif which == "phi4_lm_head_M4":
        d = WL.phi4_u2("lm_head", M=4)
    elif which == "split_k_M4":
        d = _rand_nbits(17, 4, 70, 8192, 2, 64, F32, "uniform")
    elif which == "phi4_down_M1":
        d = WL.phi4_u2("down", M=1)
    elif which == "phi4_qkv_M8_f16":
        N, K = WL.PHI4_SHAPES["qkv"]
        d = _rand_nbits(19, 8, N, K, 2, 64, F16, "tensor")
    elif which == "phi4_gate_up_M64_f32":
        d = WL.phi4_u2("gate_up", M=64)
    else:
        d = WL.prefill_u2(which.split("_", 1)[1])
    t = nbits_case(d)

    def call(out):
        if d.get("uniform_zp") is not None:
            qg.qgemm_nbits_uniform_zp(t["A"], t["W"], t["scales"], d["uniform_zp"], out, bits=d["bits"],
                                      block_size=d["block_size"])
        else:
            qg.qgemm_nbits(t["A"], t["W"], t["scales"], t["zero_points"], out, bits=d["bits"],
                           block_size=d["block_size"])

    return (d["M"], d["N"], F32), call


@pytest.mark.parametrize("which", REPEAT_CASES)
def test_129_calls_bit_identical(qg, which):
    (M, N, yd), call = _repeat_case(qg, which)
    Y0 = y_tensor(M, N, yd)
    Y = y_tensor(M, N, yd)
    call(Y0)
    torch().cuda.synchronize()
    assert not torch().isnan(Y0).any()
    for i in range(128):
        Y.fill_(float("nan"))
        call(Y)
        assert torch().equal(Y, Y0), "call %d differs from call 0" % (i + 1)
    assert qg.qg_read_device_fault() == 0


# --------------------------------------------------------- workloads, full size
def test_tiny_u4_full(qg):
    d = WL.tiny_u4()
    Y = _run_nbits(qg, d, F32)
    assert O.max_rel_l2(to64(Y), oracle_nbits(d)) <= 1e-4


@pytest.mark.parametrize("shape", list(WL.PHI4_SHAPES))
@pytest.mark.parametrize("M", [1, 4])
def test_phi4_u2_decode_sampled_rows(qg, shape, M):
    d = WL.phi4_u2(shape, M=M)
    Y = _run_nbits(qg, d, F32)
    rows = sample_rows(d["N"], 48)
    ref = oracle_nbits(d, rows=rows)
    assert O.max_rel_l2(to64(Y)[:, rows], ref) <= 1e-4


@pytest.mark.parametrize("shape", list(WL.NF4_SHAPES))
@pytest.mark.parametrize("M", [1, 4, 16, 64])
@pytest.mark.parametrize("ad", [BF16, F16])
def test_nf4_sampled_rows(qg, shape, M, ad):
    d = WL.nf4(shape, M, ad)
    Y = y_tensor(M, d["N"], ad)
    qg.qgemm_codebook4(act_tensor(d["A"], ad), dev(d["W"]), dev(d["codebook"]), dev(d["absmax"]), Y, block_size=64)
    torch().cuda.synchronize()
    rows = sample_rows(d["N"], 24)
    ref = O.qgemm_codebook4(d["A"], d["W"], d["codebook"], d["absmax"], M=M, N=d["N"], K=d["K"], block_size=64,
                            a_dtype=ad, rows=rows)
    assert O.max_rel_l2(to64(Y)[:, rows], ref) <= 5e-3


@pytest.mark.parametrize("shape", list(WL.PREFILL_SHAPES))
def test_prefill_u2_sampled(qg, shape):
    d = WL.prefill_u2(shape)
    Y = _run_nbits(qg, d, F32)
    g = np.random.default_rng(3)
    mrows = np.sort(g.choice(d["M"], size=16, replace=False))
    rows = sample_rows(d["N"], 16)
    sub = dict(d)
    sub["A"] = d["A"][mrows]
    sub["M"] = len(mrows)
    ref = oracle_nbits(sub, rows=rows)
    assert O.max_rel_l2(to64(Y)[mrows][:, rows], ref) <= 5e-3
