"""GPU parity of the 2-bit MatMulNBits GEMV / small-M GEMM that runs on warp-level
MMAs (block 64, K a multiple of 512; M <= 4 with fp32 activations, M <= 8 with
fp16 / bf16 ones): every column layout of the kernel (activation rows x fp16
terms per block = 1, 2, 4 or 8), every zero-point mode and output type, K from
one span to several ragged K chunks, N with a ragged last tile.

Bars: max relative L2 1e-4 (fp32 activations and output), 5e-3 otherwise; the
one-hot activations recover a dequantized weight column bit for bit; an
all-zero activation row gives exact zeros; activation rows of very different
magnitudes are normalised separately.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import BF16, F16, F32, nbits_case, oracle_nbits, sample_rows, to64, tol_for, torch, y_tensor

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


def _case(seed, M, N, K, ad, zp_mode):
    g = WL.rng(seed)
    d = dict(M=M, N=N, K=K, bits=2, block_size=64, a_dtype=ad)
    d["W"] = WL.packed_codes(g, N, K, 2)
    d["scales"] = WL.fp16_uniform(g, (N, K // 64), 0.01, 0.05)
    d["zero_points"] = WL.fp16_uniform_int(g, (N, K // 64), 0, 3) if zp_mode == "tensor" else None
    d["uniform_zp"] = 1.5 if zp_mode == "uniform" else None
    d["A"] = WL.activations(g, M, K, ad)
    return d


def _run(qg, d, yd):
    t = nbits_case(d)
    Y = y_tensor(d["M"], d["N"], yd)
    if d.get("uniform_zp") is not None:
        qg.qgemm_nbits_uniform_zp(t["A"], t["W"], t["scales"], d["uniform_zp"], Y, bits=2, block_size=64)
    else:
        qg.qgemm_nbits(t["A"], t["W"], t["scales"], t["zero_points"], Y, bits=2, block_size=64)
    torch().cuda.synchronize()
    return Y


CASES = [
    # (M, N, K, a_dtype, zp_mode, y_dtype)
    (1, 333, 512, F32, "uniform", F32),     # one span
    (1, 17, 1536, F32, "tensor", F32),      # two tiles, the second with one row
    (1, 1000, 5120, F32, "none", F32),
    (1, 100, 17920, F32, "uniform", F32),   # 35 spans: three K chunks, the last one ragged
    (1, 64, 8704, F32, "tensor", F32),      # 17 spans: two chunks of 9 and 8
    (2, 301, 2048, F32, "tensor", F32),
    (2, 96, 17920, F32, "uniform", F32),
    (3, 150, 1536, F32, "uniform", F32),    # 3 rows in the 4-row layout
    (4, 301, 5120, F32, "tensor", F32),
    (4, 48, 1024, F32, "none", F16),
    (1, 301, 5120, F16, "uniform", F32),
    (1, 301, 17920, BF16, "tensor", BF16),
    (2, 200, 2048, BF16, "none", F32),
    (4, 130, 5120, F16, "tensor", F16),
    (5, 97, 1536, BF16, "uniform", F32),    # 5 rows in the 8-row layout
    (8, 97, 5120, F16, "uniform", F32),
    (8, 40, 17920, BF16, "tensor", BF16),
    (2, 150, 8704, F32, "tensor", F32),     # 16-row tiles with two activation rows
    (4, 70, 8704, F16, "uniform", F32),
    (8, 200, 5120, BF16, "none", F32),      # eight B columns per block: B fragments in the ring's stages
    (4, 130, 17920, F16, "uniform", F16),   # long K: two launches of two activation rows
    (3, 97, 17920, BF16, "none", F32),      # the same, the second launch with one row
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "M%d_N%d_K%d_a%d_%s_y%d" % c)
def test_mma_gemv_parity(qg, case):
    M, N, K, ad, zpm, yd = case
    d = _case(21, M, N, K, ad, zpm)
    Y = _run(qg, d, yd)
    err = O.max_rel_l2(to64(Y), oracle_nbits(d))
    assert err <= tol_for(ad, yd), err


# Row counts around the dealing of fills over the 152 CTAs of a GB300: whole
# rounds of 2 x 152 fills by tile, then one leftover fill per CTA, then a
# second (32-row tiles of 16-row fills at short K; 16-row tiles of 8-row
# fills at K = 17920).
FILL_CASES = [
    # (M, N, K, a_dtype, zp_mode)
    (1, 4864, 512, F32, "uniform"),    # one whole round, nothing left over
    (1, 4880, 512, F32, "tensor"),     # one leftover fill: a tile holding one fill
    (1, 5128, 512, F32, "uniform"),    # 17 leftover fills, the last one 8 rows
    (1, 7704, 512, F32, "none"),       # more leftover fills than CTAs, the last one partial
    (4, 4880, 1024, F32, "tensor"),    # four activation rows
    (8, 5128, 512, F16, "uniform"),    # eight 16-bit rows
    (1, 2440, 17920, F32, "uniform"),  # 8-row fills: one leftover
    (1, 5120, 17920, F32, "tensor"),   # the down shape: 32 leftover fills
]


@pytest.mark.parametrize("case", FILL_CASES, ids=lambda c: "M%d_N%d_K%d_a%d_%s" % c)
def test_mma_gemv_fill_dealing(qg, case):
    """Every output row, whichever CTA, tile and fill holds it, against the oracle."""
    M, N, K, ad, zpm = case
    d = _case(33, M, N, K, ad, zpm)
    Y = _run(qg, d, F32)
    err = O.max_rel_l2(to64(Y), oracle_nbits(d))
    assert err <= tol_for(ad, F32), err
    assert qg.qg_test_gemv_plan(M if M <= 4 or ad != F32 else 4, N, K, ad, {"none": 0, "tensor": 1, "uniform": 2}[zpm]) is not None


@pytest.mark.parametrize("M", [1, 2, 4])
def test_mma_gemv_onehot_exact(qg, M):
    """A = e_k rows (fp32): each output is the dequantized weight w[n, k] bit for bit."""
    N, K = 70, 1024
    d = _case(5, M, N, K, F32, "tensor")
    deq = O.dequant_nbits(d["W"], d["scales"], d["zero_points"], N=N, K=K, bits=2, block_size=64)
    ks = [0, 1, 7, 8, 9, 15, 16, 63, 64, 255, 256, 511, 512, 777, 1000, 1023][: 4 * M]
    for i in range(0, len(ks), M):
        d["A"] = np.zeros((M, K), np.float32)
        for m in range(M):
            d["A"][m, ks[i + m]] = 1.0
        Y = _run(qg, d, F32).cpu().numpy()
        for m in range(M):
            assert np.array_equal(Y[m], deq[:, ks[i + m]]), (M, ks[i + m])


def test_mma_gemv_zero_row_and_separate_row_scales(qg):
    """Row 0 all zeros (exact zero output), rows 1-3 of magnitudes 2^-60, 1 and 2^70:
    each row is normalised by its own largest magnitude."""
    M, N, K = 4, 200, 2048
    d = _case(8, M, N, K, F32, "uniform")
    A = d["A"].astype(np.float64)
    A[0] = 0.0
    A[1] *= 2.0 ** -60
    A[3] *= 2.0 ** 70
    d["A"] = A.astype(np.float32)
    Y = _run(qg, d, F32)
    y = Y.cpu().numpy()
    assert np.all(y[0] == 0.0)
    ref = oracle_nbits(d)
    for m in (1, 2, 3):
        assert O.max_rel_l2(to64(Y)[m:m + 1], ref[m:m + 1]) <= 1e-4, m


def test_mma_gemv_plans_reach_both_tile_shapes(qg):
    """The shapes above reach both variants of the kernel: 32-row tiles with the
    block parameters staged beside the codes (every phi4-14B K=5120 shape), and
    16-row tiles whose consumer warps copy the block parameters per span (long
    K at M = 1: the down projection, K=17920); a K that is not a multiple of 512
    takes another path."""
    zp = {"none": 0, "tensor": 1, "uniform": 2}
    for s, (N, K) in WL.PHI4_SHAPES.items():
        plan = qg.qg_test_gemv_plan(1, N, K, F32, zp["uniform"])
        assert plan is not None, s
        assert plan["rows_per_tile"] == (16 if K == 17920 else 32), (s, plan)
        assert 1 <= plan["ctas"] <= N and plan["stages"] >= 4, (s, plan)
    plans = [qg.qg_test_gemv_plan(c[0], c[1], c[2], c[3], zp[c[4]]) for c in CASES]
    assert {p["rows_per_tile"] for p in plans if p is not None} == {16, 32}
    # M = 2 with fp32 activations: at K = 8704 (17 spans x 4 B columns, two spans
    # for some warps) only 16-row tiles fit beside the B fragments; at K = 17920
    # nothing does, and two one-row launches serve it
    assert qg.qg_test_gemv_plan(2, 150, 8704, F32, 1)["rows_per_tile"] == 16
    assert qg.qg_test_gemv_plan(2, 96, 17920, F32, 2)["rows_per_tile"] == 16
    assert qg.qg_test_gemv_plan(3, 96, 17920, F32, 2) is None
    assert qg.qg_test_gemv_plan(1, 100, 1536 + 64, F32, 2) is None
    # 16-bit activations, 3-4 rows at K = 17920: four B columns per block leave
    # no room for the ring, two launches of two rows take 16-row tiles; with a
    # zero-point tensor (its staging buffers) two rows miss the fourth stage too
    assert qg.qg_test_gemv_plan(4, 5120, 17920, F16, 2)["rows_per_tile"] == 16
    assert qg.qg_test_gemv_plan(3, 5120, 17920, BF16, 0)["rows_per_tile"] == 16
    assert qg.qg_test_gemv_plan(4, 5120, 17920, F16, 1) is None


@pytest.mark.parametrize("case", [
    (5, 130, 1536, "uniform", F32),    # one group of four rows and one of one
    (9, 97, 5120, "tensor", F32),
    (13, 200, 2048, "none", F16),      # a 16-bit output
    (8, 70, 4608, "tensor", F32),      # two full groups
])
def test_mma_gemv_fp32_row_groups(qg, case):
    """fp32 activations with more than four rows: one launch per group of four
    rows, each against the oracle's fp64 result."""
    M, N, K, zpm, yd = case
    d = _case(23, M, N, K, F32, zpm)
    plan = qg.qg_test_gemv_plan(M, N, K, F32, {"none": 0, "tensor": 1, "uniform": 2}[zpm])
    assert plan is not None
    Y = _run(qg, d, yd)
    err = O.max_rel_l2(to64(Y), oracle_nbits(d))
    assert err <= tol_for(F32, yd), err


@pytest.mark.parametrize("M", [64, 2048])
def test_mma_gemv_fp32_prefill_gate_up_sampled(qg, M):
    """The phi4-14B gate_up projection (35840 x 5120, u2 block 64, zero point
    1.5) with fp32 activations at M = 64 and M = 2048: every activation row,
    on sampled weight rows (the first and last tiles included), at the fp32 bar;
    a second call is bit-identical."""
    d = WL.phi4_u2("gate_up", M=M)
    Y = _run(qg, d, F32)
    rows = np.unique(np.concatenate([sample_rows(d["N"], 40, seed=5), np.arange(d["N"] - 40, d["N"], 7)]))
    got = to64(Y)[:, rows]
    err = O.max_rel_l2(got, oracle_nbits(d, rows=rows))
    assert err <= 1e-4, err
    assert torch().equal(_run(qg, d, F32), Y)


def test_fp32_split_precision_rows_and_workspace(qg):
    """fp32 activations and output with M >= 16 on the tensor cores by split precision: rows of very
    different magnitudes (each scaled by its own power of two), a zero row (exact zeros), a zero-point
    tensor, at the fp32 bar per row; with a workspace too small for the split activations the call takes
    the tensor-pipe GEMV row groups instead and agrees within the same bar."""
    t = torch()
    M, N, K = 40, 300, 2048
    d = _case(29, M, N, K, F32, "tensor")
    A = d["A"].astype(np.float64)
    A[1] = 0.0
    A[2] *= 2.0 ** -60
    A[3] *= 2.0 ** 70
    d["A"] = A.astype(np.float32)
    tv = nbits_case(d)
    ref = oracle_nbits(d)
    Y = y_tensor(M, N, F32)
    qg.qgemm_nbits(tv["A"], tv["W"], tv["scales"], tv["zero_points"], Y, bits=2, block_size=64)
    t.cuda.synchronize()
    y = Y.cpu().numpy()
    assert np.all(y[1] == 0.0)
    for m in [0] + list(range(2, M)):
        assert O.max_rel_l2(to64(Y)[m:m + 1], ref[m:m + 1]) <= 1e-4, m
    small = t.empty(16, dtype=t.uint8, device="cuda")
    Y2 = y_tensor(M, N, F32)
    qg.qgemm_nbits(tv["A"], tv["W"], tv["scales"], tv["zero_points"], Y2, bits=2, block_size=64, workspace=small)
    t.cuda.synchronize()
    assert O.max_rel_l2(to64(Y2), ref) <= 1e-4
    assert qg.qgemm_workspace_bytes(F32, M, N, K, 2, 64) >= 2 * M * K * 2
