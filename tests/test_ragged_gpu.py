"""GPU parity of the ragged expert GEMM (qmoe_ragged_mm) against the CPU oracle.

Row counts per expert cover empty experts, the SIMT range (1..8 rows), one and
several 256-row tensor-core tiles and ragged tails; N is not a multiple of the
weight tile, so the last tile of an expert overlaps the next expert's rows of
the stacked weight tensor and its extra columns must be dropped.  Full-size
128-expert top-8 prompt on sampled (row, column) pairs.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import dev, torch

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


DT = {0: "float32", 1: "float16", 2: "bfloat16"}


def _x(d, x_dtype):
    t = torch()
    X16 = d["X"]
    if x_dtype == 1:
        return dev(X16, t.float16), X16, O.F16
    x32 = X16.view(np.float16).astype(np.float32)
    if x_dtype == 0:
        return dev(x32), x32, O.F32
    xb = t.from_numpy(x32).to(t.bfloat16)
    bits = xb.view(t.int16).numpy().view(np.uint16)
    return xb.cuda(), bits, O.BF16


def _run(qg, d, Xd, y_dtype):
    t = torch()
    T = int(d["offsets"][-1])
    Y = t.full((T, d["N"]), float("nan"), dtype=getattr(t, DT[y_dtype]), device="cuda")
    zp = None if d["zero_points"] is None else dev(d["zero_points"], t.float16)
    qg.qmoe_ragged_mm(Xd, d["offsets"], dev(d["W"]), dev(d["scales"], t.float16), zp, Y, bits=d["bits"],
                      block_size=d["block_size"])
    t.cuda.synchronize()
    return Y


COUNTS = [3, 0, 17, 280, 1, 259, 8, 9, 0, 256]


@pytest.mark.parametrize("bits,bs,x_dtype,y_dtype,zp", [
    (4, 64, 1, 1, False),   # the Xfp16_Wu4_Yfp16 leaf
    (4, 32, 1, 0, True),
    (4, 128, 2, 2, True),
    (2, 64, 1, 0, False),
    (8, 64, 2, 1, True),
    (4, 64, 0, 0, True),    # fp32 activations: every expert on the SIMT path
])
def test_ragged_matches_oracle(qg, bits, bs, x_dtype, y_dtype, zp):
    d = WL.ragged(num_experts=len(COUNTS), N=200, K=512, bits=bits, block_size=bs, with_zp=zp, counts=COUNTS,
                  seed=bits + bs)
    Xd, Xo, od = _x(d, x_dtype)
    Y = _run(qg, d, Xd, y_dtype)
    ref = O.qmoe_ragged_mm(Xo, d["offsets"], d["W"], d["scales"], d["zero_points"], N=d["N"], K=d["K"],
                           bits=bits, block_size=bs, x_dtype=od)
    got = Y.float().double().cpu().numpy()
    tol = 1e-4 if (x_dtype == 0 and y_dtype == 0) else 5e-3
    assert O.max_rel_l2(got, ref) <= tol


def test_ragged_decode_burst_all_simt(qg):
    """A few tokens over many experts: every expert has 0..8 rows."""
    counts = [1, 0, 2, 8, 0, 0, 3, 1, 5, 0, 4, 7]
    d = WL.ragged(num_experts=len(counts), N=96, K=256, bits=4, block_size=32, with_zp=True, counts=counts, seed=3)
    Xd, Xo, od = _x(d, 1)
    Y = _run(qg, d, Xd, 1)
    ref = O.qmoe_ragged_mm(Xo, d["offsets"], d["W"], d["scales"], d["zero_points"], N=96, K=256, bits=4,
                           block_size=32, x_dtype=od)
    assert O.max_rel_l2(Y.float().double().cpu().numpy(), ref) <= 5e-3


def test_ragged_repeat_bit_identical(qg):
    d = WL.ragged(num_experts=len(COUNTS), N=200, K=512, bits=4, block_size=64, counts=COUNTS, seed=8)
    Xd, _, _ = _x(d, 1)
    Y0 = _run(qg, d, Xd, 1)
    for _ in range(8):
        assert torch().equal(_run(qg, d, Xd, 1), Y0)


def test_ragged_refusals_and_empty(qg):
    t = torch()
    d = WL.ragged(num_experts=3, N=64, K=64, bits=4, block_size=32, counts=[2, 0, 3], seed=2)
    Xd, _, _ = _x(d, 1)
    W, S = dev(d["W"]), dev(d["scales"], t.float16)
    Y = t.zeros((5, 64), dtype=t.float16, device="cuda")
    call = lambda off, bits=4, W_=W: qg.qmoe_ragged_mm(Xd, off, W_, S, None, Y, bits=bits, block_size=32, raw=True)
    assert call([0, 2, 2, 5]) == qg.QG_OK
    assert call([1, 2, 2, 5]) == qg.QG_ERR_INVALID_ARG  # must start at 0
    assert call([0, 3, 2, 5]) == qg.QG_ERR_INVALID_ARG  # decreasing
    assert call([0, 2, 2, 5], bits=3) == qg.QG_ERR_UNSUPPORTED
    # u2 with K = 32 and an odd N: one expert's codes are 8 * N bytes, not a multiple of 16
    W2 = t.zeros((3, 63, 8), dtype=t.uint8, device="cuda")
    S2 = t.zeros((3, 63, 1), dtype=t.float16, device="cuda")
    X2 = t.zeros((5, 32), dtype=t.float16, device="cuda")
    Y2 = t.zeros((5, 63), dtype=t.float16, device="cuda")
    assert qg.qmoe_ragged_mm(X2, [0, 2, 2, 5], W2, S2, None, Y2, bits=2, block_size=32, raw=True) == \
        qg.QG_ERR_UNSUPPORTED
    # no rows at all
    Y0 = t.zeros((0, 64), dtype=t.float16, device="cuda")
    X0 = t.zeros((0, 64), dtype=t.float16, device="cuda")
    assert qg.qmoe_ragged_mm(X0, [0, 0, 0, 0], W, S, None, Y0, bits=4, block_size=32, raw=True) == qg.QG_OK
    t.cuda.synchronize()


@pytest.mark.parametrize("N,K", [(1536, 2048), (5760, 2880)])
def test_ragged_prompt_128_experts_top8_full_size(qg, N, K):
    """fc1 of a 128-expert top-8 layer over 2048 tokens (16384 rows), u4 block 32, fp16 in and out: the
    2048 / 768 layer (grouped tensor-core launch) and the 2880-wide one (90 blocks per row: parameter rows
    not a multiple of 16 bytes, so every expert takes the SIMT path); sampled rows of sampled experts
    against the oracle."""
    d = WL.ragged(N=N, K=K)
    Xd, Xo, od = _x(d, 1)
    Y = _run(qg, d, Xd, 1)
    off = d["offsets"]
    g = np.random.default_rng(5)
    cols = np.unique(np.concatenate([[0, d["N"] - 1], g.choice(d["N"], 62, replace=False)])).astype(np.int64)
    for e in sorted(set(g.choice(d["num_experts"], 6, replace=False).tolist()) | {0, d["num_experts"] - 1}):
        a, b = int(off[e]), int(off[e + 1])
        if a == b:
            continue
        rows = sorted({a, b - 1, int(g.integers(a, b))})
        ref = O.qgemm_nbits(Xo[rows], d["W"][e], d["scales"][e], None, M=len(rows), N=d["N"], K=d["K"], bits=4,
                            block_size=32, a_dtype=od, rows=cols)
        got = Y[rows][:, cols].float().double().cpu().numpy()
        assert O.max_rel_l2(got, ref) <= 5e-3, e
    assert not torch().isnan(Y).any()


def _run_dev(qg, d, Xd, y_dtype, extra_rows=0, offsets=None, status=None):
    """The device-offset entry point; X and Y hold extra_rows rows past T (Y's NaN there must stay)."""
    t = torch()
    off = np.asarray(d["offsets"] if offsets is None else offsets, np.int64)
    T = int(d["offsets"][-1])
    if extra_rows:
        Xd = t.cat([Xd, t.zeros((extra_rows, Xd.shape[1]), dtype=Xd.dtype, device="cuda")])
    Y = t.full((T + extra_rows, d["N"]), float("nan"), dtype=getattr(t, DT[y_dtype]), device="cuda")
    zp = None if d["zero_points"] is None else dev(d["zero_points"], t.float16)
    s = qg.qmoe_ragged_mm_device_offsets(Xd, t.from_numpy(off).cuda(), dev(d["W"]), dev(d["scales"], t.float16), zp,
                                         Y, bits=d["bits"], block_size=d["block_size"], status=status, raw=True)
    t.cuda.synchronize()
    return s, Y


@pytest.mark.parametrize("bits,bs,x_dtype,y_dtype,zp", [
    (4, 64, 1, 1, False),
    (4, 32, 2, 0, True),
    (2, 64, 1, 0, False),
    (8, 128, 2, 2, True),
])
def test_ragged_device_offsets_match_oracle(qg, bits, bs, x_dtype, y_dtype, zp):
    """Offsets in device memory: every expert with rows (1..8 included) runs in the grouped tensor-core
    launch, sized for max_rows; rows of Y past offsets[E] stay untouched."""
    t = torch()
    d = WL.ragged(num_experts=len(COUNTS), N=200, K=512, bits=bits, block_size=bs, with_zp=zp, counts=COUNTS,
                  seed=bits + bs + 1)
    Xd, Xo, od = _x(d, x_dtype)
    status = t.zeros(1, dtype=t.int32, device="cuda")
    s, Y = _run_dev(qg, d, Xd, y_dtype, extra_rows=300, status=status)
    assert s == qg.QG_OK
    assert int(status.item()) == 0
    T = int(d["offsets"][-1])
    ref = O.qmoe_ragged_mm(Xo, d["offsets"], d["W"], d["scales"], d["zero_points"], N=d["N"], K=d["K"],
                           bits=bits, block_size=bs, x_dtype=od)
    got = Y[:T].float().double().cpu().numpy()
    assert O.max_rel_l2(got, ref) <= 5e-3
    assert t.isnan(Y[T:].float()).all()
    # repeated calls are bit-identical
    _, Y2 = _run_dev(qg, d, Xd, y_dtype, extra_rows=300)
    assert t.equal(Y2[:T], Y[:T])


def test_ragged_device_offsets_refusals(qg):
    """Offsets the grouped launch refuses (not starting at 0, decreasing, past max_rows) compute nothing
    and set the status word; host-side refusals come before any launch."""
    t = torch()
    d = WL.ragged(num_experts=4, N=96, K=256, bits=4, block_size=32, counts=[5, 20, 0, 7], seed=4)
    Xd, _, _ = _x(d, 1)
    for bad in ([1, 5, 25, 25, 32], [0, 5, 3, 25, 32], [0, 5, 25, 25, 40]):
        status = t.zeros(1, dtype=t.int32, device="cuda")
        s, Y = _run_dev(qg, d, Xd, 1, offsets=bad, status=status)
        assert s == qg.QG_OK
        assert int(status.item()) == 1, bad
        assert t.isnan(Y.float()).all(), bad
    W, S = dev(d["W"]), dev(d["scales"], t.float16)
    off = t.from_numpy(np.asarray(d["offsets"], np.int64)).cuda()
    Y = t.zeros((32, 96), dtype=t.float16, device="cuda")
    x32 = t.zeros((32, 256), dtype=t.float32, device="cuda")
    assert qg.qmoe_ragged_mm_device_offsets(x32, off, W, S, None, Y, bits=4, block_size=32, raw=True) == \
        qg.QG_ERR_UNSUPPORTED  # fp32 activations: not on the grouped launch
    assert qg.qmoe_ragged_mm_device_offsets(Xd, off, W, S, None, Y, bits=3, block_size=32, raw=True) == \
        qg.QG_ERR_UNSUPPORTED
    assert qg.qmoe_ragged_mm_device_offsets_workspace_bytes(0) == 0
    assert qg.qmoe_ragged_mm_device_offsets_workspace_bytes(257) == 0
    t.cuda.synchronize()


def test_ragged_device_offsets_prompt_full_size(qg):
    """The 128-expert top-8 2048 / 768 layer's fc1 over 2048 tokens with device offsets: sampled rows of
    sampled experts against the oracle."""
    d = WL.ragged(N=1536, K=2048)
    Xd, Xo, od = _x(d, 1)
    s, Y = _run_dev(qg, d, Xd, 1)
    assert s == qg.QG_OK
    off = d["offsets"]
    g = np.random.default_rng(7)
    cols = np.unique(np.concatenate([[0, d["N"] - 1], g.choice(d["N"], 62, replace=False)])).astype(np.int64)
    for e in sorted(set(g.choice(d["num_experts"], 6, replace=False).tolist()) | {0, d["num_experts"] - 1}):
        a, b = int(off[e]), int(off[e + 1])
        if a == b:
            continue
        rows = sorted({a, b - 1, int(g.integers(a, b))})
        ref = O.qgemm_nbits(Xo[rows], d["W"][e], d["scales"][e], None, M=len(rows), N=d["N"], K=d["K"], bits=4,
                            block_size=32, a_dtype=od, rows=cols)
        got = Y[rows][:, cols].float().double().cpu().numpy()
        assert O.max_rel_l2(got, ref) <= 5e-3, e
    assert not torch().isnan(Y).any()
