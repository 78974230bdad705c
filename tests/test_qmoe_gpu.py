"""GPU parity of the fused single-token QMoE decode against the CPU oracle.

Covers the grid of hip-ep #1328 "Test plan" (block 32 / 64 / 128 x zero points
x bias), the 128-expert top-8 2880/2880 workload, 129 bit-identical calls, the
fused decode against the unfused chain of GEMV calls, both SwiGLU layouts and
an out-of-range expert id.
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


def _dev_case(d):
    t = torch()
    h = lambda a: None if a is None else dev(a, t.float16)
    return dict(x=h(d["x"]), ids=dev(d["ids"]), weights=dev(d["weights"]), fc1_w=dev(d["fc1_w"]),
                fc1_scales=h(d["fc1_scales"]), fc1_zp=h(d["fc1_zp"]), fc1_bias=h(d["fc1_bias"]),
                fc2_w=dev(d["fc2_w"]), fc2_scales=h(d["fc2_scales"]), fc2_zp=h(d["fc2_zp"]),
                fc2_bias=h(d["fc2_bias"]))


def _run(qg, d, T, interleaved=0, status=None, workspace=None):
    t = torch()
    y = t.full((d["hidden"],), float("nan"), dtype=t.float16, device="cuda")
    qg.qmoe_decode_fused(T["x"], T["ids"], T["weights"], num_experts=d["num_experts"], fc1_w=T["fc1_w"],
                         fc1_scales=T["fc1_scales"], fc1_zp=T["fc1_zp"], fc1_bias=T["fc1_bias"], fc2_w=T["fc2_w"],
                         fc2_scales=T["fc2_scales"], fc2_zp=T["fc2_zp"], fc2_bias=T["fc2_bias"], bits=d["bits"],
                         block_size=d["block_size"], y=y, swiglu_interleaved=interleaved, status=status,
                         workspace=workspace)
    t.cuda.synchronize()
    return y


def _oracle(d, ids=None, interleaved=0):
    return O.qmoe_decode(d["x"], d["ids"] if ids is None else ids, d["weights"], num_experts=d["num_experts"],
                         fc1_w=d["fc1_w"], fc1_scales=d["fc1_scales"], fc1_zp=d["fc1_zp"], fc1_bias=d["fc1_bias"],
                         fc2_w=d["fc2_w"], fc2_scales=d["fc2_scales"], fc2_zp=d["fc2_zp"], fc2_bias=d["fc2_bias"],
                         hidden=d["hidden"], inter=d["inter"], bits=d["bits"], block_size=d["block_size"],
                         swiglu_interleaved=interleaved)


def _relerr(y, ref):
    return O.max_rel_l2(y.float().double().cpu().numpy().reshape(1, -1), ref.reshape(1, -1))


@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
def test_qmoe_grid(qg, bs, with_zp, with_bias):
    d = WL.qmoe(num_experts=16, k=4, hidden=512, inter=768, block_size=bs, with_zp=with_zp, with_bias=with_bias,
                seed=bs + 2 * with_zp + with_bias)
    y = _run(qg, d, _dev_case(d))
    ref, bad = _oracle(d)
    assert bad == 0
    assert _relerr(y, ref) <= 5e-3


@pytest.mark.parametrize("with_zp", [False, True])
def test_qmoe_128_experts_top8_2880(qg, with_zp):
    d = WL.qmoe(with_zp=with_zp)
    T = _dev_case(d)
    y0 = _run(qg, d, T)
    ref, bad = _oracle(d)
    assert bad == 0
    assert _relerr(y0, ref) <= 5e-3
    # 128 more calls, each bit-identical to the first
    for i in range(128):
        y = _run(qg, d, T)
        assert torch().equal(y, y0), i
    assert qg.qg_read_device_fault() == 0


def test_qmoe_bias_not_16_byte_aligned(qg):
    """Biases that start 2 bytes past a 16-byte boundary take the scalar copy
    into shared memory."""
    t = torch()
    d = WL.qmoe(num_experts=8, k=3, hidden=512, inter=768, block_size=32, with_bias=True, seed=11)
    T = _dev_case(d)
    for key in ("fc1_bias", "fc2_bias"):
        b = T[key]
        buf = t.empty(b.numel() + 8, dtype=t.float16, device="cuda")
        view = buf[1:1 + b.numel()].view(b.shape)
        view.copy_(b)
        assert view.data_ptr() % 16 != 0
        T[key] = view
    y = _run(qg, d, T)
    ref, bad = _oracle(d)
    assert bad == 0
    assert _relerr(y, ref) <= 5e-3


def test_qmoe_interleaved_swiglu(qg):
    d = WL.qmoe(num_experts=8, k=3, hidden=256, inter=384, block_size=32, seed=4)
    y = _run(qg, d, _dev_case(d), interleaved=1)
    ref, _ = _oracle(d, interleaved=1)
    assert _relerr(y, ref) <= 5e-3


def test_qmoe_fused_matches_unfused_chain(qg):
    """The fused decode against the chain of qgemm_nbits GEMVs (fp32 out) with
    bias, SwiGLU and the weighted sum done by torch in fp64."""
    t = torch()
    d = WL.qmoe(num_experts=8, k=4, hidden=512, inter=512, block_size=64, with_zp=True, seed=6)
    T = _dev_case(d)
    y = _run(qg, d, T)
    H, I = d["hidden"], d["inter"]
    acc = t.zeros(H, dtype=t.float64, device="cuda")
    x = T["x"].view(1, H)
    for j, e in enumerate(d["ids"].tolist()):
        g = t.empty(1, 2 * I, device="cuda")
        qg.qgemm_nbits(x, T["fc1_w"][e], T["fc1_scales"][e], T["fc1_zp"][e], g, bits=4, block_size=64)
        g = g.double()[0] + T["fc1_bias"][e].double()
        h = (g[:I] / (1 + t.exp(-g[:I])) * g[I:]).float().view(1, I)
        o = t.empty(1, H, device="cuda")
        qg.qgemm_nbits(h, T["fc2_w"][e], T["fc2_scales"][e], T["fc2_zp"][e], o, bits=4, block_size=64)
        acc += float(d["weights"][j]) * (o.double()[0] + T["fc2_bias"][e].double())
    chain = acc.cpu().numpy()
    assert O.max_rel_l2(y.double().cpu().numpy().reshape(1, -1), chain.reshape(1, -1)) <= 2e-3
    ref, _ = _oracle(d)
    assert O.max_rel_l2(chain.reshape(1, -1), ref.reshape(1, -1)) <= 1e-4


def test_qmoe_out_of_range_id_sets_status_and_adds_nothing(qg):
    t = torch()
    d = WL.qmoe(num_experts=8, k=4, hidden=256, inter=256, block_size=32, seed=8)
    ids = d["ids"].copy()
    ids[2] = 8  # == num_experts: out of range
    d2 = dict(d)
    d2["ids"] = ids
    status = t.full((1,), -1, dtype=t.int32, device="cuda")
    y = _run(qg, d2, _dev_case(d2), status=status)
    assert int(status.item()) == 1
    ref, bad = _oracle(d2)
    assert bad == 1
    assert _relerr(y, ref) <= 5e-3
    status.fill_(-1)
    _run(qg, d, _dev_case(d), status=status)
    assert int(status.item()) == 0


@pytest.mark.parametrize("k", [1, 5, 8])
def test_qmoe_dirty_workspace(qg, k):
    """The workspace needs no initial contents: a workspace full of 0xA5
    bytes gives the same bits as a zeroed one, call after call, and every
    call writes the status."""
    t = torch()
    d = WL.qmoe(num_experts=16, k=k, hidden=1024, inter=512, block_size=64, with_zp=True, with_bias=True, seed=20 + k)
    T = _dev_case(d)
    nbytes = qg.qmoe_decode_workspace_bytes(k, 1024, 512)
    y0 = _run(qg, d, T, workspace=t.zeros(nbytes, dtype=t.uint8, device="cuda"))
    ref, _ = _oracle(d)
    assert _relerr(y0, ref) <= 5e-3
    ws = t.full((nbytes,), 0xA5, dtype=t.uint8, device="cuda")
    status = t.full((1,), -1, dtype=t.int32, device="cuda")
    for i in range(3):
        status.fill_(-1)
        y = _run(qg, d, T, status=status, workspace=ws)
        assert t.equal(y, y0), i
        assert int(status.item()) == 0
