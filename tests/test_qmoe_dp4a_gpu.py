"""GPU parity of the int8-activation (dp4a) QMoE decode against the CPU oracle.

The grid of hip-ep #1328 "Test plan" (fp and dp4a x block size 32 / 64 / 128 x
zero points x bias) for the dp4a variant, u2 codes, both SwiGLU layouts, the
128-expert top-8 2880/2880 workload with 129 bit-identical calls, an
out-of-range expert id and the refusals.  The fc1 output, read back from the
documented workspace layout (g [k][2*inter] fp32 first), is compared with the
oracle's at fp32 rounding level: the quantization of x and the integer dot
products agree exactly, so a single differing int8 code would show.
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


def _run(qg, d, T, interleaved=0, status=None, workspace=None, ids=None):
    t = torch()
    y = t.full((d["hidden"],), float("nan"), dtype=t.float16, device="cuda")
    qg.qmoe_decode_fused_dp4a(T["x"], T["ids"] if ids is None else ids, T["weights"], num_experts=d["num_experts"],
                              fc1_w=T["fc1_w"], fc1_scales=T["fc1_scales"], fc1_zp=T["fc1_zp"],
                              fc1_bias=T["fc1_bias"], fc2_w=T["fc2_w"], fc2_scales=T["fc2_scales"],
                              fc2_zp=T["fc2_zp"], fc2_bias=T["fc2_bias"], bits=d["bits"], block_size=d["block_size"],
                              y=y, swiglu_interleaved=interleaved, status=status, workspace=workspace)
    t.cuda.synchronize()
    return y


def _oracle(d, ids=None, interleaved=0, return_g=False):
    return O.qmoe_decode_dp4a(d["x"], d["ids"] if ids is None else ids, d["weights"], num_experts=d["num_experts"],
                              fc1_w=d["fc1_w"], fc1_scales=d["fc1_scales"], fc1_zp=d["fc1_zp"],
                              fc1_bias=d["fc1_bias"], fc2_w=d["fc2_w"], fc2_scales=d["fc2_scales"],
                              fc2_zp=d["fc2_zp"], fc2_bias=d["fc2_bias"], hidden=d["hidden"], inter=d["inter"],
                              bits=d["bits"], block_size=d["block_size"], swiglu_interleaved=interleaved,
                              return_g=return_g)


def _relerr(y, ref):
    return O.max_rel_l2(y.float().double().cpu().numpy().reshape(1, -1), ref.reshape(1, -1))


@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
def test_dp4a_grid(qg, bs, with_zp, with_bias):
    d = WL.qmoe(num_experts=16, k=4, hidden=512, inter=768, block_size=bs, with_zp=with_zp, with_bias=with_bias,
                seed=bs + 2 * with_zp + with_bias)
    y = _run(qg, d, _dev_case(d))
    ref, bad = _oracle(d)
    assert bad == 0
    assert _relerr(y, ref) <= 5e-3


@pytest.mark.parametrize("bs", [32, 64, 128, 256])
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("hidden,inter", [(512, 768), (288, 160), (2048, 512)])
def test_dp4a_fc1_integer_parts_exact(qg, bs, bits, hidden, inter):
    """One slot: the fc1 output in the workspace equals the oracle's to fp32
    rounding (every int8 code of x and every integer dot identical).  The
    shapes reach every int8 path: the SIMT kernel with 16-lane groups (512),
    with 32-lane groups (2048; u4 with 16-row tiles), and the plain-load
    kernel for the u2 rows of (288, 160), which are not a multiple of 16
    bytes."""
    if hidden % bs or inter % bs:
        pytest.skip("shape not a multiple of the block")
    t = torch()
    d = WL.qmoe(num_experts=4, k=1, hidden=hidden, inter=inter, block_size=bs, with_zp=True, with_bias=True,
                bits=bits, seed=bs + bits)
    T = _dev_case(d)
    ws = t.zeros(qg.qmoe_decode_workspace_bytes(1, hidden, inter), dtype=t.uint8, device="cuda")
    y = _run(qg, d, T, workspace=ws)
    ref, bad, g_ref = _oracle(d, return_g=True)
    assert bad == 0
    g = ws[: 2 * inter * 4].view(t.float32).double().cpu().numpy()
    assert O.max_rel_l2(g.reshape(1, -1), g_ref.reshape(1, -1)) <= 2e-6
    assert _relerr(y, ref) <= 5e-3


def test_dp4a_interleaved_swiglu(qg):
    d = WL.qmoe(num_experts=8, k=3, hidden=256, inter=384, block_size=32, seed=4)
    y = _run(qg, d, _dev_case(d), interleaved=1)
    ref, _ = _oracle(d, interleaved=1)
    assert _relerr(y, ref) <= 5e-3


@pytest.mark.parametrize("with_zp", [False, True])
def test_dp4a_128_experts_top8_2880(qg, with_zp):
    d = WL.qmoe(with_zp=with_zp)
    T = _dev_case(d)
    y0 = _run(qg, d, T)
    ref, bad = _oracle(d)
    assert bad == 0
    assert _relerr(y0, ref) <= 5e-3
    for i in range(128):
        y = _run(qg, d, T)
        assert torch().equal(y, y0), i
    # the int8 decode stays close to the fp decode (activation quantization error only)
    fp_ref, _ = O.qmoe_decode(d["x"], d["ids"], d["weights"], num_experts=d["num_experts"], fc1_w=d["fc1_w"],
                              fc1_scales=d["fc1_scales"], fc1_zp=d["fc1_zp"], fc1_bias=d["fc1_bias"],
                              fc2_w=d["fc2_w"], fc2_scales=d["fc2_scales"], fc2_zp=d["fc2_zp"],
                              fc2_bias=d["fc2_bias"], hidden=d["hidden"], inter=d["inter"], bits=4, block_size=32)
    assert _relerr(y0, fp_ref) <= 5e-2


def test_dp4a_out_of_range_id(qg):
    t = torch()
    d = WL.qmoe(num_experts=8, k=3, hidden=256, inter=256, block_size=64, seed=9)
    T = _dev_case(d)
    bad_ids = d["ids"].copy()
    bad_ids[1] = -3
    status = t.full((1,), -1, dtype=t.int32, device="cuda")
    y = _run(qg, d, T, status=status, ids=dev(bad_ids))
    assert int(status.item()) == 1
    keep = np.array([0, 2])
    d2 = dict(d, ids=d["ids"][keep], weights=d["weights"][keep])
    ref, _ = _oracle(d2)
    assert _relerr(y, ref) <= 5e-3


def test_dp4a_refusals(qg):
    t = torch()
    d = WL.qmoe(num_experts=4, k=2, hidden=256, inter=256, block_size=32, seed=3)
    T = _dev_case(d)
    y = t.empty(256, dtype=t.float16, device="cuda")
    common = dict(num_experts=4, fc1_w=T["fc1_w"], fc1_scales=T["fc1_scales"], fc1_zp=None, fc1_bias=None,
                  fc2_w=T["fc2_w"], fc2_scales=T["fc2_scales"], fc2_zp=None, fc2_bias=None, y=y, raw=True)
    assert qg.qmoe_decode_fused_dp4a(T["x"], T["ids"], T["weights"], bits=4, block_size=16, **common) == \
        qg.QG_ERR_UNSUPPORTED
    assert qg.qmoe_decode_fused_dp4a(T["x"], T["ids"], T["weights"], bits=3, block_size=32, **common) == \
        qg.QG_ERR_UNSUPPORTED
    assert qg.qmoe_decode_fused_dp4a(T["x"], T["ids"], T["weights"], bits=4, block_size=32, **common) == qg.QG_OK
    t.cuda.synchronize()
