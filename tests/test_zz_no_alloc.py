"""qmoe_decode_fused_noalloc: the QMoE decode for callers that cannot allocate.

Some callers cannot allocate device memory at decode time (a runtime that
forbids allocation on its hot path, an embedded host, a C caller without an
allocator), so they cannot pass the workspace qmoe_decode_fused needs.  The
no-allocation entry point uses the library's own fixed device scratch
instead.  This file checks, through the C ABI, that it returns what the
workspace entry point returns on the same inputs, on two calls in a row (the
second call finds the first call's leftovers in the shared scratch), and that
shapes too large for the scratch are refused without touching the output.

It is named so that pytest collects it last, and it must pass both on its own
in a fresh process and after the rest of the suite.
"""
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


def _args(d):
    t = torch()
    h = lambda a: None if a is None else dev(a, t.float16)
    return dict(num_experts=d["num_experts"], fc1_w=dev(d["fc1_w"]), fc1_scales=h(d["fc1_scales"]),
                fc1_zp=h(d["fc1_zp"]), fc1_bias=h(d["fc1_bias"]), fc2_w=dev(d["fc2_w"]),
                fc2_scales=h(d["fc2_scales"]), fc2_zp=h(d["fc2_zp"]), fc2_bias=h(d["fc2_bias"]), bits=d["bits"],
                block_size=d["block_size"]), h(d["x"]), dev(d["ids"]), dev(d["weights"])


@pytest.mark.parametrize("with_zp", [False, True])
def test_noalloc_matches_workspace_entry_point_twice(qg, with_zp):
    t = torch()
    # the 128-expert top-8 2880/2880 block-32 workload, then a smaller one, so the
    # second no-allocation call runs over the first one's leftovers
    cases = [WL.qmoe(with_zp=with_zp), WL.qmoe(num_experts=16, k=4, hidden=512, inter=768, block_size=64,
                                                with_zp=with_zp, seed=5)]
    for d in cases:
        kw, x, ids, w = _args(d)
        y_ref = t.full((d["hidden"],), float("nan"), dtype=t.float16, device="cuda")
        qg.qmoe_decode_fused(x, ids, w, y=y_ref, **kw)
        for _ in range(2):
            y = t.full((d["hidden"],), float("nan"), dtype=t.float16, device="cuda")
            status = t.full((1,), -1, dtype=t.int32, device="cuda")
            qg.qmoe_decode_fused_noalloc(x, ids, w, y=y, status=status, **kw)
            t.cuda.synchronize()
            assert int(status.item()) == 0
            err = O.max_rel_l2(y.double().cpu().numpy().reshape(1, -1), y_ref.double().cpu().numpy().reshape(1, -1))
            assert err <= 5e-3
            assert t.equal(y, y_ref)  # same kernels, same order: identical in fact


def test_noalloc_refuses_shapes_beyond_its_scratch(qg):
    t = torch()
    d = WL.qmoe(num_experts=4, k=4, hidden=256, inter=256, block_size=32, seed=2)
    kw, x, ids, w = _args(d)
    big_k = 64  # 64 slots x (2*16384 + 512) x 4 bytes is far beyond the fixed scratch
    assert qg.qmoe_decode_workspace_bytes(big_k, 512, 16384) > qg.QG_QMOE_NOALLOC_SCRATCH_BYTES
    L = qg.lib()
    import ctypes

    y = t.full((512,), float("nan"), dtype=t.float16, device="cuda")
    p = lambda a: ctypes.c_void_p(a.data_ptr())
    st = L.qmoe_decode_fused_noalloc(p(y), p(ids), p(w), big_k, 4, p(kw["fc1_w"]), p(kw["fc1_scales"]), None, None,
                                     p(kw["fc2_w"]), p(kw["fc2_scales"]), None, None, 512, 16384, 4, 32, 0, p(y),
                                     None, ctypes.c_void_p(t.cuda.current_stream().cuda_stream))
    assert st == qg.QG_ERR_UNSUPPORTED
    t.cuda.synchronize()
    assert bool(y.isnan().all())
