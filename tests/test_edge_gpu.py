"""Edge cases and error behaviour of the C ABI on the GPU.

Refused arguments launch nothing (hip-ep #1328, "Test plan"); a pending,
unrelated CUDA error is cleared on entry and not reported as the call's own
(hip-ep #1328, "What"); empty shapes are no-ops and K == 0 writes zeros.
Every failure here is made on the host: nothing faults, traps or hangs.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import F32, dev, nbits_case, oracle_nbits, to64, torch, y_tensor

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


def _case(M=2, N=64, K=512, bits=2, bs=64):
    g = WL.rng(21)
    d = dict(M=M, N=N, K=K, bits=bits, block_size=bs, a_dtype=F32, uniform_zp=None)
    d["W"] = WL.packed_codes(g, N, K, bits)
    d["scales"] = WL.fp16_uniform(g, (N, K // bs), 0.01, 0.05)
    d["zero_points"] = WL.fp16_uniform_int(g, (N, K // bs), 0, 2 ** bits - 1)
    d["A"] = WL.activations(g, M, K, F32)
    return d


def _raw_nbits(qg, A, W, S, Z, Y, M, N, K, bits, bs, ws=None, wsb=0, a_dtype=0, y_dtype=0):
    L = qg.lib()
    p = lambda t: None if t is None else ctypes.c_void_p(t if isinstance(t, int) else t.data_ptr())
    s = ctypes.c_void_p(torch().cuda.current_stream().cuda_stream)
    return L.qgemm_nbits(p(A), a_dtype, p(W), p(S), p(Z), p(Y), y_dtype, M, N, K, bits, bs, p(ws), wsb, s)


def test_refused_arguments_launch_nothing(qg):
    d = _case()
    T = nbits_case(d)
    A, W, S, Z = T["A"], T["W"], T["scales"], T["zero_points"]
    Y = y_tensor(2, 64, F32)
    sentinel = Y.clone()
    M, N, K = 2, 64, 512
    cases = {
        "block 16": (dict(bs=16), qg.QG_ERR_UNSUPPORTED),
        "block 48": (dict(bs=48), qg.QG_ERR_UNSUPPORTED),
        "bits 5": (dict(bits=5), qg.QG_ERR_UNSUPPORTED),
        "bits 16": (dict(bits=16), qg.QG_ERR_UNSUPPORTED),
        "K not a multiple of the block": (dict(K=500, bs=32), qg.QG_ERR_INVALID_ARG),
        "negative M": (dict(M=-1), qg.QG_ERR_INVALID_ARG),
        "null A": (dict(A=None), qg.QG_ERR_INVALID_ARG),
        "null W": (dict(W=None), qg.QG_ERR_INVALID_ARG),
        "null scales": (dict(S=None), qg.QG_ERR_INVALID_ARG),
        "null Y": (dict(Y=None), qg.QG_ERR_INVALID_ARG),
        "misaligned W": (dict(W=W.data_ptr() + 8), qg.QG_ERR_INVALID_ARG),
        "misaligned A": (dict(A=A.data_ptr() + 4), qg.QG_ERR_INVALID_ARG),
        "bad a dtype": (dict(a_dtype=7), qg.QG_ERR_INVALID_ARG),
        "bad y dtype": (dict(y_dtype=-1), qg.QG_ERR_INVALID_ARG),
    }
    for name, (kw, expect) in cases.items():
        args = dict(A=A, W=W, S=S, Z=Z, Y=Y, M=M, N=N, K=K, bits=2, bs=64)
        args.update(kw)
        st = _raw_nbits(qg, **args)
        assert st == expect, (name, st)
    torch().cuda.synchronize()
    assert torch().equal(Y.isnan(), sentinel.isnan())


def test_workspace_too_small_is_refused(qg):
    # a long-K, multi-row shape needs split-K partials in the workspace
    M, N, K = 4, 70, 8192
    need = qg.qgemm_workspace_bytes(0, M, N, K, 2, 64)
    assert need > 0
    d = _case(M, N, K)
    T = nbits_case(d)
    Y = y_tensor(M, N, F32)
    ws = torch().empty(need, dtype=torch().uint8, device="cuda")
    assert _raw_nbits(qg, T["A"], T["W"], T["scales"], None, Y, M, N, K, 2, 64, ws, need - 16) == \
        qg.QG_ERR_WORKSPACE_TOO_SMALL
    assert _raw_nbits(qg, T["A"], T["W"], T["scales"], None, Y, M, N, K, 2, 64, None, 0) == \
        qg.QG_ERR_WORKSPACE_TOO_SMALL
    assert _raw_nbits(qg, T["A"], T["W"], T["scales"], None, Y, M, N, K, 2, 64, ws, need) == qg.QG_OK


def test_empty_shapes(qg):
    t = torch()
    d = _case()
    T = nbits_case(d)
    Y = y_tensor(2, 64, F32)
    assert _raw_nbits(qg, T["A"], T["W"], T["scales"], None, Y, 0, 64, 512, 2, 64) == qg.QG_OK
    assert _raw_nbits(qg, T["A"], T["W"], T["scales"], None, Y, 2, 0, 512, 2, 64) == qg.QG_OK
    assert _raw_nbits(qg, None, None, None, None, None, 0, 0, 512, 2, 64) == qg.QG_OK
    t.cuda.synchronize()
    assert bool(Y.isnan().all())  # untouched
    assert _raw_nbits(qg, T["A"], T["W"], T["scales"], None, Y, 2, 64, 0, 2, 64) == qg.QG_OK
    t.cuda.synchronize()
    assert bool((Y == 0).all())


def _cudart():
    # the library links the shared CUDA runtime, so this is the same instance
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    pytest.skip("libcudart not loadable by name")


def test_first_call_over_a_pending_error_succeeds(qg):
    rt = _cudart()
    rt.cudaMalloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t]
    rt.cudaGetLastError.restype = ctypes.c_int
    rt.cudaPeekAtLastError.restype = ctypes.c_int
    d = _case(1, 300, 1536)
    T = nbits_case(d)
    Y = y_tensor(1, 300, F32)
    p = ctypes.c_void_p()
    assert rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(1 << 60)) != 0  # fails, leaves a pending error
    assert rt.cudaPeekAtLastError() != 0
    st = _raw_nbits(qg, T["A"], T["W"], T["scales"], T["zero_points"], Y, 1, 300, 1536, 2, 64)
    assert st == qg.QG_OK
    torch().cuda.synchronize()
    assert O.max_rel_l2(to64(Y), oracle_nbits(d)) <= 1e-4
    # and the QMoE entry point too
    q = WL.qmoe(num_experts=4, k=2, hidden=256, inter=256, block_size=32, seed=3)
    assert rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(1 << 60)) != 0
    t = torch()
    h = lambda a: None if a is None else dev(a, t.float16)
    y = t.empty(256, dtype=t.float16, device="cuda")
    qg.qmoe_decode_fused(h(q["x"]), dev(q["ids"]), dev(q["weights"]), num_experts=4, fc1_w=dev(q["fc1_w"]),
                         fc1_scales=h(q["fc1_scales"]), fc1_zp=None, fc1_bias=h(q["fc1_bias"]), fc2_w=dev(q["fc2_w"]),
                         fc2_scales=h(q["fc2_scales"]), fc2_zp=None, fc2_bias=h(q["fc2_bias"]), bits=4,
                         block_size=32, y=y)
    t.cuda.synchronize()
    ref, _ = O.qmoe_decode(q["x"], q["ids"], q["weights"], num_experts=4, fc1_w=q["fc1_w"],
                           fc1_scales=q["fc1_scales"], fc1_zp=None, fc1_bias=q["fc1_bias"], fc2_w=q["fc2_w"],
                           fc2_scales=q["fc2_scales"], fc2_zp=None, fc2_bias=q["fc2_bias"], hidden=256, inter=256,
                           bits=4, block_size=32)
    assert O.max_rel_l2(y.double().cpu().numpy().reshape(1, -1), ref.reshape(1, -1)) <= 5e-3


def test_qmoe_refusals(qg):
    t = torch()
    q = WL.qmoe(num_experts=4, k=2, hidden=256, inter=256, block_size=32, seed=3)
    h = lambda a: None if a is None else dev(a, t.float16)
    y = t.full((256,), float("nan"), dtype=t.float16, device="cuda")
    base = dict(num_experts=4, fc1_w=dev(q["fc1_w"]), fc1_scales=h(q["fc1_scales"]), fc1_zp=None,
                fc1_bias=h(q["fc1_bias"]), fc2_w=dev(q["fc2_w"]), fc2_scales=h(q["fc2_scales"]), fc2_zp=None,
                fc2_bias=h(q["fc2_bias"]), bits=4, block_size=32, y=y, raw=True)
    x, ids, w = h(q["x"]), dev(q["ids"]), dev(q["weights"])
    assert qg.qmoe_decode_fused(x, ids, w, **dict(base, block_size=16)) == qg.QG_ERR_UNSUPPORTED
    assert qg.qmoe_decode_fused(x, ids, w, **dict(base, bits=3)) == qg.QG_ERR_UNSUPPORTED
    assert qg.qmoe_decode_fused(x, ids, w, **dict(base, fc1_w=None)) == qg.QG_ERR_INVALID_ARG
    assert qg.qmoe_decode_fused(x, ids, w, **dict(base, swiglu_interleaved=2)) == qg.QG_ERR_INVALID_ARG
    assert qg.qmoe_decode_fused(x, ids, w, **dict(base, workspace=t.empty(16, dtype=t.uint8, device="cuda"))) == \
        qg.QG_ERR_WORKSPACE_TOO_SMALL
    t.cuda.synchronize()
    assert bool(y.isnan().all())


def test_no_device_fault_recorded(qg):
    assert qg.qg_read_device_fault() == 0
