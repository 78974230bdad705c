"""Failure detection on the GPU without a fault: a bounded pipeline wait that
runs out.

Every wait of the library's kernels on a pipeline stage is bounded; one that
gives up records a bit in the device fault word, ends its warp and lets the
CTA finish instead of hanging.  The test hook of include/qgemm_testing.h runs
that wait in a pipeline-shaped kernel whose producer never fills the stage,
with a 200 us bound: the call must return, the word must carry
FAULT_WAIT_FULL, and the context must stay usable (a parity check right after).
"""
import pytest

import oracle as O
import workloads as WL
from gpu_util import F32, nbits_case, oracle_nbits, to64, torch, y_tensor

pytestmark = pytest.mark.gpu

FAULT_WAIT_FULL = 1


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


def test_filled_stage_completes_without_fault(qg):
    t = torch()
    assert qg.qg_read_device_fault() == 0
    out = t.full((3,), -1, dtype=t.int32, device="cuda")
    qg.qg_test_bounded_wait(True, 200, out)
    t.cuda.synchronize()
    assert out.tolist() == [1, 1, 1]
    assert qg.qg_read_device_fault() == 0


@pytest.mark.parametrize("limit_us", [200, 5000])
def test_wait_that_runs_out_is_reported_and_the_context_survives(qg, limit_us):
    t = torch()
    assert qg.qg_read_device_fault() == 0
    out = t.full((3,), -1, dtype=t.int32, device="cuda")
    a, b = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
    a.record()
    qg.qg_test_bounded_wait(False, limit_us, out)
    b.record()
    t.cuda.synchronize()
    assert out.tolist() == [0, 0, 0]                  # every consumer warp gave up
    assert a.elapsed_time(b) * 1e3 >= 0.9 * limit_us  # ... after its bound, not before
    assert qg.qg_read_device_fault() == FAULT_WAIT_FULL
    assert qg.qg_read_device_fault() == 0             # the read cleared the word
    # the context is intact: a GEMV right after matches the oracle
    d = WL.phi4_u2("o", M=1)
    T = nbits_case(d)
    Y = y_tensor(1, d["N"], F32)
    qg.qgemm_nbits_uniform_zp(T["A"], T["W"], T["scales"], 1.5, Y, bits=2, block_size=64)
    t.cuda.synchronize()
    assert O.max_rel_l2(to64(Y), oracle_nbits(d)) <= 1e-4
    assert qg.qg_read_device_fault() == 0


def test_hook_refuses_bad_arguments(qg):
    t = torch()
    out = t.zeros(3, dtype=t.int32, device="cuda")
    assert qg.qg_test_bounded_wait(False, 0, out, raw=True) == qg.QG_ERR_INVALID_ARG
    assert qg.qg_test_bounded_wait(False, 2000001, out, raw=True) == qg.QG_ERR_INVALID_ARG
