"""GPU parity of the codebook GEMM with a nested (double-quantized) absmax.

The expansion is compared bit for bit with the oracle (it is read back from the
front of the workspace, where the library documents it); the GEMM itself on
the SIMT (M <= 8) and tensor-core (M >= 9, 16-bit activations) paths against the
oracle's GEMM on the oracle's expansion.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import act_tensor, dev, to64, torch, y_tensor

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


def _run(qg, d, workspace=None):
    Y = y_tensor(d["M"], d["N"], d["a_dtype"])
    qg.qgemm_codebook4_nested(act_tensor(d["A"], d["a_dtype"]), dev(d["W"]), dev(d["codebook"]), dev(d["absmax_q"]),
                              dev(d["absmax_table"]), dev(d["absmax2"]), d["absmax_offset"], Y,
                              block_size=d["block_size"], nested_block=d["nested_block"], workspace=workspace)
    torch().cuda.synchronize()
    return Y


def _oracle(d):
    return O.qgemm_codebook4_nested(d["A"], d["W"], d["codebook"], d["absmax_q"], d["absmax_table"], d["absmax2"],
                                    d["absmax_offset"], M=d["M"], N=d["N"], K=d["K"], block_size=d["block_size"],
                                    nested_block=d["nested_block"], a_dtype=d["a_dtype"])


@pytest.mark.parametrize("M,a_dtype", [(1, 2), (4, 1), (16, 2), (64, 1), (3, 0)])
@pytest.mark.parametrize("nested_block", [256, 100])
def test_nested_codebook_parity(qg, M, a_dtype, nested_block):
    d = WL.nf4_nested((700, 1024), M, a_dtype, seed=M, nested_block=nested_block)
    Y = _run(qg, d)
    tol = 1e-4 if a_dtype == 0 else 5e-3
    assert O.max_rel_l2(to64(Y), _oracle(d)) <= tol


def test_nested_expansion_bit_exact(qg):
    t = torch()
    d = WL.nf4_nested((333, 1536), 1, 2, seed=7, nested_block=100)
    ws = t.zeros(qg.qgemm_codebook4_nested_workspace_bytes(2, 1, d["N"], d["K"], 64), dtype=t.uint8, device="cuda")
    _run(qg, d, workspace=ws)
    n = d["absmax_q"].size
    got = ws[: 4 * n].view(t.float32).cpu().numpy()
    ref = O.nested_absmax(d["absmax_q"], d["absmax_table"], d["absmax2"], d["absmax_offset"], d["nested_block"])
    assert np.array_equal(got.view(np.uint32), ref.reshape(-1).view(np.uint32))


def test_nested_refusals(qg):
    t = torch()
    d = WL.nf4_nested((64, 256), 1, 2, seed=1)
    A, W, cb = act_tensor(d["A"], 2), dev(d["W"]), dev(d["codebook"])
    qa, tab, a2 = dev(d["absmax_q"]), dev(d["absmax_table"]), dev(d["absmax2"])
    Y = y_tensor(1, 64, 2)
    f = lambda off=0.06, nb=256, tab_=tab: qg.qgemm_codebook4_nested(A, W, cb, qa, tab_, a2, off, Y, block_size=64,
                                                                   nested_block=nb, raw=True)
    assert f() == qg.QG_OK
    assert f(nb=0) == qg.QG_ERR_INVALID_ARG
    assert f(off=float("nan")) == qg.QG_ERR_INVALID_ARG
    tab_odd = t.zeros(258, dtype=t.float16, device="cuda")[1:257]  # a pointer 2 bytes past a 4-byte boundary
    assert qg.qgemm_codebook4_nested(A, W, cb, qa, tab_odd, a2, 0.06, Y, block_size=64, raw=True) == \
        qg.QG_ERR_INVALID_ARG  # table not 4-byte aligned
    t.cuda.synchronize()
