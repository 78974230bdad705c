"""Helpers shared by the GPU tests: move seeded numpy inputs to the device and
compare library outputs with the oracle."""
from __future__ import annotations

import numpy as np

import oracle as O

F32, F16, BF16 = 0, 1, 2


def torch():
    import torch as _t

    return _t


def dev(a: np.ndarray, dtype=None):
    """numpy -> CUDA tensor.  uint16 arrays become float16/bfloat16 when dtype says so."""
    t = torch()
    x = t.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        x = x.view(t.int16)
        if dtype is not None:
            x = x.view(dtype)
    return x.to("cuda")


def act_tensor(A: np.ndarray, a_dtype: int):
    t = torch()
    if a_dtype == F32:
        return dev(A)
    return dev(A, t.float16 if a_dtype == F16 else t.bfloat16)


def y_tensor(M, N, y_dtype):
    t = torch()
    dt = {F32: t.float32, F16: t.float16, BF16: t.bfloat16}[y_dtype]
    return t.full((M, N), float("nan"), dtype=dt, device="cuda")


def to64(Y) -> np.ndarray:
    return Y.float().double().cpu().numpy()


def nbits_case(d, device_zp=True):
    """Device tensors for an nbits workload dict from workloads.py."""
    t = torch()
    out = dict(A=act_tensor(d["A"], d["a_dtype"]), W=dev(d["W"]), scales=dev(d["scales"], t.float16))
    out["zero_points"] = dev(d["zero_points"], t.float16) if (device_zp and d.get("zero_points") is not None) else None
    return out


def oracle_nbits(d, rows=None, use_uniform=True):
    uz = d.get("uniform_zp") if use_uniform else None
    zp = None if uz is not None else d.get("zero_points")
    return O.qgemm_nbits(d["A"], d["W"], d["scales"], zp, M=d["M"], N=d["N"], K=d["K"], bits=d["bits"],
                         block_size=d["block_size"], uniform_zp=uz, a_dtype=d["a_dtype"], rows=rows)


def tol_for(a_dtype, y_dtype):
    """The parity bar: max relative L2 error 1e-4 for fp32 activations with fp32
    output, 5e-3 for fp16/bf16 activations or a 16-bit output."""
    return 1e-4 if (a_dtype == F32 and y_dtype == F32) else 5e-3


def sample_rows(N, count, seed=1):
    g = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, N - 1], g.choice(N, size=min(count, N), replace=False)]))
    return rows.astype(np.int64)
