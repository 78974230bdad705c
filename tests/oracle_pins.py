"""Pins for the CPU oracle: checks against facts that do not come from the oracle.

Each ``check_*`` function takes a loaded oracle library (so that the same
checks can be run against deliberately broken copies of the oracle in
``test_oracle_mutants.py``) and raises ``AssertionError`` on a mismatch.

What pins what:
  * fp16 / bf16 decoding     -- numpy's float16 and torch's bfloat16
                                conversions on all 65536 bit patterns;
  * unpacking / bit order    -- hand-worked fixtures in tests/golden and
                                numpy.unpackbits(bitorder="little");
  * dequantization           -- hand-worked fixtures; closed forms computed
                                with exact rational arithmetic;
  * matmul index arithmetic  -- one-hot activations; brute-force int64
                                products with an integer codebook; numpy's
                                fp64 matmul on the oracle's dequantized matrix;
  * uniform zero point       -- scalar path vs a full tensor of the value;
  * QMoE composition         -- hand-worked fixture; the fused decode vs the
                                unfused chain (oracle GEMMs + numpy bias,
                                SwiGLU and weighted sum); one-hot slot weights;
  * E4M3 decoding            -- torch's float8_e4m3fn conversion on all 256
                                bit patterns;
  * int8 activations (dp4a)  -- hand-worked quantizer fixture (exact steps,
                                ties to even, zero block); bound, range and
                                oddness properties on random blocks; the fused
                                int8 decode vs the chain quantizer -> oracle
                                fp64 GEMM on q8*sx -> numpy bias / SwiGLU /
                                weighted sum;
  * nested absmax            -- hand-worked fixture; table[q] = q with an
                                affine second level reduces to the plain
                                codebook GEMM;
  * ragged expert GEMM       -- hand-worked fixture (an expert with no rows);
                                segment by segment equal to the MatMulNBits
                                oracle; bad offsets refused;
  * embedding gather         -- hand-worked fixture (u4 with and without zero
                                points, E4M3); numpy row selection of the
                                dequantized table; torch's float8 decode times
                                the scale.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np

import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _codes_via_unpackbits(W: np.ndarray, bits: int) -> np.ndarray:
    """Codes from packed bytes using numpy.unpackbits (LSB-first per byte)."""
    b = np.unpackbits(W, axis=-1, bitorder="little").reshape(W.shape[0], -1, bits)
    weights = (1 << np.arange(bits)).astype(np.int64)
    return (b.astype(np.int64) * weights).sum(axis=-1)


def _h2f(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _bf2f(bits: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------------------
def check_half_decode(lib):
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = allp.view(np.float16).astype(np.float64)
    got = np.array([lib.oracle_half_to_double(int(p)) for p in allp])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, got[0x8000]) == -1.0


def check_bf16_decode(lib):
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = _bf2f(allp)
    got = np.array([lib.oracle_bf16_to_double(int(p)) for p in allp])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def check_unpack_vs_unpackbits(lib):
    g = np.random.default_rng(11)
    for bits in (2, 3, 4, 8):
        N, K = 5, 96
        W = g.integers(0, 256, size=(N, K * bits // 8), dtype=np.uint8)
        # scale 1, zero point 0 makes the dequantized value the code itself
        ones = np.full((N, K // 32), np.float16(1.0).view(np.uint16), dtype=np.uint16)
        deq = O.dequant_nbits(W, ones, None, N=N, K=K, bits=bits, block_size=32, uniform_zp=0.0, lib=lib)
        assert np.array_equal(deq.astype(np.int64), _codes_via_unpackbits(W, bits))
        for (n, k) in [(0, 0), (1, 5), (4, K - 1), (3, 17)]:
            assert lib.oracle_code(W.ctypes.data, K, n, k, bits) == _codes_via_unpackbits(W, bits)[n, k]


def check_golden_u2(lib):
    d = _golden("u2_handworked.json")
    W = np.array(d["W"], dtype=np.uint8)
    S = np.array(d["scales_f16"], dtype=np.uint16)
    Z = np.array(d["zero_points_f16"], dtype=np.uint16)
    A = np.array(d["A"], dtype=np.float32)
    kw = dict(N=d["N"], K=d["K"], bits=d["bits"], block_size=d["block_size"], lib=lib)
    for deq in (O.dequant_nbits(W, S, Z, **kw), O.dequant_nbits(W, S, None, uniform_zp=d["uniform_zp"], **kw)):
        assert np.array_equal(deq, np.array(d["dequant"], dtype=np.float32))
    Y = O.qgemm_nbits(A, W, S, None, M=A.shape[0], uniform_zp=d["uniform_zp"], **kw)
    assert np.array_equal(Y, np.array(d["Y"]))
    Y = O.qgemm_nbits(A, W, S, Z, M=A.shape[0], **kw)
    assert np.array_equal(Y, np.array(d["Y"]))


def check_golden_u4(lib):
    d = _golden("u4_handworked.json")
    W = np.array(d["W"], dtype=np.uint8)
    S = np.array(d["scales_f16"], dtype=np.uint16)
    Z = np.array(d["zero_points_f16"], dtype=np.uint16)
    A = np.array(d["A"], dtype=np.float32)
    kw = dict(N=d["N"], K=d["K"], bits=d["bits"], block_size=d["block_size"], lib=lib)
    assert np.array_equal(O.dequant_nbits(W, S, Z, **kw), np.array(d["dequant"], dtype=np.float32))
    assert np.array_equal(O.dequant_nbits(W, S, None, **kw), np.array(d["dequant_no_zp"], dtype=np.float32))
    assert np.array_equal(O.qgemm_nbits(A, W, S, Z, M=2, **kw), np.array(d["Y"]))
    assert np.array_equal(O.qgemm_nbits(A, W, S, None, M=2, **kw), np.array(d["Y_no_zp"]))


def check_golden_u8(lib):
    d = _golden("u8_handworked.json")
    W = np.array(d["W"], dtype=np.uint8)
    S = np.array(d["scales_f16"], dtype=np.uint16)
    Z = np.array(d["zero_points_f16"], dtype=np.uint16)
    A = np.array(d["A"], dtype=np.float32)
    kw = dict(N=d["N"], K=d["K"], bits=d["bits"], block_size=d["block_size"], lib=lib)
    for n in range(d["N"]):
        for k in range(d["K"]):
            assert O.code(W, d["K"], n, k, 8, lib=lib) == d["codes"][n][k]
    assert np.array_equal(O.dequant_nbits(W, S, Z, **kw), np.array(d["dequant"], dtype=np.float32))
    assert np.array_equal(O.dequant_nbits(W, S, None, **kw), np.array(d["dequant_no_zp"], dtype=np.float32))
    assert np.array_equal(O.qgemm_nbits(A, W, S, Z, M=2, **kw), np.array(d["Y"]))
    assert np.array_equal(O.qgemm_nbits(A, W, S, None, M=2, **kw), np.array(d["Y_no_zp"]))


def check_golden_u3(lib):
    d = _golden("u3_handworked.json")
    W = np.array(d["W"], dtype=np.uint8)
    S = np.array(d["scales_f16"], dtype=np.uint16)
    Z = np.array(d["zero_points_f16"], dtype=np.uint16)
    A = np.array(d["A"], dtype=np.float32)
    kw = dict(N=d["N"], K=d["K"], bits=d["bits"], block_size=d["block_size"], lib=lib)
    for n in range(d["N"]):
        for k in range(d["K"]):
            assert O.code(W, d["K"], n, k, 3, lib=lib) == d["codes"][n][k]
    assert np.array_equal(O.dequant_nbits(W, S, Z, **kw), np.array(d["dequant"], dtype=np.float32))
    assert np.array_equal(O.dequant_nbits(W, S, None, **kw), np.array(d["dequant_no_zp"], dtype=np.float32))
    assert np.array_equal(O.qgemm_nbits(A, W, S, Z, M=2, **kw), np.array(d["Y"]))
    assert np.array_equal(O.qgemm_nbits(A, W, S, None, M=2, **kw), np.array(d["Y_no_zp"]))


def check_golden_codebook(lib):
    d = _golden("codebook4_handworked.json")
    W = np.array(d["W"], dtype=np.uint8)
    C = np.array(d["codebook"], dtype=np.float32)
    AM = np.array(d["absmax"], dtype=np.float32)
    A = np.array(d["A"], dtype=np.float32)
    kw = dict(N=d["N"], K=d["K"], block_size=d["block_size"], lib=lib)
    assert np.array_equal(O.dequant_codebook4(W, C, AM, **kw), np.array(d["dequant"], dtype=np.float32))
    assert np.array_equal(O.qgemm_codebook4(A, W, C, AM, M=2, **kw), np.array(d["Y"]))


def _pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack integer codes LSB-first along the last axis (numpy.packbits)."""
    c = np.asarray(codes, dtype=np.uint8)
    b = ((c[..., None] >> np.arange(bits)) & 1).astype(np.uint8)
    b = b.reshape(*c.shape[:-1], c.shape[-1] * bits)
    pad = (-b.shape[-1]) % 8
    if pad:
        b = np.concatenate([b, np.zeros((*b.shape[:-1], pad), np.uint8)], axis=-1)
    return np.packbits(b, axis=-1, bitorder="little")


def check_golden_qmoe(lib):
    d = _golden("qmoe_handworked.json")
    bits = d["bits"]
    fc1_w = _pack_codes(np.array(d["fc1_codes"]), bits)
    fc2_w = _pack_codes(np.array(d["fc2_codes"]), bits)
    kw = dict(num_experts=d["num_experts"], fc1_w=fc1_w, fc1_scales=np.array(d["fc1_scales_f16"], np.uint16),
              fc1_zp=None, fc1_bias=np.array(d["fc1_bias_f16"], np.uint16), fc2_w=fc2_w,
              fc2_scales=np.array(d["fc2_scales_f16"], np.uint16), fc2_zp=None,
              fc2_bias=np.array(d["fc2_bias_f16"], np.uint16), hidden=d["hidden"], inter=d["inter"],
              bits=bits, block_size=d["block_size"], lib=lib)
    x = np.array(d["x_f16"], np.uint16)
    w = np.array(d["weights"], np.float32)
    y, bad = O.qmoe_decode(x, np.array(d["ids"], np.int32), w, **kw)
    assert bad == 0
    np.testing.assert_allclose(y, d["y"], rtol=1e-14, atol=0)
    y, bad = O.qmoe_decode(x, np.array(d["ids_bad"], np.int32), w, **kw)
    assert bad == d["bad_slots"]
    np.testing.assert_allclose(y, d["y_bad"], rtol=1e-14, atol=0)


def check_onehot(lib):
    """A = e_k recovers column k of the dequantized matrix exactly."""
    g = np.random.default_rng(5)
    for bits in (2, 4):
        N, K, bs = 7, 128, 32
        W = g.integers(0, 256, size=(N, K * bits // 8), dtype=np.uint8)
        S = g.uniform(0.01, 0.05, size=(N, K // bs)).astype(np.float16).view(np.uint16)
        Z = g.integers(0, 2 ** bits, size=(N, K // bs)).astype(np.float16).view(np.uint16)
        deq = O.dequant_nbits(W, S, Z, N=N, K=K, bits=bits, block_size=bs, lib=lib)
        A = np.eye(K, dtype=np.float32)[[0, 1, 37, K - 1]]
        Y = O.qgemm_nbits(A, W, S, Z, M=4, N=N, K=K, bits=bits, block_size=bs, lib=lib)
        assert np.array_equal(Y, deq[:, [0, 1, 37, K - 1]].T.astype(np.float64))
        # and the dequantized value is exact: (q - zp) * s needs at most 17 significant bits
        codes = _codes_via_unpackbits(W, bits)
        exact = (codes - _h2f(Z).repeat(bs, axis=1)) * _h2f(S).repeat(bs, axis=1)
        assert np.array_equal(deq.astype(np.float64), exact)


def check_uniform_vs_tensor(lib):
    g = np.random.default_rng(6)
    for bits, zpv in ((2, 1.5), (4, 7.0), (4, 8.5)):
        N, K, bs = 9, 256, 64
        W = g.integers(0, 256, size=(N, K * bits // 8), dtype=np.uint8)
        S = g.uniform(0.01, 0.05, size=(N, K // bs)).astype(np.float16).view(np.uint16)
        Z = np.full((N, K // bs), np.float16(zpv).view(np.uint16), dtype=np.uint16)
        A = g.standard_normal((3, K)).astype(np.float32)
        kw = dict(M=3, N=N, K=K, bits=bits, block_size=bs, lib=lib)
        assert np.array_equal(O.qgemm_nbits(A, W, S, Z, **kw), O.qgemm_nbits(A, W, S, None, uniform_zp=zpv, **kw))


def check_closed_form(lib):
    """All codes equal c and A = 1:  y_n = sum_b bs * (c - zp_nb) * s_nb  (exact rationals)."""
    g = np.random.default_rng(7)
    for bits, byte_for_code in ((2, {1: 0x55, 2: 0xAA, 3: 0xFF}), (4, {5: 0x55, 10: 0xAA, 15: 0xFF})):
        N, K, bs = 4, 256, 64
        S = g.uniform(0.01, 0.05, size=(N, K // bs)).astype(np.float16).view(np.uint16)
        Z = g.integers(0, 2 ** bits, size=(N, K // bs)).astype(np.float16).view(np.uint16)
        A = np.ones((1, K), np.float32)
        for c, byte in byte_for_code.items():
            W = np.full((N, K * bits // 8), byte, np.uint8)
            Y = O.qgemm_nbits(A, W, S, Z, M=1, N=N, K=K, bits=bits, block_size=bs, lib=lib)
            for n in range(N):
                exact = sum(Fraction(bs) * (c - Fraction(float(_h2f(Z[n, b])))) * Fraction(float(_h2f(S[n, b])))
                            for b in range(K // bs))
                assert Fraction(Y[0, n]) == exact, (bits, c, n)


def check_integer_codebook(lib):
    """Codebook [0..15], absmax 1, integer A: an int64 matmul of the codes."""
    g = np.random.default_rng(8)
    N, K, bs, M = 6, 192, 64, 3
    W = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    C = np.arange(16, dtype=np.float32)
    AM = np.ones((N, K // bs), np.float32)
    Ai = g.integers(-3, 4, size=(M, K)).astype(np.int64)
    Y = O.qgemm_codebook4(Ai.astype(np.float32), W, C, AM, M=M, N=N, K=K, block_size=bs, lib=lib)
    exact = Ai @ _codes_via_unpackbits(W, 4).T
    assert np.array_equal(Y, exact.astype(np.float64))


def check_library_matmul(lib):
    """The oracle's fp64 loop equals numpy's fp64 matmul of A and its dequantized W."""
    import torch

    g = np.random.default_rng(9)
    M, N, K, bs = 3, 37, 320, 64
    A32 = g.standard_normal((M, K)).astype(np.float32)
    A16 = A32.astype(np.float16).view(np.uint16)
    Abf = torch.from_numpy(A32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for bits in (2, 4):
        W = g.integers(0, 256, size=(N, K * bits // 8), dtype=np.uint8)
        S = g.uniform(0.005, 0.05, size=(N, K // bs)).astype(np.float16).view(np.uint16)
        Z = g.integers(0, 2 ** bits, size=(N, K // bs)).astype(np.float16).view(np.uint16)
        for zp, uz in ((Z, None), (None, None), (None, 1.5)):
            deq = O.dequant_nbits(W, S, zp, N=N, K=K, bits=bits, block_size=bs, uniform_zp=uz, lib=lib).astype(np.float64)
            for A, ad, A64 in ((A32, O.F32, A32.astype(np.float64)), (A16, O.F16, _h2f(A16)), (Abf, O.BF16, _bf2f(Abf))):
                Y = O.qgemm_nbits(A, W, S, zp, M=M, N=N, K=K, bits=bits, block_size=bs, uniform_zp=uz, a_dtype=ad, lib=lib)
                np.testing.assert_allclose(Y, A64 @ deq.T, rtol=1e-12, atol=1e-12)
    W = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    C = np.sort(g.uniform(-1, 1, 16)).astype(np.float32)
    AM = g.uniform(0.02, 0.1, size=(N, K // bs)).astype(np.float32)
    deq = O.dequant_codebook4(W, C, AM, N=N, K=K, block_size=bs, lib=lib).astype(np.float64)
    Y = O.qgemm_codebook4(A16, W, C, AM, M=M, N=N, K=K, block_size=bs, a_dtype=O.F16, lib=lib)
    np.testing.assert_allclose(Y, _h2f(A16) @ deq.T, rtol=1e-12, atol=1e-12)
    # the codebook dequant is C[q] * absmax in fp32 (library: numpy float32 multiply)
    codes = _codes_via_unpackbits(W, 4)
    assert np.array_equal(O.dequant_codebook4(W, C, AM, N=N, K=K, block_size=bs, lib=lib),
                          C[codes] * AM.repeat(bs, axis=1))


def check_rows_subset(lib):
    g = np.random.default_rng(10)
    M, N, K, bs, bits = 2, 50, 128, 32, 4
    W = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    S = g.uniform(0.01, 0.05, size=(N, K // bs)).astype(np.float16).view(np.uint16)
    A = g.standard_normal((M, K)).astype(np.float32)
    full = O.qgemm_nbits(A, W, S, None, M=M, N=N, K=K, bits=bits, block_size=bs, lib=lib)
    rows = np.array([49, 0, 17, 17, 3])
    sub = O.qgemm_nbits(A, W, S, None, M=M, N=N, K=K, bits=bits, block_size=bs, rows=rows, lib=lib)
    assert np.array_equal(sub, full[:, rows])


def _qmoe_case(seed, E=5, k=3, H=64, I=96, bs=32, with_zp=True, with_bias=True):
    g = np.random.default_rng(seed)
    d = dict(num_experts=E, hidden=H, inter=I, bits=4, block_size=bs)
    d["fc1_w"] = g.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8)
    d["fc2_w"] = g.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    d["fc1_scales"] = g.uniform(0.005, 0.02, (E, 2 * I, H // bs)).astype(np.float16).view(np.uint16)
    d["fc2_scales"] = g.uniform(0.005, 0.02, (E, H, I // bs)).astype(np.float16).view(np.uint16)
    d["fc1_zp"] = g.integers(0, 16, (E, 2 * I, H // bs)).astype(np.float16).view(np.uint16) if with_zp else None
    d["fc2_zp"] = g.integers(0, 16, (E, H, I // bs)).astype(np.float16).view(np.uint16) if with_zp else None
    d["fc1_bias"] = (g.standard_normal((E, 2 * I)) * 0.01).astype(np.float16).view(np.uint16) if with_bias else None
    d["fc2_bias"] = (g.standard_normal((E, H)) * 0.01).astype(np.float16).view(np.uint16) if with_bias else None
    x = g.standard_normal(H).astype(np.float16).view(np.uint16)
    ids = g.choice(E, size=k, replace=False).astype(np.int32)
    w = g.uniform(0.1, 1.0, size=k).astype(np.float32)
    return d, x, ids, w


def _unfused_chain(lib, d, x, ids, w, interleaved):
    """The unfused chain: oracle GEMMs for fc1 and fc2, numpy for the rest."""
    H, I, bs = d["hidden"], d["inter"], d["block_size"]
    y = np.zeros(H)
    for j, e in enumerate(ids):
        z1 = None if d["fc1_zp"] is None else d["fc1_zp"][e]
        z2 = None if d["fc2_zp"] is None else d["fc2_zp"][e]
        gvec = O.qgemm_nbits(x.reshape(1, H), d["fc1_w"][e], d["fc1_scales"][e], z1, M=1, N=2 * I, K=H, bits=4,
                             block_size=bs, a_dtype=O.F16, lib=lib)[0]
        if d["fc1_bias"] is not None:
            gvec = gvec + _h2f(d["fc1_bias"][e])
        gate, up = (gvec[0::2], gvec[1::2]) if interleaved else (gvec[:I], gvec[I:])
        h = gate / (1.0 + np.exp(-gate)) * up
        o = O.qgemm_nbits(h.reshape(1, I), d["fc2_w"][e], d["fc2_scales"][e], z2, M=1, N=H, K=I, bits=4,
                          block_size=bs, a_dtype=O.F64, lib=lib)[0]
        if d["fc2_bias"] is not None:
            o = o + _h2f(d["fc2_bias"][e])
        y = y + float(w[j]) * o
    return y


def check_qmoe_chain(lib):
    for seed, zp, bias in ((1, True, True), (2, False, True), (3, True, False)):
        d, x, ids, w = _qmoe_case(seed, with_zp=zp, with_bias=bias)
        for inter_flag in (0, 1):
            y, bad = O.qmoe_decode(x, ids, w, swiglu_interleaved=inter_flag, lib=lib, **d)
            assert bad == 0
            np.testing.assert_allclose(y, _unfused_chain(lib, d, x, ids, w, inter_flag), rtol=1e-12, atol=1e-13)
    # one-hot slot weights reproduce one expert's chain alone
    d, x, ids, w = _qmoe_case(4)
    for j in range(len(ids)):
        onehot = np.zeros(len(ids), np.float32)
        onehot[j] = 1.0
        y, _ = O.qmoe_decode(x, ids, onehot, lib=lib, **d)
        np.testing.assert_allclose(y, _unfused_chain(lib, d, x, ids[j:j + 1], onehot[j:j + 1], 0),
                                   rtol=1e-12, atol=1e-13)


def check_uniform_detection(lib):
    h = lambda v: int(np.float16(v).view(np.uint16))
    assert O.fp16_uniform_value(np.full(1000, h(1.5), np.uint16), lib=lib) == (True, 1.5)
    t = np.full(1000, h(1.5), np.uint16)
    t[999] = h(2.5)
    assert O.fp16_uniform_value(t, lib=lib) == (False, None)
    t = np.full(10, 0, np.uint16)
    t[3] = 0x8000  # -0 next to +0: different bit patterns
    assert O.fp16_uniform_value(t, lib=lib) == (False, None)
    assert O.fp16_uniform_value(np.full(10, 0x7E00, np.uint16), lib=lib) == (False, None)  # NaN
    assert O.fp16_uniform_value(np.zeros(0, np.uint16), lib=lib) == (False, None)
    assert O.fp16_uniform_value(np.array([h(-3.0)], np.uint16), lib=lib) == (True, -3.0)


# ---------------------------------------------------------------------------
def _e4m3_via_torch(b: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.asarray(b, dtype=np.uint8).copy()).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def check_e4m3_decode(lib):
    """All 256 E4M3 patterns against torch's float8_e4m3fn conversion."""
    got = np.array([O.e4m3_to_double(b, lib) for b in range(256)])
    ref = _e4m3_via_torch(np.arange(256))
    assert np.array_equal(got, ref, equal_nan=True)
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(ref[~np.isnan(ref)]))


def _exact(got, want):
    want = np.asarray(want, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.array_equal(got, want), (got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def check_golden_gather(lib):
    g = _golden("gather_handworked.json")
    u = g["u4"]
    W = np.array(u["W"], dtype=np.uint8)
    sc = np.array(u["scales_f16"], dtype=np.uint16)
    zp = np.array(u["zero_points_f16"], dtype=np.uint16)
    out, bad = O.gather_block_quantized(u["indices"], W, sc, zp, V=u["V"], D=u["D"], fmt=O.W_U4,
                                        block_size=u["block_size"], lib=lib)
    _exact(out, u["out"])
    assert bad == u["bad"]
    out, bad = O.gather_block_quantized(u["indices"], W, sc, None, V=u["V"], D=u["D"], fmt=O.W_U4,
                                        block_size=u["block_size"], lib=lib)
    _exact(out, u["out_no_zp"])
    assert bad == u["bad"]
    e = g["e4m3"]
    out, bad = O.gather_block_quantized(e["indices"], np.array(e["W"], dtype=np.uint8),
                                        np.array(e["scales_f16"], dtype=np.uint16), None, V=e["V"], D=e["D"],
                                        fmt=O.W_E4M3, block_size=e["block_size"], lib=lib)
    _exact(out, e["out"])
    assert bad == e["bad"]


def check_gather_rows(lib):
    """The gather equals row selection (numpy fancy indexing, negative indices
    wrapped by numpy) of the dequantized table; E4M3 tables equal torch's
    float8 decode times the fp16 scale in fp32 (numpy)."""
    rng = np.random.default_rng(11)
    V, D, bs = 37, 96, 32
    idx = np.array([0, 36, -1, -37, 5, 5, 12, -20, 30], dtype=np.int64)
    for fmt, bits in ((O.W_U2, 2), (O.W_U4, 4), (O.W_U8, 8)):
        W = rng.integers(0, 256, size=(V, D * bits // 8), dtype=np.uint8)
        sc = rng.uniform(-0.1, 0.1, size=(V, D // bs)).astype(np.float16).view(np.uint16)
        zp = rng.integers(0, 1 << bits, size=(V, D // bs)).astype(np.float16).view(np.uint16)
        for z, zmode in ((zp, O.ZP_TENSOR), (None, O.ZP_NONE)):
            table = O.dequant_nbits(W, sc, z, N=V, K=D, bits=bits, block_size=bs, lib=lib)
            out, bad = O.gather_block_quantized(idx, W, sc, z, V=V, D=D, fmt=fmt, block_size=bs, lib=lib)
            assert bad == 0
            _exact(out, table[idx])
    W = rng.integers(0, 256, size=(V, D), dtype=np.uint8)
    W[W & 0x7F == 0x7F] = 0x3F  # no NaN patterns, so that exact equality applies
    sc = rng.uniform(-4, 4, size=(V, D // bs)).astype(np.float16)
    table = (_e4m3_via_torch(W).astype(np.float32) * np.repeat(sc.astype(np.float32), bs, axis=1)).astype(np.float32)
    out, bad = O.gather_block_quantized(idx, W, sc.view(np.uint16), None, V=V, D=D, fmt=O.W_E4M3, block_size=bs,
                                        lib=lib)
    assert bad == 0
    _exact(out, table[idx])
    out, bad = O.gather_block_quantized(np.array([V, -V - 1, 0]), W, sc.view(np.uint16), None, V=V, D=D,
                                        fmt=O.W_E4M3, block_size=bs, lib=lib)
    assert bad == 2
    _exact(out[:2], np.zeros((2, D)))
    _exact(out[2], table[0])


# ---------------------------------------------------------------------------
def check_golden_i8_quant(lib):
    g = _golden("i8_quant_handworked.json")
    q8, sx = O.quantize_i8_blocks(np.array(g["v"], dtype=np.float32), g["block_size"], lib=lib)
    assert q8.tolist() == g["q8"], q8.tolist()
    assert sx.tolist() == g["sx"], sx.tolist()


def check_i8_quant_properties(lib):
    """Random blocks over a wide range of magnitudes: |q| <= 127, the block's
    largest magnitude maps to +-127, the rounding error is at most half a step,
    and the quantizer is odd (q(-v) = -q(v))."""
    rng = np.random.default_rng(21)
    bs = 32
    mags = np.repeat(10.0 ** rng.uniform(-30, 30, size=64), bs)
    v = (rng.standard_normal(64 * bs) * mags).astype(np.float32)
    v[5 * bs:6 * bs] = 0.0
    q8, sx = O.quantize_i8_blocks(v, bs, lib=lib)
    qn, sxn = O.quantize_i8_blocks(-v, bs, lib=lib)
    assert np.array_equal(qn, -q8) and np.array_equal(sxn, sx)
    assert np.abs(q8.astype(np.int64)).max() <= 127
    for b in range(64):
        blk = slice(b * bs, (b + 1) * bs)
        vb, qb = v[blk].astype(np.float64), q8[blk].astype(np.float64)
        if not np.any(vb):
            assert sx[b] == 0 and not np.any(qb)
            continue
        i = int(np.argmax(np.abs(vb)))
        assert abs(qb[i]) == 127 and np.sign(qb[i]) == np.sign(vb[i])
        assert np.all(np.abs(qb * float(sx[b]) - vb) <= 0.5001 * float(sx[b]))


def _dp4a_chain(lib, d, x, ids, w, interleaved):
    """The int8-activation decode as a chain of pinned pieces: the quantizer,
    the oracle's fp64 GEMM on the dequantized activations q8 * sx (exact in
    fp64), numpy for bias, SwiGLU (rounded to fp32, as the quantizer's input)
    and the weighted sum."""
    H, I, bs = d["hidden"], d["inter"], d["block_size"]

    def deq(v):
        q8, sx = O.quantize_i8_blocks(v, bs, lib=lib)
        return q8.astype(np.float64) * np.repeat(sx.astype(np.float64), bs)

    y = np.zeros(H)
    xa = deq(_h2f(x).astype(np.float32))
    for j, e in enumerate(ids):
        z1 = None if d["fc1_zp"] is None else d["fc1_zp"][e]
        z2 = None if d["fc2_zp"] is None else d["fc2_zp"][e]
        gvec = O.qgemm_nbits(xa.reshape(1, H), d["fc1_w"][e], d["fc1_scales"][e], z1, M=1, N=2 * I, K=H, bits=4,
                             block_size=bs, a_dtype=O.F64, lib=lib)[0]
        if d["fc1_bias"] is not None:
            gvec = gvec + _h2f(d["fc1_bias"][e])
        gate, up = (gvec[0::2], gvec[1::2]) if interleaved else (gvec[:I], gvec[I:])
        h = (gate / (1.0 + np.exp(-gate)) * up).astype(np.float32)
        o = O.qgemm_nbits(deq(h).reshape(1, I), d["fc2_w"][e], d["fc2_scales"][e], z2, M=1, N=H, K=I, bits=4,
                          block_size=bs, a_dtype=O.F64, lib=lib)[0]
        if d["fc2_bias"] is not None:
            o = o + _h2f(d["fc2_bias"][e])
        y = y + float(w[j]) * o
    return y


def check_qmoe_dp4a_chain(lib):
    for seed, zp, bias in ((1, True, True), (2, False, True), (3, True, False)):
        d, x, ids, w = _qmoe_case(seed, with_zp=zp, with_bias=bias)
        for inter_flag in (0, 1):
            y, bad = O.qmoe_decode_dp4a(x, ids, w, swiglu_interleaved=inter_flag, lib=lib, **d)
            assert bad == 0
            np.testing.assert_allclose(y, _dp4a_chain(lib, d, x, ids, w, inter_flag), rtol=1e-10, atol=1e-12)
    d, x, ids, w = _qmoe_case(5)
    bad_ids = ids.copy()
    bad_ids[1] = d["num_experts"]
    y, bad = O.qmoe_decode_dp4a(x, bad_ids, w, lib=lib, **d)
    assert bad == 1
    keep = np.array([0, 2])
    np.testing.assert_allclose(y, _dp4a_chain(lib, d, x, ids[keep], w[keep], 0), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------
def check_golden_ragged(lib):
    g = _golden("ragged_handworked.json")
    Y = O.qmoe_ragged_mm(np.array(g["X"], dtype=np.float32), g["offsets"], np.array(g["W"], dtype=np.uint8),
                         np.array(g["scales_f16"], dtype=np.uint16), None, N=g["N"], K=g["K"], bits=4,
                         block_size=g["block_size"], lib=lib)
    assert Y.tolist() == g["Y"], Y.tolist()


def check_ragged_vs_per_expert(lib):
    """The ragged GEMM equals, segment by segment, the (pinned) MatMulNBits
    oracle applied to the segment's rows with that expert's weight."""
    rng = np.random.default_rng(31)
    E, N, K, bs = 6, 20, 96, 32
    offsets = np.array([0, 3, 3, 4, 11, 11, 15], dtype=np.int64)  # experts 1 and 4 own no rows
    T = int(offsets[-1])
    for bits in (2, 4):
        W = rng.integers(0, 256, size=(E, N, K * bits // 8), dtype=np.uint8)
        sc = rng.uniform(0.005, 0.05, size=(E, N, K // bs)).astype(np.float16).view(np.uint16)
        zp = rng.integers(0, 1 << bits, size=(E, N, K // bs)).astype(np.float16).view(np.uint16)
        X = rng.standard_normal((T, K)).astype(np.float16)
        for z in (zp, None):
            Y = O.qmoe_ragged_mm(X.view(np.uint16), offsets, W, sc, z, N=N, K=K, bits=bits, block_size=bs,
                                 x_dtype=O.F16, lib=lib)
            for e in range(E):
                a, b = int(offsets[e]), int(offsets[e + 1])
                if a == b:
                    continue
                ref = O.qgemm_nbits(X[a:b].view(np.uint16), W[e], sc[e], None if z is None else z[e], M=b - a, N=N,
                                    K=K, bits=bits, block_size=bs, a_dtype=O.F16, lib=lib)
                assert np.array_equal(Y[a:b], ref), e


def check_ragged_bad_offsets(lib):
    W = np.zeros((2, 2, 16), dtype=np.uint8)
    sc = np.zeros((2, 2, 1), dtype=np.uint16)
    for bad in ([1, 2, 3], [0, 3, 2]):
        try:
            O.qmoe_ragged_mm(np.zeros((3, 32), np.float32), bad, W, sc, N=2, K=32, bits=4, block_size=32, lib=lib)
        except ValueError:
            continue
        raise AssertionError("offsets %s accepted" % bad)


# ---------------------------------------------------------------------------
def check_golden_nested_absmax(lib):
    g = _golden("nested_absmax_handworked.json")
    table = ((np.arange(256) - 128) / 128).astype(np.float32)  # the fixture's table rule
    got = O.nested_absmax(np.array(g["qa"], dtype=np.uint8), table, np.array(g["absmax2"], dtype=np.float32),
                          g["offset"], g["nested_block"], lib=lib)
    assert got.tolist() == g["absmax"], got.tolist()


def check_nested_reduces_to_plain(lib):
    """table[q] = q, absmax2 = 2, offset = 0.5: absmax = 2 q + 0.5 exactly, so the
    nested GEMM equals the (pinned) plain codebook GEMM on that absmax."""
    rng = np.random.default_rng(41)
    M, N, K, bs, nbl = 3, 37, 256, 64, 16
    W = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    cb = rng.standard_normal(16).astype(np.float32)
    qa = rng.integers(0, 256, size=(N, K // bs), dtype=np.uint8)
    nblocks = -(-qa.size // nbl)
    A = rng.standard_normal((M, K)).astype(np.float32)
    table = np.arange(256, dtype=np.float32)
    absmax2 = np.full(nblocks, 2.0, dtype=np.float32)
    y = O.qgemm_codebook4_nested(A, W, cb, qa, table, absmax2, 0.5, M=M, N=N, K=K, block_size=bs, nested_block=nbl,
                                 lib=lib)
    ref = O.qgemm_codebook4(A, W, cb, (2.0 * qa.astype(np.float64) + 0.5).astype(np.float32), M=M, N=N, K=K,
                            block_size=bs, lib=lib)
    assert np.array_equal(y, ref)
    # a second-level scale per group of nested_block values in flat order
    absmax2 = (1.0 + np.arange(nblocks)).astype(np.float32)
    got = O.nested_absmax(qa, table, absmax2, 0.0, nbl, lib=lib)
    flat = qa.reshape(-1).astype(np.float64) * np.repeat(absmax2.astype(np.float64), nbl)[: qa.size]
    assert np.array_equal(got.reshape(-1).astype(np.float64), flat)


def check_golden_packed_zp(lib):
    g = _golden("packed_zp_handworked.json")
    for c in g["unpack"]:
        got = O.unpack_zero_points(np.array(c["bytes"], dtype=np.uint8), N=c["N"], nb=c["nb"], bits=c["bits"], lib=lib)
        assert got.reshape(-1).tolist() == c["zero_points"], (c["bits"], got.tolist())
    e = g["gemm"]
    y = O.qgemm_nbits_packed_zp(np.array(e["A"], dtype=np.float32).reshape(e["M"], e["K"]),
                                np.array(e["W"], dtype=np.uint8).reshape(e["N"], -1),
                                np.array(e["scales_f16"], dtype=np.uint16).reshape(e["N"], -1),
                                np.array(e["zp_packed"], dtype=np.uint8).reshape(e["N"], -1), M=e["M"], N=e["N"],
                                K=e["K"], bits=e["bits"], block_size=e["block_size"], lib=lib)
    assert y.reshape(-1).tolist() == e["Y"], y


def _pack_fields(z, bits):
    """Pack an [N, nb] integer array bit by bit: field b of a row at bits
    b*bits .. b*bits+bits-1 of the row's bit string, rows padded to bytes."""
    N, nb = z.shape
    nbytes = (nb * bits + 7) // 8
    out = np.zeros((N, nbytes), dtype=np.uint8)
    for n in range(N):
        bitlist = []
        for b in range(nb):
            bitlist += [(int(z[n, b]) >> t) & 1 for t in range(bits)]
        bitlist += [0] * (8 * nbytes - len(bitlist))
        for i in range(nbytes):
            out[n, i] = sum(bitlist[8 * i + t] << t for t in range(8))
    return out


def check_packed_zp_roundtrip_and_reduction(lib):
    """Unpacking inverts a bit-by-bit packer (odd field counts, fields that
    straddle bytes, padded rows), and the packed-zero-point GEMM equals the
    (pinned) zero-point-tensor GEMM on the same integers."""
    rng = np.random.default_rng(53)
    for bits in (2, 3, 4, 8):
        for nb in (1, 3, 7, 90):
            z = rng.integers(0, 1 << bits, size=(5, nb))
            got = O.unpack_zero_points(_pack_fields(z, bits), N=5, nb=nb, bits=bits, lib=lib)
            assert np.array_equal(got, z), (bits, nb)
    for bits, bs in ((2, 64), (3, 32), (4, 32), (8, 128)):
        M, N, K = 3, 29, 256
        nb = K // bs
        W = rng.integers(0, 256, size=(N, K * bits // 8), dtype=np.uint8)
        S = rng.uniform(0.01, 0.05, size=(N, nb)).astype(np.float16).view(np.uint16)
        z = rng.integers(0, 1 << bits, size=(N, nb))
        A = rng.standard_normal((M, K)).astype(np.float32)
        y = O.qgemm_nbits_packed_zp(A, W, S, _pack_fields(z, bits), M=M, N=N, K=K, bits=bits, block_size=bs, lib=lib)
        ref = O.qgemm_nbits(A, W, S, z.astype(np.float16).view(np.uint16), M=M, N=N, K=K, bits=bits, block_size=bs,
                            lib=lib)
        assert np.array_equal(y, ref), bits


ALL_CHECKS = [
    check_half_decode, check_bf16_decode, check_unpack_vs_unpackbits, check_golden_u2, check_golden_u3, check_golden_u4, check_golden_u8,
    check_golden_codebook, check_golden_qmoe, check_onehot, check_uniform_vs_tensor, check_closed_form,
    check_integer_codebook, check_library_matmul, check_rows_subset, check_qmoe_chain, check_uniform_detection,
    check_e4m3_decode, check_golden_gather, check_gather_rows,
    check_golden_i8_quant, check_i8_quant_properties, check_qmoe_dp4a_chain,
    check_golden_ragged, check_ragged_vs_per_expert, check_ragged_bad_offsets,
    check_golden_nested_absmax, check_nested_reduces_to_plain,
    check_golden_packed_zp, check_packed_zp_roundtrip_and_reduction,
]
