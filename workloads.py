"""Seeded synthetic inputs for the blockwise-dequant GEMV/GEMM and QMoE workloads.

This module only draws numbers.  It holds none of the method's arithmetic (no
unpacking, dequantization or matmul), so that the CPU oracle and the GPU
library can both be fed from it without sharing any computation.

Uniform codes packed along K are exactly uniform random bytes, so packed
weights are drawn byte-wise.  fp16 / bf16 tensors are returned as their
uint16 bit patterns.  Every generator takes a numpy ``Generator``; the
workload builders seed one ``PCG64`` per workload (seed 0 by default) and
draw in a fixed order: codes, scales, zero points, absmax / codebook, bias,
activations, routing.

Shapes and value distributions follow the workloads of the source pages:
  * hip-ep #1318 "Performance" (phi4-14B 2-bit export: MatMulNBits bits=2,
    block 64, fp16 zero points all 1.5, fp32 activations);
  * hip-ep #1328 "Test plan" / "Performance" (fused QMoE decode, u4, block
    32/64/128, optional zero points and bias; GPT-OSS-20B-like 2880/2880);
  * bitsandbytes #1979 "Summary" (NF4/FP4 codebook GEMM at small M, GQA k/v,
    MoE expert shapes).
The pages measured real checkpoints and a 40-shape sweep that is not
available; these synthetic tensors of the same shapes stand in for them.
"""
from __future__ import annotations

from statistics import NormalDist

import numpy as np

F32, F16, BF16 = 0, 1, 2

# phi4-14B linear layers (N, K): hidden 5120, intermediate 17920, vocab 100352
PHI4_SHAPES = {
    "qkv": (7680, 5120),
    "o": (5120, 5120),
    "gate_up": (35840, 5120),
    "down": (5120, 17920),
    "lm_head": (100352, 5120),
}

NF4_SHAPES = {
    "square": (4096, 4096),
    "gqa_kv": (1024, 4096),
    "up": (14336, 4096),
    "down": (4096, 14336),
}

PREFILL_SHAPES = {
    "gate_up": (35840, 5120),
    "down": (5120, 17920),
}


def rng(seed: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def packed_codes(g: np.random.Generator, N: int, K: int, bits: int) -> np.ndarray:
    """[N, K*bits/8] uint8: uniform codes in [0, 2^bits) packed along K."""
    assert (K * bits) % 8 == 0
    return g.integers(0, 256, size=(N, K * bits // 8), dtype=np.uint8)


def fp16_uniform(g: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    """fp16 bit patterns of U(lo, hi) draws (rounded to fp16)."""
    return g.uniform(lo, hi, size=shape).astype(np.float16).view(np.uint16)


def fp16_uniform_int(g: np.random.Generator, shape, lo: int, hi: int) -> np.ndarray:
    """fp16 bit patterns of integers uniform in [lo, hi]."""
    return g.integers(lo, hi + 1, size=shape).astype(np.float16).view(np.uint16)


def fp16_const(shape, value: float) -> np.ndarray:
    return np.full(shape, value, dtype=np.float16).view(np.uint16)


def fp16_normal(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (g.standard_normal(size=shape) * std).astype(np.float16).view(np.uint16)


def f32_uniform(g: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return g.uniform(lo, hi, size=shape).astype(np.float32)


def f32_normal(g: np.random.Generator, shape) -> np.ndarray:
    return g.standard_normal(size=shape).astype(np.float32)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float32 values, round-to-nearest-even (via torch)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def activations(g: np.random.Generator, M: int, K: int, a_dtype: int) -> np.ndarray:
    """A ~ N(0, 1) as float32, or fp16 / bf16 bit patterns (uint16)."""
    x = f32_normal(g, (M, K))
    if a_dtype == F32:
        return x
    if a_dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    return bf16_bits_from_f32(x)


def nf4_codebook() -> np.ndarray:
    """16 fp32 entries: normal quantiles scaled into [-1, 1], with an exact 0.

    8 positive and 7 negative quantiles of N(0, 1) at evenly spaced
    probabilities in (1/2, 31/32], each side divided by its largest value,
    plus 0 -- the NF4 idea (equal-mass bins of a normal), built here from the
    inverse normal CDF rather than from any library's constants.
    """
    nd = NormalDist()
    top = 1.0 - 1.0 / 32.0
    pos = [nd.inv_cdf(p) for p in np.linspace(0.5, top, 9)[1:]]
    neg = [-nd.inv_cdf(p) for p in np.linspace(0.5, top, 8)[1:]]
    vals = [v / pos[-1] for v in pos] + [v / -neg[-1] for v in neg] + [0.0]
    cb = np.array(sorted(vals), dtype=np.float32)
    assert cb.size == 16 and cb[0] == -1.0 and cb[-1] == 1.0 and 0.0 in cb
    return cb


# ---------------------------------------------------------------------------
# Workload builders.  Each returns a dict of numpy arrays plus the sizes.
# ---------------------------------------------------------------------------

def tiny_u4(seed: int = 0) -> dict:
    """M=1, K=256, N=128, u4 block 64, fp16 scales U(0.005, 0.02), fp16 zero
    points uniform integers in [0, 15], fp32 A ~ N(0,1), fp32 out."""
    g = rng(seed)
    M, N, K, bits, bs = 1, 128, 256, 4, 64
    W = packed_codes(g, N, K, bits)
    scales = fp16_uniform(g, (N, K // bs), 0.005, 0.02)
    zp = fp16_uniform_int(g, (N, K // bs), 0, 15)
    A = activations(g, M, K, F32)
    return dict(M=M, N=N, K=K, bits=bits, block_size=bs, W=W, scales=scales, zero_points=zp, A=A,
                a_dtype=F32)


def phi4_u8(shape: str, M: int = 1, seed: int = 0) -> dict:
    """The phi4-14B decode shapes with 8-bit codes: block 64, fp16 scales
    U(0.0005, 0.002) (|w| of the same order as the u2 workload), zero points
    all 128 (the midpoint, passed as a scalar), fp32 A ~ N(0,1), fp32 out."""
    N, K = PHI4_SHAPES[shape]
    g = rng(seed)
    bits, bs = 8, 64
    W = packed_codes(g, N, K, bits)
    scales = fp16_uniform(g, (N, K // bs), 0.0005, 0.002)
    A = activations(g, M, K, F32)
    return dict(M=M, N=N, K=K, bits=bits, block_size=bs, W=W, scales=scales, zero_points=None,
                uniform_zp=128.0, A=A, a_dtype=F32)


def phi4_u2(shape: str, M: int = 1, seed: int = 0, full_zp_tensor: bool = False) -> dict:
    """phi4-14B-shaped 2-bit decode: u2 block 64, fp16 scales U(0.01, 0.05),
    zero points all exactly 1.5 (scalar path; optionally also as a full fp16
    tensor), fp32 A ~ N(0,1), fp32 out."""
    N, K = PHI4_SHAPES[shape]
    g = rng(seed)
    bits, bs = 2, 64
    W = packed_codes(g, N, K, bits)
    scales = fp16_uniform(g, (N, K // bs), 0.01, 0.05)
    zp = fp16_const((N, K // bs), 1.5) if full_zp_tensor else None
    A = activations(g, M, K, F32)
    return dict(M=M, N=N, K=K, bits=bits, block_size=bs, W=W, scales=scales, zero_points=zp,
                uniform_zp=1.5, A=A, a_dtype=F32)


def packed_zp(N: int, K: int, M: int = 1, bits: int = 4, block_size: int = 32, a_dtype: int = F32,
              seed: int = 0, scale_range=(0.005, 0.02)) -> dict:
    """MatMulNBits with packed unsigned-integer zero points: codes uniform,
    fp16 scales U(scale_range), zero points as uniform random bytes
    [N, ceil(nb*bits/8)] (uniform fields; any pad bits random too), A ~ N(0,1)
    in a_dtype."""
    g = rng(seed)
    nb = K // block_size
    W = packed_codes(g, N, K, bits)
    scales = fp16_uniform(g, (N, nb), *scale_range)
    zp_packed = g.integers(0, 256, size=(N, (nb * bits + 7) // 8), dtype=np.uint8)
    A = activations(g, M, K, a_dtype)
    return dict(M=M, N=N, K=K, bits=bits, block_size=block_size, W=W, scales=scales, zp_packed=zp_packed, A=A,
                a_dtype=a_dtype)


def nf4(shape: str, M: int, a_dtype: int, seed: int = 0) -> dict:
    """NF4-style codebook GEMM: 4-bit codes uniform, fp32 absmax per 64-element
    block U(0.02, 0.1), 16-entry normal-quantile codebook, A ~ N(0,1) in bf16
    or fp16; the output takes A's dtype."""
    N, K = NF4_SHAPES[shape] if isinstance(shape, str) else shape
    g = rng(seed)
    bs = 64
    W = packed_codes(g, N, K, 4)
    absmax = f32_uniform(g, (N, K // bs), 0.02, 0.1)
    codebook = nf4_codebook()
    A = activations(g, M, K, a_dtype)
    return dict(M=M, N=N, K=K, block_size=bs, W=W, absmax=absmax, codebook=codebook, A=A, a_dtype=a_dtype)


def qmoe(num_experts: int = 128, k: int = 8, hidden: int = 2880, inter: int = 2880, block_size: int = 32,
         with_zp: bool = False, with_bias: bool = True, seed: int = 0, bits: int = 4) -> dict:
    """One-token QMoE decode: fc1 [E][2I][H] and fc2 [E][H][I] codes (u4 unless
    bits says otherwise), fp16 scales U(0.005, 0.02), optional fp16 zero points
    (integers in [0, 2^bits - 1]),
    fp16 bias ~ N(0, 0.01), fp16 x ~ N(0, 1); k distinct expert ids and
    softmax weights over k N(0, 1) logits (fp64 softmax rounded to fp32)."""
    g = rng(seed)
    E, H, I, bs = num_experts, hidden, inter, block_size
    fc1_w = packed_codes(g, E * 2 * I, H, bits).reshape(E, 2 * I, H * bits // 8)
    fc2_w = packed_codes(g, E * H, I, bits).reshape(E, H, I * bits // 8)
    fc1_scales = fp16_uniform(g, (E, 2 * I, H // bs), 0.005, 0.02)
    fc2_scales = fp16_uniform(g, (E, H, I // bs), 0.005, 0.02)
    fc1_zp = fp16_uniform_int(g, (E, 2 * I, H // bs), 0, (1 << bits) - 1) if with_zp else None
    fc2_zp = fp16_uniform_int(g, (E, H, I // bs), 0, (1 << bits) - 1) if with_zp else None
    fc1_bias = fp16_normal(g, (E, 2 * I), 0.01) if with_bias else None
    fc2_bias = fp16_normal(g, (E, H), 0.01) if with_bias else None
    x = fp16_normal(g, (H,), 1.0)
    ids, weights = routing(g, E, k)
    return dict(num_experts=E, k=k, hidden=H, inter=I, bits=bits, block_size=bs, fc1_w=fc1_w,
                fc1_scales=fc1_scales, fc1_zp=fc1_zp, fc1_bias=fc1_bias, fc2_w=fc2_w, fc2_scales=fc2_scales,
                fc2_zp=fc2_zp, fc2_bias=fc2_bias, x=x, ids=ids, weights=weights)


def routing(g: np.random.Generator, num_experts: int, k: int):
    """k distinct expert ids and fp32 softmax weights over k N(0,1) logits."""
    ids = g.choice(num_experts, size=k, replace=False).astype(np.int32)
    logits = g.standard_normal(size=k)
    e = np.exp(logits - logits.max())
    weights = (e / e.sum()).astype(np.float32)
    return ids, weights


def prefill_u2(shape: str, M: int = 2048, seed: int = 0) -> dict:
    """Prefill-sized 2-bit GEMM: fp16 A ~ N(0,1), u2 block 64, fp16 scales
    U(0.01, 0.05), zero points all 1.5 (scalar), fp32 out."""
    N, K = PREFILL_SHAPES[shape] if isinstance(shape, str) else shape
    g = rng(seed)
    bits, bs = 2, 64
    W = packed_codes(g, N, K, bits)
    scales = fp16_uniform(g, (N, K // bs), 0.01, 0.05)
    A = activations(g, M, K, F16)
    return dict(M=M, N=N, K=K, bits=bits, block_size=bs, W=W, scales=scales, zero_points=None,
                uniform_zp=1.5, A=A, a_dtype=F16)


# Embedding tables: the kernel test table's gather_block_quantized leaves
# (int64 indices, u4 / u8 / fp8 table, fp16 output), on phi4-14B's
# embedding shape (vocab 100352, hidden 5120) looked up for a 2048-token
# prompt.  Table formats: 0 u2, 1 u4, 2 u8, 3 E4M3.
EMBED_BITS = {0: 2, 1: 4, 2: 8, 3: 8}


def embedding(fmt: int, V: int = 100352, D: int = 5120, n: int = 2048, block_size: int = 32,
              zero_points: bool = True, seed: int = 0) -> dict:
    """Table codes (uniform bytes; E4M3 tables without the two NaN patterns),
    fp16 scales U(0.005, 0.02), fp16 integer zero points (integer formats) and
    n token ids uniform in [0, V)."""
    g = rng(seed)
    bits = EMBED_BITS[fmt]
    W = packed_codes(g, V, D, bits)
    if fmt == 3:
        W[(W & 0x7F) == 0x7F] ^= 1  # 0x7F / 0xFF (NaN) -> 0x7E / 0xFE
    scales = fp16_uniform(g, (V, D // block_size), 0.005, 0.02)
    zp = fp16_uniform_int(g, (V, D // block_size), 0, (1 << bits) - 1) if (zero_points and fmt != 3) else None
    idx = g.integers(0, V, size=n, dtype=np.int64)
    return dict(fmt=fmt, V=V, D=D, n=n, block_size=block_size, W=W, scales=scales, zero_points=zp, indices=idx)


def ragged(num_experts: int = 128, tokens: int = 2048, k: int = 8, N: int = 1536, K: int = 2048, bits: int = 4,
           block_size: int = 32, with_zp: bool = False, seed: int = 0, counts=None) -> dict:
    """Ragged expert GEMM (the kernel test table's qmoe_ragged_mm leaf, u4 / fp16): by default the fc1 GEMM
    (2 x 768 outputs, hidden 2048) of the 128-expert top-8 "2048 / 768" MoE layer of hip-ep #1328
    "Performance", over a 2048-token prompt.  Each token picks k distinct experts
    uniformly (or `counts` gives the rows per expert); X rows grouped by expert ~ N(0, 1) fp16; codes
    uniform; fp16 scales U(0.005, 0.02); optional fp16 integer zero points."""
    g = rng(seed)
    E = num_experts
    W = packed_codes(g, E * N, K, bits).reshape(E, N, K * bits // 8)
    scales = fp16_uniform(g, (E, N, K // block_size), 0.005, 0.02)
    zp = fp16_uniform_int(g, (E, N, K // block_size), 0, (1 << bits) - 1) if with_zp else None
    if counts is None:
        picks = np.concatenate([g.choice(E, size=k, replace=False) for _ in range(tokens)])
        counts = np.bincount(picks, minlength=E)
    counts = np.asarray(counts, dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    X = fp16_normal(g, (int(offsets[-1]), K), 1.0)
    return dict(num_experts=E, N=N, K=K, bits=bits, block_size=block_size, W=W, scales=scales, zero_points=zp,
                offsets=offsets, X=X)


def nf4_nested(shape, M: int, a_dtype: int, seed: int = 0, nested_block: int = 256) -> dict:
    """NF4-style codebook GEMM with a nested absmax: the nf4 workload's codes, codebook and activations;
    absmax stored as uniform 8-bit codes into a 256-entry table evenly spaced over [-1, 1] (fp32), one fp32
    second-level scale U(0.01, 0.03) per nested_block values and offset 0.06 (so absmax spans about
    [0.03, 0.09], the plain workload's range)."""
    d = nf4(shape, M, a_dtype, seed)
    g = rng(seed + 1000)
    n = d["N"] * (d["K"] // d["block_size"])
    d.pop("absmax")
    d["absmax_q"] = g.integers(0, 256, size=(d["N"], d["K"] // d["block_size"]), dtype=np.uint8)
    d["absmax_table"] = np.linspace(-1.0, 1.0, 256).astype(np.float32)
    d["absmax2"] = f32_uniform(g, (-(-n // nested_block),), 0.01, 0.03)
    d["absmax_offset"] = 0.06
    d["nested_block"] = nested_block
    return d
