// qg_simt.cu -- SIMT blockwise-dequant GEMV / small-M GEMM for sm_103a.
//
// Computes Y[m][n] = sum_k A[m][k] * w[n][k] for small M, with w the
// blockwise dequantized weight:
//   nbits:    w = (q - zp) * s      (MatMulNBits; hip-ep #1318, "What",
//                                     Commit 1: u2 GEMV reading fp32 A and
//                                     writing fp32 C directly)
//   codebook: w = C[q] * absmax     (NF4/FP4; bitsandbytes #1979, "Summary":
//                                     codes decoded inside the GEMM, decoded
//                                     values reused across the M rows)
//   dp4a:     nbits codes against int8 activations quantized per block
//             (the int8-activation QMoE decode; hip-ep #1328, "Summary")
// Zero points: none, a scalar, an fp16 tensor, or bits-wide integers packed
// per row (staged as bytes, each block's field widened where it is used).
//
// Design (GB300-first; the pages' RDNA design -- dot2, DPP, LDS centroids --
// is prior art only):
//  * Weights stream through shared memory.  One producer warp per CTA moves
//    tiles of SR whole rows (codes + per-block parameters) with 1-D bulk
//    copies (TMA engine) into an NST-deep ring guarded by mbarriers, so the
//    consumer warps never wait on HBM latency and hold no load registers.
//  * Each consumer warp owns one K-slice and keeps the activations of that
//    slice in registers for the whole kernel.  A slice is LPR lanes x KPL
//    consecutive k; with LPR = 16 a warp works on two rows at once (one per
//    half-warp), which lets 64 codes per lane tile K = 5120 without idle
//    lanes.  A lane's codes of one row are one 16-byte shared-memory load.
//  * Unpacking costs one LOP per code: a code masked in place inside its
//    32-bit word IS an fp32 subnormal equal to q * 2^(pos - 149).  The
//    activations are pre-scaled by 2^(126 - pos) (and by a per-lane power of
//    two that normalises their magnitude), so one packed fp32x2 FMA per two
//    codes accumulates a * q exactly as an ordinary FMA would.  The zero
//    point and the scale are applied once per block per row:
//        sum_k a_k (q_k - zp) s = s * (sum_k a_k q_k - zp * sum_k a_k).
//  * int8 activations: each lane quantizes its slice per block after
//    staging and keeps it as packed int8 words that pair with the codes as
//    one AND of a code word yields them; the row loop is dp4a (four 8-bit
//    products per instruction), one flush s * sx * (sum - zp * sum q8) per
//    block.
//  * The row loop has no data-dependent branches: lanes past the end of K
//    read an in-bounds clamped address and are masked once per tile.
//  * Reductions run in a fixed order: a transposed butterfly over the lanes
//    of a row, then the K-slices of a row summed in slice order in shared
//    memory (one named barrier per row group), then (for very long K)
//    split-K partials summed in split order by a second kernel.  No atomics,
//    no dependence on timing: every call on the same inputs is
//    bit-identical (hip-ep #1328, "Why").
//  * Every wait is bounded (see qg_device.cuh): a stuck pipeline records a
//    fault bit and the kernel returns instead of hanging.
#include <algorithm>
#include <atomic>

#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr int kMaxStages = 16;
constexpr int kLutOff = 512;  // after the 2 x kMaxStages mbarriers and the abort flag
static_assert(2 * kMaxStages * 8 + 16 <= kLutOff, "shared-memory header overlaps the codebook table");

// Most consumer warps a CTA may have (launch bound), by activation rows held.
__host__ __device__ constexpr int max_consumer_warps(int mt) { return mt == 1 ? 15 : 11; }
// IT, the rows each lane group computes per tile, is 8, or 16 for full-warp
// lane groups whose stages stay small (fewer, larger stages for the producer
// warp, which competes for issue slots with the consumer warps).  A lane feeds
// IT x MT values into the per-tile transposed reduction (at most one per lane
// of its group).

enum { A_ROWS = 0, A_SWIGLU = 1 };

struct GemvArgs {
    const void *A;
    int a_dtype;
    const uint8_t *W;
    const unsigned char *params;  // fp16 scales (nbits) or fp32 absmax (codebook), [N][nb]
    const uint16_t *zp;           // fp16 zero points [N][nb] (ZP_TENSOR)
    const uint8_t *zpk;           // bits-wide zero points packed per row, rows padded to bytes (ZP_PACKED)
    int zp_mode;
    int zrow;                     // staged zero-point bytes per row: nb * 2, ceil(nb * bits / 8), or 0
    float zpv;  // zero point for ZP_UNIFORM / ZP_NONE
    const float *codebook;
    void *Y;
    int y_dtype;
    float *partial;  // split-K partials [splits][M][N], or nullptr
    int M, N, K, bs, nb, row_bytes, m0;
    int S_total, S_cta, G, SR, NST;
    int fast_tx;  // bytes of a whole aligned stage (codes + parameters [+ zero points]); 0: no fast path
    int a_off, a_rstride;  // shared-memory staging of the activations: offset, floats per staged row
    int bias_off;          // shared-memory copy of the CTA's expert bias row (QMoE), or 0: read from global
    int w_pitch, stage_bytes, s_off, z_off, red_off, stage_off, ntiles;
    unsigned *fault;
    // Slots (the experts of a QMoE decode): tile t covers rows of slot
    // t / tiles_per_slot; slot j reads the weights of expert ids[j].  Plain
    // GEMMs have one slot and ids == nullptr.
    int tiles_per_slot;
    int cps;  // CTAs per expert slot (slot mode), or 0: tiles dealt round-robin over the grid
    const int32_t *ids;
    int num_experts;
    size_t w_slot_stride, p_slot_stride, z_slot_stride;  // bytes per expert
    int a_mode;               // A_ROWS, or A_SWIGLU: slot j's activation is silu(gate) * up of g[j]
    const float *gbuf;        // A_SWIGLU: fc1 output [slots][2 * K]
    int swiglu_interleaved;
    float *out_f32;           // slot outputs [slots][N] (QMoE), with bias added
    const uint16_t *bias;     // fp16 [experts][N], or nullptr
    int bias_bulk;            // the producer stages the expert's bias row (one bulk copy), not the consumers
};

// u3: 32 codes in 3 words; bit position of code i of the group after its
// shift (see dot_group_u3), always below 21 so that the 3-bit field stays
// below the exponent.
__host__ __device__ constexpr int pos_u3(int i) {
    return i < 7 ? 3 * i
                 : (i < 10 ? 3 * i - 21
                           : (i == 10 ? 0
                                      : (i < 18 ? 3 * i - 32
                                                : (i < 21 ? 3 * i - 54
                                                          : (i == 21 ? 0 : (i < 29 ? 3 * i - 64 : 3 * i - 87))))));
}
template <int BITS>
__host__ __device__ constexpr int pos_exp(int i) {
    // bit position of code i of a 32-bit word after the single split shift
    // (a masked code must sit below bit 23, the exponent's lowest bit):
    // u2: codes 0..10 in place (bits 2i), codes 11..15 from word >> 22;
    // u4: codes 0..4 in place (bits 4i), codes 5..7 from word >> 20;
    // u8: codes 0, 1 in place (bits 8i), codes 2, 3 from word >> 16;
    // u3: position inside a 32-code group of 3 words (pos_u3).
    return BITS == 3 ? pos_u3(i)
                     : (BITS == 2 ? (i < 11 ? 2 * i : 2 * (i - 11))
                                  : (BITS == 4 ? (i < 5 ? 4 * i : 4 * (i - 5)) : (i < 2 ? 8 * i : 8 * (i - 2))));
}
// Codes per unpack unit: one 32-bit word, or a 3-word group for u3.
__host__ __device__ constexpr int unit_codes(int bits) { return bits == 3 ? 32 : 32 / bits; }
__host__ __device__ constexpr int kpl_of(int vec, int bits) { return vec * 8 / bits; }
template <int BITS>
__host__ __device__ constexpr int split_lo() { return BITS == 2 ? 11 : (BITS == 4 ? 5 : 2); }
template <int BITS>
__host__ __device__ constexpr int split_shift() { return BITS == 2 ? 22 : (BITS == 4 ? 20 : 16); }

template <int VEC>
__device__ __forceinline__ void load_words(const unsigned char *p, uint32_t (&x)[VEC / 4]) {
    if constexpr (VEC == 24) {  // u3: two 3-word groups, 8-byte aligned
        const uint2 a = *reinterpret_cast<const uint2 *>(p), b = *reinterpret_cast<const uint2 *>(p + 8),
                    c = *reinterpret_cast<const uint2 *>(p + 16);
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y; x[4] = c.x; x[5] = c.y;
    } else if constexpr (VEC == 12) {  // u3: one 3-word group, 4-byte aligned
        const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
        x[0] = q[0]; x[1] = q[1]; x[2] = q[2];
    } else if constexpr (VEC == 16) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
    } else if constexpr (VEC == 8) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        x[0] = v.x;
        x[1] = v.y;
    } else {
        x[0] = *reinterpret_cast<const uint32_t *>(p);
    }
}

// acc[m] += sum over the codes of word x of ap[m][.] * (code as subnormal)
template <int BITS, int MT, int KPL>
__device__ __forceinline__ void dot_word_nbits(uint32_t x, const float (&ap)[MT][KPL], int j, float2 (&acc)[MT]) {
    constexpr int CPW = 32 / BITS;
    constexpr int LO = split_lo<BITS>();
    constexpr int SH = split_shift<BITS>();
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    const uint32_t xh = x >> SH;
#pragma unroll
    for (int i = 0; i < CPW; i += 2) {
        const float f0 = __uint_as_float((i < LO ? x : xh) & (MASK << pos_exp<BITS>(i)));
        const float f1 = __uint_as_float((i + 1 < LO ? x : xh) & (MASK << pos_exp<BITS>(i + 1)));
#pragma unroll
        for (int m = 0; m < MT; ++m)
            acc[m] = ffma2(make_float2(ap[m][j * CPW + i], ap[m][j * CPW + i + 1]), make_float2(f0, f1), acc[m]);
    }
}

// u3: acc[m] += sum over the 32 codes of the 3-word group (w0, w1, w2) of
// ap[m][g * 32 + .] * (code as subnormal).  Code i sits at bit 3i of the
// group's 96-bit string: codes 0-6, 11-17 and 22-28 are masked in place,
// codes 7-9, 18-20 and 29-31 after one shift of their word, and codes 10 and
// 21, which cross a word boundary, after a funnel shift of two words.
template <int MT, int KPL>
__device__ __forceinline__ void dot_group_u3(uint32_t w0, uint32_t w1, uint32_t w2, const float (&ap)[MT][KPL], int g,
                                             float2 (&acc)[MT]) {
    const uint32_t a = w0 >> 21, b = w1 >> 22, c = w2 >> 23;
    const uint32_t f10 = __funnelshift_r(w0, w1, 30), f21 = __funnelshift_r(w1, w2, 31);
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t src = i < 7 ? w0 : (i < 10 ? a : (i == 10 ? f10 : (i < 18 ? w1 : (i < 21 ? b : (i == 21 ? f21 : (i < 29 ? w2 : c))))));
        f[i] = __uint_as_float(src & (7u << pos_u3(i)));
    }
#pragma unroll
    for (int i = 0; i < 32; i += 2)
#pragma unroll
        for (int m = 0; m < MT; ++m)
            acc[m] = ffma2(make_float2(ap[m][g * 32 + i], ap[m][g * 32 + i + 1]), make_float2(f[i], f[i + 1]), acc[m]);
}

// acc[m] += sum over the 8 codes of word x of ap[m][.] * C[code]; the
// codebook sits in shared memory replicated per lane (entry q of lane l at
// word q*32 + l), so the 32 lanes' lookups never share a bank.
template <int MT, int KPL>
__device__ __forceinline__ void dot_word_codebook(uint32_t x, const float (&ap)[MT][KPL], int j, float2 (&acc)[MT],
                                                  const float *lut_lane) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const float c0 = lut_lane[((x >> (4 * i)) & 15u) * 32];
        const float c1 = lut_lane[((x >> (4 * i + 4)) & 15u) * 32];
#pragma unroll
        for (int m = 0; m < MT; ++m)
            acc[m] = ffma2(make_float2(ap[m][j * 8 + i], ap[m][j * 8 + i + 1]), make_float2(c0, c1), acc[m]);
    }
}

// ---- int8 activations (WK_DP4A)
__device__ __forceinline__ int dp4a_us(uint32_t codes, uint32_t acts, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(codes), "r"(acts), "r"(c));
    return d;
}

// Activation word and byte that pair with lane-local code k: one AND of a u4
// code word yields its codes 0, 2, 4, 6 (then 1, 3, 5, 7 after a 4-bit
// shift); one of a u2 word its codes t, t + 4, t + 8, t + 12 after a 2t shift.
template <int BITS>
__host__ __device__ constexpr int dp4a_word(int k) {
    return BITS == 4 ? 2 * (k / 8) + (k % 8) % 2 : 4 * (k / 16) + (k % 16) % 4;
}
template <int BITS>
__host__ __device__ constexpr int dp4a_byte(int k) {
    return BITS == 4 ? (k % 8) / 2 : (k % 16) / 4;
}

// acc += dot of the codes of word x with their int8 activations a[0 ..]
template <int BITS>
__device__ __forceinline__ int dot_word_dp4a(uint32_t x, const uint32_t *a, int acc) {
    if constexpr (BITS == 4) {
        acc = dp4a_us(x & 0x0f0f0f0fu, a[0], acc);
        acc = dp4a_us((x >> 4) & 0x0f0f0f0fu, a[1], acc);
    } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) acc = dp4a_us((x >> (2 * t)) & 0x03030303u, a[t], acc);
    }
    return acc;
}

// The lane's KPL activations quantized to int8 per block of bs values: step
// sx = (largest magnitude of the block) / 127 (a block of more than KPL values
// spans bs / KPL neighbouring lanes), q = round-to-nearest-even(v / sx)
// clamped to +-127 (both divisions IEEE round-to-nearest), all zero for an
// all-zero block.  Packed into the words dot_word_dp4a pairs with the codes;
// per block part of the lane its step and the sum of its q.
template <int BITS, int KPL, int BPL>
__device__ __forceinline__ void prepare_dp4a(const float (&v)[KPL], int bs, uint32_t (&aq)[KPL / 4],
                                             float (&sxb)[BPL], float (&fsq)[BPL]) {
    constexpr int PART = KPL / BPL;
    const int lb = bs > KPL ? bs / KPL : 1;  // lanes per block
#pragma unroll
    for (int w = 0; w < KPL / 4; ++w) aq[w] = 0u;
#pragma unroll
    for (int b = 0; b < BPL; ++b) {
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < PART; ++i) a = fmaxf(a, fabsf(v[b * PART + i]));
        for (int off = 1; off < lb; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        const float sx = a > 0.f ? __fdiv_rn(a, 127.f) : 0.f;
        int sq = 0;
#pragma unroll
        for (int i = 0; i < PART; ++i) {
            const int k = b * PART + i;
            int q = 0;
            if (a > 0.f) q = max(-127, min(127, __float2int_rn(__fdiv_rn(v[k], sx))));
            sq += q;
            aq[dp4a_word<BITS>(k)] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * dp4a_byte<BITS>(k));
        }
        sxb[b] = sx;
        fsq[b] = static_cast<float>(sq);
    }
}

// One tile's int8-activation dot products for one lane: ITER rows, each the
// sum over the lane's blocks of s * sx * (sum q8 * q - zp * sum q8).
template <bool ZPT, int BITS, int VEC, int BPL, int ITER, int KPL = kpl_of(VEC, BITS)>
__device__ __forceinline__ void tile_dot_dp4a(const unsigned char *wp, const unsigned char *sp, const unsigned char *zpp,
                                              int row_stride, int prow_stride, int zrow_stride,
                                              const uint32_t (&aq)[KPL / 4], const float (&sxb)[BPL],
                                              const float (&fsq)[BPL], float zdef, float (&racc)[ITER]) {
    constexpr int WPL = VEC / 4;
    constexpr int AW = (32 / BITS) / 4;  // activation words per code word
#pragma unroll
    for (int i = 0; i < ITER; ++i) {
        uint32_t x[WPL];
        load_words<VEC>(wp, x);
        float rv = 0.f;
#pragma unroll
        for (int b = 0; b < BPL; ++b) {
            int acc = 0;
#pragma unroll
            for (int j = b * (WPL / BPL); j < (b + 1) * (WPL / BPL); ++j) acc = dot_word_dp4a<BITS>(x[j], &aq[j * AW], acc);
            const float s = h2f(*reinterpret_cast<const uint16_t *>(sp + b * 2));
            const float z = ZPT ? h2f(*reinterpret_cast<const uint16_t *>(zpp + b * 2)) : zdef;
            rv = fmaf(s * sxb[b], static_cast<float>(acc) - z * fsq[b], rv);
        }
        racc[i] = rv;
        wp += row_stride;
        sp += prow_stride;
        zpp += zrow_stride;
    }
}

// One tile's dot products for one lane: ITER rows (stride `row_stride` in the
// stage) times this lane's KPL codes, scaled per block; racc[i * MT + m] gets
// row i, activation row m.  ZPM: 1 a zero point per block and row in fp16,
// 2 the same packed as BITS-wide integers (zsh: the bit of the lane's first
// block in the byte zpp points at), 0 the scalar zero point folded into zah.  The lane's power-of-two activation
// scale e2 is folded into the constants: c23 = 2^23 e2c, ahat and zah are
// pre-multiplied by e2c = min(e2, 2^104) (exact scalings, and 2^23 e2c stays
// finite), so no multiply per row remains; in the rare case that a lane of
// the warp has e2 > 2^104 (activations of 2^105 or more) the remaining power
// of two `post` is applied to the row sums once per tile.
template <int ZPM, int BITS, int VEC, int MT, int BPL, int WK, int ITER, int KPL = kpl_of(VEC, BITS)>
__device__ __forceinline__ void tile_dot(const unsigned char *wp, const unsigned char *sp, const unsigned char *zpp,
                                         int zsh, int row_stride, int prow_stride, int zrow_stride,
                                         const float (&ap)[MT][KPL],
                                         const float (&c23)[MT], const float (&ahat)[MT][BPL],
                                         const float (&zah)[MT][BPL], const float *lut_lane, float (&racc)[ITER * MT],
                                         const float (&post)[MT], bool need_post) {
    constexpr int WPL = VEC / 4;
#pragma unroll
    for (int i = 0; i < ITER; ++i) {
        uint32_t x[WPL];
        load_words<VEC>(wp, x);
        float rv[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) rv[m] = 0.f;
#pragma unroll
        for (int b = 0; b < BPL; ++b) {
            float2 acc0[MT], acc1[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) acc0[m] = acc1[m] = make_float2(0.f, 0.f);
            if constexpr (BITS == 3) {  // 3-word groups of 32 codes; a block holds whole groups
                constexpr int NG = WPL / 3;
#pragma unroll
                for (int gi = b * (NG / BPL); gi < (b + 1) * (NG / BPL); ++gi) {
                    if (gi & 1) dot_group_u3<MT, KPL>(x[3 * gi], x[3 * gi + 1], x[3 * gi + 2], ap, gi, acc1);
                    else dot_group_u3<MT, KPL>(x[3 * gi], x[3 * gi + 1], x[3 * gi + 2], ap, gi, acc0);
                }
            } else
#pragma unroll
            for (int j = b * (WPL / BPL); j < (b + 1) * (WPL / BPL); ++j) {
                if constexpr (WK == WK_NBITS) {
                    if (j & 1) dot_word_nbits<BITS, MT, KPL>(x[j], ap, j, acc1);
                    else dot_word_nbits<BITS, MT, KPL>(x[j], ap, j, acc0);
                } else {
                    if (j & 1) dot_word_codebook<MT, KPL>(x[j], ap, j, acc1, lut_lane);
                    else dot_word_codebook<MT, KPL>(x[j], ap, j, acc0, lut_lane);
                }
            }
            if constexpr (WK == WK_NBITS) {
                const float s = h2f(*reinterpret_cast<const uint16_t *>(sp + b * 2));
                if constexpr (ZPM != 0) {
                    float z;
                    if constexpr (ZPM == 1) {
                        z = h2f(*reinterpret_cast<const uint16_t *>(zpp + b * 2));
                    } else {  // the block's BITS-wide field; only 3-bit fields cross a byte
                        const int bit = zsh + b * BITS, by = bit >> 3, sh = bit & 7;
                        uint32_t v = zpp[by];
                        if (BITS == 3 && sh > 5) v |= static_cast<uint32_t>(zpp[by + 1]) << 8;
                        z = static_cast<float>((v >> sh) & ((1u << BITS) - 1u));
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const float P = (acc0[m].x + acc0[m].y) + (acc1[m].x + acc1[m].y);
                        rv[m] = fmaf(s, fmaf(P, c23[m], -(z * ahat[m][b])), rv[m]);
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const float P = (acc0[m].x + acc0[m].y) + (acc1[m].x + acc1[m].y);
                        rv[m] = fmaf(s, fmaf(P, c23[m], -zah[m][b]), rv[m]);
                    }
                }
            } else {
                const float am = *reinterpret_cast<const float *>(sp + b * 4);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float P = (acc0[m].x + acc0[m].y) + (acc1[m].x + acc1[m].y);
                    rv[m] = fmaf(am, P, rv[m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) racc[i * MT + m] = rv[m];  // e2 already folded in (codebook: e2 = 1)
        wp += row_stride;
        sp += prow_stride;
        zpp += zrow_stride;
    }
    if (need_post) {  // warp-uniform
#pragma unroll
        for (int i = 0; i < ITER; ++i)
#pragma unroll
            for (int m = 0; m < MT; ++m) racc[i * MT + m] *= post[m];
    }
}

// Fixed-order transposed reduction of V values held by each lane of an
// LPR-lane group: returns, on lane l, the group sum of value index
// (l % LPR) / (LPR / V).
template <int V, int LPR>
__device__ __forceinline__ float transpose_reduce(float (&v)[V], int lane) {
    static_assert(V <= LPR, "one value per lane at most");
#pragma unroll
    for (int cnt = V, off = LPR / 2; cnt > 1; cnt >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < cnt / 2; ++j) {
            const float send = upper ? v[j] : v[j + cnt / 2];
            const float keep = upper ? v[j + cnt / 2] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float r = v[0];
#pragma unroll
    for (int off = LPR / V / 2; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

// Stage this CTA's slice of the activation rows m0 .. m0+MT-1 in shared
// memory as fp32, with coalesced 16-byte loads by all consumer threads.  The
// staged row keeps each lane's KPL values contiguous with a 16-byte pad after
// them, so that the lanes' later 16-byte reads of their own values fall in
// distinct bank groups.  Values past K or past M are zero.
template <int MT, int KPL>
__device__ __forceinline__ void stage_activations(const GemvArgs &p, float *as, int kc0, int nslots, int tid, int nthr) {
    constexpr int PITCH = KPL + 4;  // floats per lane slot
    if (p.a_dtype == 0) {
        const int nv = nslots * (KPL / 4);  // float4 per staged row
        // two groups per thread and pass, both loads issued first
        for (int i0 = tid; i0 < MT * nv; i0 += 2 * nthr) {
            float4 val[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * nthr;
                const int m = i / nv, v = i - m * nv;
                const int k = kc0 + 4 * v, am = p.m0 + m;
                val[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < MT * nv && am < p.M && k < p.K)
                    val[u] = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p.A) +
                                                                    static_cast<size_t>(am) * p.K + k));
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * nthr;
                if (i >= MT * nv) break;
                const int m = i / nv, v = i - m * nv;
                *reinterpret_cast<float4 *>(as + m * p.a_rstride + (v / (KPL / 4)) * PITCH + (v % (KPL / 4)) * 4) = val[u];
            }
        }
    } else {
        const bool f16 = p.a_dtype == 1;
        const int nv = nslots * (KPL / 8);  // 8-element groups per staged row
        // two groups per thread and pass, both loads issued first
        for (int i0 = tid; i0 < MT * nv; i0 += 2 * nthr) {
            uint4 rw[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * nthr;
                const int m = i / nv, v = i - m * nv;
                const int k = kc0 + 8 * v, am = p.m0 + m;
                rw[u] = make_uint4(0u, 0u, 0u, 0u);
                if (i < MT * nv && am < p.M && k < p.K)
                    rw[u] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.A) +
                                                                  static_cast<size_t>(am) * p.K + k));
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * nthr;
                if (i >= MT * nv) break;
                const int m = i / nv, v = i - m * nv;
                const uint32_t w4[4] = {rw[u].x, rw[u].y, rw[u].z, rw[u].w};
                float f[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint16_t lo = static_cast<uint16_t>(w4[q] & 0xFFFFu), hi = static_cast<uint16_t>(w4[q] >> 16);
                    f[2 * q] = f16 ? h2f(lo) : bf2f(lo);
                    f[2 * q + 1] = f16 ? h2f(hi) : bf2f(hi);
                }
                float *d = as + m * p.a_rstride + (v / (KPL / 8)) * PITCH + (v % (KPL / 8)) * 8;
                *reinterpret_cast<float4 *>(d) = make_float4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<float4 *>(d + 4) = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
    }
}

// Normalise a lane's activations by a power of two per row and fold in the
// code positions (MatMulNBits), computing the block sums on the way.  a_hat
// = a * 2^-E with |a_hat| < 2; a' = a_hat * 2^(126 - pos), so that a' times
// the subnormal code at pos equals a_hat * q * 2^-23 exactly.
template <int BITS, int MT, int KPL, int BPL, int WK>
__device__ __forceinline__ void prepare_activations(float (&ap)[MT][KPL], float (&e2)[MT], float (&ahat)[MT][BPL]) {
    constexpr int CPW = unit_codes(BITS);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < KPL; ++i) amax = fmaxf(amax, fabsf(ap[m][i]));
        e2[m] = 1.f;
#pragma unroll
        for (int b = 0; b < BPL; ++b) ahat[m][b] = 0.f;
        if constexpr (WK == WK_NBITS) {
            const uint32_t ex = (__float_as_uint(amax) >> 23) & 0xFFu;
            int E = ex == 0u ? -126 : (ex == 255u ? 0 : static_cast<int>(ex) - 127);
            if (amax == 0.f) E = 0;
            const float inv = exp2i(-E);
            e2[m] = exp2i(E);
#pragma unroll
            for (int i = 0; i < KPL; ++i) {
                const float ah = ap[m][i] * inv;
                ahat[m][i / (KPL / BPL)] += ah;
                ap[m][i] = ah * exp2i(126 - pos_exp<BITS>(i % CPW));
            }
        }
    }
}

// Stage the fused QMoE fc2 activation row h = silu(gate) * up of expert
// slot `sl` (gate = g[0:K], up = g[K:2K] of that slot's fc1 output, or the
// even / odd elements), in the same padded layout as stage_activations; all
// consumer threads, coalesced 16-byte loads.  Values past K are zero.
template <int KPL>
__device__ __forceinline__ void stage_swiglu_activations(const GemvArgs &p, float *as, int sl, int kc0, int nslots,
                                                         int tid, int nthr) {
    constexpr int PITCH = KPL + 4;
    const float *gs = p.gbuf + static_cast<size_t>(sl) * 2 * p.K;
    const int nv = nslots * (KPL / 4);
    for (int v = tid; v < nv; v += nthr) {
        const int k = kc0 + 4 * v;
        float h[4] = {0.f, 0.f, 0.f, 0.f};
        if (k < p.K) {
            float gate[4], up[4];
            if (p.swiglu_interleaved) {
                const float4 a = *reinterpret_cast<const float4 *>(gs + 2 * k);
                const float4 b = *reinterpret_cast<const float4 *>(gs + 2 * k + 4);
                gate[0] = a.x; up[0] = a.y; gate[1] = a.z; up[1] = a.w;
                gate[2] = b.x; up[2] = b.y; gate[3] = b.z; up[3] = b.w;
            } else {
                const float4 a = *reinterpret_cast<const float4 *>(gs + k);
                const float4 b = *reinterpret_cast<const float4 *>(gs + p.K + k);
                gate[0] = a.x; gate[1] = a.y; gate[2] = a.z; gate[3] = a.w;
                up[0] = b.x; up[1] = b.y; up[2] = b.z; up[3] = b.w;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) h[i] = gate[i] / (1.f + expf(-gate[i])) * up[i];
        }
        *reinterpret_cast<float4 *>(as + (v / (KPL / 4)) * PITCH + (v % (KPL / 4)) * 4) = make_float4(h[0], h[1], h[2], h[3]);
    }
}

// General stage fill (ragged last tile, split K, unaligned sizes, invalid
// expert): lane parts first, then the expected byte count, then the bulk parts.
template <int LPR, int VEC, int BITS>
__device__ __forceinline__ void fill_stage_general(const GemvArgs &p, unsigned char *st, const unsigned char *Wb,
                                                   const unsigned char *Pb, const unsigned char *Zb, int r0, int rows,
                                                   bool split, int kb0, int kb1, int prow, uint64_t *fullb, int lane) {
    uint32_t tx = 0;
    // codes
    if (!split) {
        const unsigned char *src = Wb + static_cast<size_t>(r0) * p.row_bytes;
        const uint32_t bytes = static_cast<uint32_t>(rows) * p.row_bytes;
        const CopyPlan cp = copy_plan(st, src, bytes);
        copy_tail_lanes(st, src, bytes, cp, lane);
        tx += cp.bulk_bytes;
    } else {
        for (int r = 0; r < rows; ++r) {
            const unsigned char *src = Wb + static_cast<size_t>(r0 + r) * p.row_bytes + kb0;
            unsigned char *dst = st + r * p.w_pitch;
            const CopyPlan cp = copy_plan(dst, src, kb1 - kb0);
            copy_tail_lanes(dst, src, kb1 - kb0, cp, lane);
            tx += cp.bulk_bytes;
        }
    }
    // block parameters (scales or absmax), then zero points
    {
        const unsigned char *src = Pb + static_cast<size_t>(r0) * prow;
        const CopyPlan cp = copy_plan(st + p.s_off, src, rows * prow);
        copy_tail_lanes(st + p.s_off, src, rows * prow, cp, lane);
        tx += cp.bulk_bytes;
    }
    if (p.zrow) {
        const unsigned char *src = Zb + static_cast<size_t>(r0) * p.zrow;
        const uint32_t zb = rows * p.zrow;
        const CopyPlan cp = copy_plan(st + p.z_off, src, zb);
        if (p.zp_mode == ZP_PACKED) {  // any byte count, any alignment: byte by byte past the bulk prefix
            for (uint32_t i = cp.bulk_bytes + lane; i < zb; i += 32) st[p.z_off + i] = __ldg(src + i);
        } else {
            copy_tail_lanes(st + p.z_off, src, zb, cp, lane);
        }
        tx += cp.bulk_bytes;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(fullb, tx);
    __syncwarp();
    // issue the bulk parts (after the expected byte count is registered)
    if (!split) {
        if (lane == 0) {
            const unsigned char *src = Wb + static_cast<size_t>(r0) * p.row_bytes;
            const CopyPlan cp = copy_plan(st, src, static_cast<uint32_t>(rows) * p.row_bytes);
            if (cp.bulk_bytes) bulk_g2s(st, src, cp.bulk_bytes, fullb);
        }
    } else {
        for (int r = lane; r < rows; r += 32) {
            const unsigned char *src = Wb + static_cast<size_t>(r0 + r) * p.row_bytes + kb0;
            unsigned char *dst = st + r * p.w_pitch;
            const CopyPlan cp = copy_plan(dst, src, kb1 - kb0);
            if (cp.bulk_bytes) bulk_g2s(dst, src, cp.bulk_bytes, fullb);
        }
    }
    if (lane == 1) {
        const unsigned char *src = Pb + static_cast<size_t>(r0) * prow;
        const CopyPlan cp = copy_plan(st + p.s_off, src, rows * prow);
        if (cp.bulk_bytes) bulk_g2s(st + p.s_off, src, cp.bulk_bytes, fullb);
    }
    if (lane == 2 && p.zrow) {
        const unsigned char *src = Zb + static_cast<size_t>(r0) * p.zrow;
        const CopyPlan cp = copy_plan(st + p.z_off, src, rows * p.zrow);
        if (cp.bulk_bytes) bulk_g2s(st + p.z_off, src, cp.bulk_bytes, fullb);
    }
}

// Producer side of a tile: add the S slice sums of each of the tile's rows in
// slice order and write the outputs (Y, split-K partials, or the QMoE slot
// outputs with the expert's bias).  `rs` holds [slice][IT * MT * H] values.
template <int MT, int LPR, int IT>
__device__ __forceinline__ void finish_tile(const GemvArgs &p, const float *rs, int s_count, int tile, int sl, int lane,
                                            const uint16_t *bias_s, int e) {
    constexpr int H = 32 / LPR;
    constexpr int RV = IT * MT;
    constexpr int VPW = RV * H;
    if (lane >= VPW) return;
    float sum = 0.f;
    for (int s = 0; s < s_count; ++s) sum += rs[s * VPW + lane];
    const int rbase = (tile - sl * p.tiles_per_slot) * p.SR;
    const int hh = lane / RV, v = lane % RV;
    const int i = v / MT, m = v % MT;
    const int row = rbase + i * H + hh;
    const int am = p.m0 + m;
    if (row >= p.N || am >= p.M) return;
    if (p.out_f32) {  // e: the slot's expert id, as the producer read it
        float o = 0.f;
        if (e >= 0 && e < p.num_experts) {
            float b = 0.f;
            if (bias_s)  // the expert's bias row, staged in shared memory by the consumer warps
                b = h2f(bias_s[row]);
            else if (p.bias)
                b = h2f(__ldg(reinterpret_cast<const unsigned short *>(p.bias) + static_cast<size_t>(e) * p.N + row));
            o = sum + b;
        }
        p.out_f32[static_cast<size_t>(sl) * p.N + row] = o;
    } else if (p.partial) {
        p.partial[(static_cast<size_t>(blockIdx.y) * p.M + am) * p.N + row] = sum;
    } else {
        store_y_elem(p.Y, p.y_dtype, static_cast<size_t>(am) * p.N + row, sum);
    }
}

template <int BITS, int VEC, int MT, int BPL, int WK, int LPR, int AM, int IT>
__global__ void __launch_bounds__((max_consumer_warps(MT) + 1) * 32, 1) gemv_kernel(const GemvArgs p) {
    constexpr int KPL = kpl_of(VEC, BITS);
    constexpr int H = 32 / LPR;         // rows a warp works on at once
    constexpr int ITER = IT;            // row iterations per tile
    constexpr int RV = IT * MT;         // values per lane in the tile's transposed reduction
    static_assert(RV <= LPR, "a lane group reduces at most one value per lane");
    constexpr int PB = WK == WK_CODEBOOK ? 4 : 2;  // bytes per block parameter
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 2 * kMaxStages * 8);
    uint64_t *bias_bar = reinterpret_cast<uint64_t *>(smem + 2 * kMaxStages * 8 + 8);  // the bias row landed
    float *lut = reinterpret_cast<float *>(smem + kLutOff);
    float *red = reinterpret_cast<float *>(smem + p.red_off);
    unsigned char *stages = smem + p.stage_off;
    const uint16_t *bias_s = p.bias_off ? reinterpret_cast<const uint16_t *>(smem + p.bias_off) : nullptr;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NWC = p.S_cta * p.G;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], p.S_cta);  // released by the warps of the group that consumed it
        }
        mbar_init(bias_bar, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    // Launched as a programmatic dependent: the set-up above overlaps the
    // preceding kernel's tail, and the next kernel may start launching as these
    // CTAs retire.  Nothing the call reads (weights, parameters, codebook,
    // activations, expert ids) or writes is touched before pdl_wait(): any
    // buffer may have been written by the preceding kernel.
    pdl_launch_dependents();
    pdl_wait();
    if constexpr (WK == WK_CODEBOOK) {
        for (int i = threadIdx.x; i < 16 * 32; i += blockDim.x) lut[i] = __ldg(p.codebook + (i >> 5));
    }
    __syncthreads();

    const bool split = gridDim.y > 1;
    const int s_begin = blockIdx.y * p.S_cta;
    const int s_count = min(p.S_cta, p.S_total - s_begin);
    const int kc0 = split ? s_begin * LPR * KPL : 0;  // first k held in a stage row
    // This CTA's tiles: t_begin, t_begin + t_stride, ... below t_end.  Plain
    // GEMMs deal tiles round-robin over the grid; with expert slots each slot
    // owns p.cps consecutive CTAs that take its tiles round-robin, so a CTA
    // works for one expert (one activation row) from start to end.
    int cta_slot = 0, t_begin = blockIdx.x, t_stride = gridDim.x, t_end = p.ntiles;
    if (p.cps > 0) {
        cta_slot = blockIdx.x / p.cps;
        t_begin = cta_slot * p.tiles_per_slot + (blockIdx.x - cta_slot * p.cps);
        t_stride = p.cps;
        t_end = min(p.ntiles, (cta_slot + 1) * p.tiles_per_slot);
    }

    // ------------------------------------------------------------ producer
    // The producer warp also finishes every tile: when a stage comes back
    // empty, the consumer warps of its group have left their slice sums of
    // that tile in the stage's reduction slot; the producer adds them in
    // slice order and writes the outputs before it refills the stage.  The
    // consumer warps therefore never wait on one another.
    if (warp == NWC) {
        const int prow = p.nb * PB;
        const int kb0 = kc0 * BITS / 8;
        const int kb1 = split ? min(p.row_bytes, (s_begin + s_count) * LPR * VEC) : p.row_bytes;
        int it = 0, slot = 0;
        uint32_t par = 1;  // parity of the empty phase that must complete before filling (it / NST)
        bool alive = true;
        // the weights are read once: evicted from L2 first, they do not push
        // out the code and operands of the launches that follow
        const uint64_t wpol = l2_evict_first();
        const int e = p.ids ? __ldg(p.ids + cta_slot) : 0;
        const bool valid = e >= 0 && e < p.num_experts;
        const int sl = cta_slot;
        // the expert's bias row for finish_tile, ahead of the weights (an
        // invalid expert's outputs are zeros and read no bias)
        const bool bias_copy = p.bias_off && p.bias_bulk && valid;
        if (bias_copy && lane == 0) {
            const uint32_t bb = static_cast<uint32_t>(p.N) * 2;
            mbar_arrive_expect_tx(bias_bar, bb);
            bulk_g2s(smem + p.bias_off, p.bias + static_cast<size_t>(e) * p.N, bb, bias_bar);
        }
        bool bias_ready = !bias_copy;
        auto wait_bias = [&]() -> bool {
            if (!bias_ready) bias_ready = mbar_wait(bias_bar, 0, abort_flag, p.fault, FAULT_WAIT_FULL);
            return bias_ready;
        };
        for (int tile = t_begin; tile < t_end; tile += t_stride, ++it) {
            if (!mbar_wait(&empty[slot], par, abort_flag, p.fault, FAULT_WAIT_EMPTY)) {
                alive = false;
                break;
            }
            const int r0 = (tile - sl * p.tiles_per_slot) * p.SR;
            const int rows = valid ? min(p.SR, p.N - r0) : 0;  // an invalid expert id copies nothing
            const int es = valid ? e : 0;
            const unsigned char *Wb = p.W + es * p.w_slot_stride;
            const unsigned char *Pb = p.params + es * p.p_slot_stride;
            const unsigned char *Zb =
                (p.zp_mode == ZP_PACKED ? p.zpk : reinterpret_cast<const unsigned char *>(p.zp)) + es * p.z_slot_stride;
            unsigned char *st = stages + static_cast<size_t>(slot) * p.stage_bytes;
            if (p.fast_tx && rows == p.SR && !split) {  // warp-uniform: a whole stage, every copy 16-byte aligned
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[slot], p.fast_tx);
                    bulk_g2s_hint(st, Wb + static_cast<size_t>(r0) * p.row_bytes, p.SR * p.row_bytes, &full[slot],
                                  wpol);
                    bulk_g2s_hint(st + p.s_off, Pb + static_cast<size_t>(r0) * prow, p.SR * prow, &full[slot], wpol);
                    if (p.zrow)
                        bulk_g2s_hint(st + p.z_off, Zb + static_cast<size_t>(r0) * p.zrow, p.SR * p.zrow, &full[slot],
                                      wpol);
                }
            } else {
                fill_stage_general<LPR, VEC, BITS>(p, st, Wb, Pb, Zb, r0, rows, split, kb0, kb1, prow, &full[slot], lane);
            }
            // finish the tile this slot held before the refill (its sums sit in
            // the reduction slot of the previous fill's parity)
            if (it >= p.NST) {
                if (!wait_bias()) {
                    alive = false;
                    break;
                }
                finish_tile<MT, LPR, IT>(p, red + (slot * 2 + par) * (p.S_cta * RV * H), s_count,
                                     tile - p.NST * t_stride, sl, lane, bias_s, e);
            }
            if (++slot == p.NST) {
                slot = 0;
                par ^= 1u;
            }
        }
        // finish the last (up to NST) tiles once their stages come back
        if (alive) {
            for (int j = max(0, it - p.NST); j < it; ++j) {
                const int sj = j % p.NST;
                if (!mbar_wait(&empty[sj], (j / p.NST) & 1, abort_flag, p.fault, FAULT_WAIT_EMPTY)) break;
                if (!wait_bias()) break;
                finish_tile<MT, LPR, IT>(p, red + (sj * 2 + ((j / p.NST) & 1)) * (p.S_cta * RV * H), s_count,
                                     t_begin + j * t_stride, sl, lane, bias_s, e);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int sigma = warp % p.S_cta, g = warp / p.S_cta;
    const int half = lane / LPR, gl = lane % LPR;  // row within the warp's pair, lane within the row
    const bool warp_active = sigma < s_count;
    const int k0 = (s_begin + sigma) * LPR * KPL + gl * KPL;
    const bool lane_active = warp_active && k0 < p.K;
    // lanes past the end of K read (in bounds) the start of the row and are masked per tile
    const int lane_boff = lane_active ? (k0 - kc0) * BITS / 8 : 0;
    const int blk0 = lane_active ? k0 / p.bs : 0;
    const float *lut_lane = lut + lane;
    const int row_stride = H * p.w_pitch;           // stage bytes between a lane's successive rows
    const int prow_stride = H * p.nb * PB;          // same for the block parameters
    const int zrow_stride = H * p.zrow;
    const int zbit0 = blk0 * BITS;  // ZP_PACKED: bit of the lane's first block in its row
    constexpr int VPW = RV * H;  // reduced values per warp and tile
    const bool writer = (gl & (LPR / RV - 1)) == 0;
    const int red_idx = sigma * VPW + half * RV + gl / (LPR / RV);

    // Activations of this lane's slice, for MT rows, kept in registers.
    float ap[MT][KPL];
    float e2[MT];
    float ahat[MT][BPL];
    float zah[MT][BPL];  // zp * ahat for a zero point that is the same for every row
    float c23[MT];       // 2^23 e2c (see tile_dot)
    float post[MT];
    bool need_post = false;
    // WK_DP4A: the lane's int8 activation words, per block part its step and sum of codes
    constexpr bool DP4A = WK == WK_DP4A;
    uint32_t aq[DP4A ? KPL / 4 : 1];
    float sxb[BPL], fsq[BPL];
    // This CTA's activation row (the same for every tile it computes): staged
    // in shared memory with coalesced loads, then each lane takes its slice.
    {
        float *as = reinterpret_cast<float *>(smem + p.a_off);
        if constexpr (AM == A_ROWS)
            stage_activations<MT, KPL>(p, as, kc0, p.S_cta * LPR, threadIdx.x, NWC * 32);
        else
            stage_swiglu_activations<KPL>(p, as, cta_slot, kc0, p.S_cta * LPR, threadIdx.x, NWC * 32);
        if (p.bias_off && !p.bias_bulk) {  // this CTA's expert bias row, for the producer's finish_tile
            uint16_t *bs = reinterpret_cast<uint16_t *>(smem + p.bias_off);
            const int be = p.ids ? __ldg(p.ids + cta_slot) : 0;
            const bool bvalid = be >= 0 && be < p.num_experts;
            const uint16_t *src = p.bias + static_cast<size_t>(bvalid ? be : 0) * p.N;
            if ((p.N & 7) == 0 && (reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0) {  // 16-byte aligned rows
                const int nv = p.N / 8;
#pragma unroll 4
                for (int i = threadIdx.x; i < nv; i += NWC * 32)
                    reinterpret_cast<uint4 *>(bs)[i] =
                        bvalid ? __ldg(reinterpret_cast<const uint4 *>(src) + i) : make_uint4(0u, 0u, 0u, 0u);
            } else {
#pragma unroll 4
                for (int i = threadIdx.x; i < p.N; i += NWC * 32) bs[i] = bvalid ? __ldg(src + i) : uint16_t(0);
            }
        }
        named_bar_sync(1, NWC * 32);
        const float *mine = as + (sigma * LPR + gl) * (KPL + 4);
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < KPL / 4; ++j) {
                const float4 v = *reinterpret_cast<const float4 *>(mine + m * p.a_rstride + 4 * j);
                ap[m][4 * j] = v.x;
                ap[m][4 * j + 1] = v.y;
                ap[m][4 * j + 2] = v.z;
                ap[m][4 * j + 3] = v.w;
            }
        if constexpr (DP4A) {
            static_assert(!DP4A || MT == 1, "int8 activations: one activation row");
            prepare_dp4a<BITS, KPL, BPL>(ap[0], p.bs, aq, sxb, fsq);
        } else {
            prepare_activations<BITS, MT, KPL, BPL, WK>(ap, e2, ahat);
            bool big = false;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float e2c = fminf(e2[m], __uint_as_float((104u + 127u) << 23));  // min(e2, 2^104)
                post[m] = e2[m] / e2c;                                    // 1, or the power of two left over
                big |= post[m] != 1.f;
                c23[m] = 8388608.f * e2c;  // 2^23 e2c: exact, finite
#pragma unroll
                for (int b = 0; b < BPL; ++b) {
                    zah[m][b] = (p.zpv * ahat[m][b]) * e2c;
                    ahat[m][b] *= e2c;
                }
            }
            need_post = __any_sync(0xffffffffu, big);
        }
    }
    const int e = p.ids ? __ldg(p.ids + cta_slot) : 0;
    const bool valid = e >= 0 && e < p.num_experts;

    // group g consumes the CTA's tiles g, g + G, g + 2G, ... (stage `it` holds
    // tile it); ring slot and phase parity are advanced incrementally
    int slot = g;
    uint32_t par = 0;
    while (slot >= p.NST) {
        slot -= p.NST;
        par ^= 1u;
    }
    for (int tile = t_begin + g * t_stride; tile < t_end; tile += p.G * t_stride) {
        const bool ok = mbar_wait(&full[slot], par, abort_flag, p.fault, FAULT_WAIT_FULL);
        const unsigned char *st = stages + static_cast<size_t>(slot) * p.stage_bytes;
        float racc[RV];
#pragma unroll
        for (int v = 0; v < RV; ++v) racc[v] = 0.f;
        if (ok && valid) {  // warp-uniform
            const unsigned char *wp = st + half * p.w_pitch + lane_boff;  // this lane's first row is `half`
            const unsigned char *sp = st + p.s_off + (half * p.nb + blk0) * PB;
            const unsigned char *zrw = st + p.z_off + half * p.zrow;  // the lane's first row of zero points
            if constexpr (DP4A) {
                if (p.zp_mode == ZP_TENSOR)
                    tile_dot_dp4a<true, BITS, VEC, BPL, ITER>(wp, sp, zrw + blk0 * 2, row_stride, prow_stride,
                                                              zrow_stride, aq, sxb, fsq, p.zpv, racc);
                else
                    tile_dot_dp4a<false, BITS, VEC, BPL, ITER>(wp, sp, zrw, row_stride, prow_stride, zrow_stride, aq,
                                                               sxb, fsq, p.zpv, racc);
            } else if (WK == WK_NBITS && p.zp_mode == ZP_TENSOR)
                tile_dot<1, BITS, VEC, MT, BPL, WK, ITER>(wp, sp, zrw + blk0 * 2, 0, row_stride, prow_stride,
                                                         zrow_stride, ap, c23, ahat, zah, lut_lane, racc, post,
                                                         need_post);
            else if (WK == WK_NBITS && AM == A_ROWS && p.zp_mode == ZP_PACKED)
                tile_dot<2, BITS, VEC, MT, BPL, WK, ITER>(wp, sp, zrw + (zbit0 >> 3), zbit0 & 7, row_stride,
                                                         prow_stride, zrow_stride, ap, c23, ahat, zah, lut_lane, racc,
                                                         post, need_post);
            else
                tile_dot<0, BITS, VEC, MT, BPL, WK, ITER>(wp, sp, zrw, 0, row_stride, prow_stride, zrow_stride, ap,
                                                         c23, ahat, zah, lut_lane, racc, post, need_post);
#pragma unroll
            for (int v = 0; v < RV; ++v) racc[v] = lane_active ? racc[v] : 0.f;
        }
        // lane l now holds, for row half `half`, the slice sum of value (l % LPR) / (LPR / RV)
        const float tot = transpose_reduce<RV, LPR>(racc, lane);
        if (writer) red[(slot * 2 + par) * (p.S_cta * VPW) + red_idx] = tot;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);  // releases the stage and this warp's slice sums

        slot += p.G;
        while (slot >= p.NST) {
            slot -= p.NST;
            par ^= 1u;
        }
    }
}

// Y = sum over splits of the partials, in split order.
__global__ void splitk_reduce_kernel(const float *__restrict__ partial, int splits, size_t MN, void *Y, int y_dtype) {
    pdl_wait();
    pdl_launch_dependents();
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < MN;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float s = 0.f;
        for (int sp = 0; sp < splits; ++sp) s += partial[sp * MN + i];
        store_y_elem(Y, y_dtype, i, s);
    }
}

// QMoE: y[r] = fp16( sum_j w_j * o_j[r] ), slots summed in slot order; a slot
// whose expert id is out of range adds nothing and sets *status to 1.
__global__ void qmoe_combine_kernel(const float *__restrict__ o, const int32_t *__restrict__ ids,
                                    const float *__restrict__ w, int k, int num_experts, int H, uint16_t *y,
                                    int *status) {
    pdl_wait();
    pdl_launch_dependents();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    int bad = 0;
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
        const int e = __ldg(ids + j);
        if (e < 0 || e >= num_experts) {
            bad = 1;
            continue;
        }
        if (r < H) acc = fmaf(__ldg(w + j), o[static_cast<size_t>(j) * H + r], acc);
    }
    if (r < H) y[r] = f2h(acc);
    if (status && r == 0) *status = bad;
}

// ---------------------------------------------------------------- host side
struct Cfg {
    int vec, lpr, mt, bpl;
    int S_total, S_cta, splits, G, SR, NST;
    int w_pitch, stage_bytes, s_off, z_off, red_off, stage_off, smem, ntiles, grid_x;
    int a_off, a_rstride, bias_off, iter;
};

inline int round_up(int x, int a) { return (x + a - 1) / a * a; }

// Static launch table: a pure function of the shape (no timing, no tuning).
// Per vector width / row-lane layout the cost is estimated as the issue work
// per useful code: idle lanes of the last K-slice, the per-row bookkeeping
// (about 12 instructions per lane and row) and, for layouts needing more
// slices than fit in one CTA, a split-K penalty.
// zrow: bytes of zero points staged per row (0: none).
bool choose_cfg(int M, int N, int K, int bits, int bs, int kind, int zrow, Cfg &c, int bias_bytes = 0) {
    const DeviceInfo &di = device_info();
    c.mt = M <= 1 ? 1 : (M <= 2 ? 2 : 4);
    if (bits == 3) c.mt = std::min(c.mt, 2);  // u3 groups of 32 codes: at most 2 activation rows in registers
    const int maxw = max_consumer_warps(c.mt);
    const int row_bytes = K * bits / 8;
    const int pb = kind == WK_CODEBOOK ? 4 : 2;
    const int nb = K / bs;
    struct Cand { int vec, lpr; };
    Cand cands[4];
    int ncand = 0;
    if (bits == 2) {
        if (c.mt == 1) { cands[ncand++] = {16, 32}; cands[ncand++] = {16, 16}; cands[ncand++] = {8, 32}; }
        else if (c.mt == 2) { cands[ncand++] = {8, 32}; cands[ncand++] = {8, 16}; cands[ncand++] = {4, 32}; }
        else { cands[ncand++] = {4, 32}; }
    } else if (bits == 3) {  // 3-word groups of 32 codes: 24 bytes (64 codes) or 12 bytes per lane
        if (c.mt == 1) { cands[ncand++] = {24, 32}; cands[ncand++] = {24, 16}; cands[ncand++] = {12, 32}; }
        else { cands[ncand++] = {12, 32}; cands[ncand++] = {12, 16}; }
    } else if (bits == 8) {  // 16 codes per 16-byte load
        if (c.mt <= 2) { cands[ncand++] = {16, 32}; cands[ncand++] = {16, 16}; }
        else { cands[ncand++] = {16, 32}; }
    } else {
        if (c.mt <= 2) { cands[ncand++] = {16, 32}; cands[ncand++] = {16, 16}; cands[ncand++] = {8, 32}; }
        else { cands[ncand++] = {8, 32}; cands[ncand++] = {4, 32}; }
    }
    double best = -1.0;
    c.vec = 0;
    for (int i = 0; i < ncand; ++i) {
        const int v = cands[i].vec, l = cands[i].lpr;
        if (row_bytes % v) continue;
        if (kind == WK_DP4A && v != 16) continue;  // int8 activations: 16-byte units only
        const int kpl = v * 8 / bits;
        const int sw = l * kpl;
        const int st = (K + sw - 1) / sw;
        const double lane_eff = static_cast<double>(K) / (static_cast<double>(st) * sw);
        const double row_eff = static_cast<double>(kpl) / (kpl + 12.0);
        const double split_pen = st > maxw ? 0.8 : 1.0;
        const double score = lane_eff * row_eff * split_pen;
        if (score > best + 1e-9) {
            best = score;
            c.vec = v;
            c.lpr = l;
        }
    }
    if (!c.vec) return false;
    const int kpl = c.vec * 8 / bits;
    c.bpl = kpl > bs ? kpl / bs : 1;
    c.S_total = (K + c.lpr * kpl - 1) / (c.lpr * kpl);
    c.splits = (c.S_total + maxw - 1) / maxw;
    c.S_cta = (c.S_total + c.splits - 1) / c.splits;
    // a stage holds one tile of SR rows; the G row groups of consumer warps take
    // stages in turn, so the stage size does not grow with the number of warps
    // 16 rows per lane group for MatMulNBits when a lane holds 32 activations and
    // the 16-row stage stays small (the codebook kernel is slower with them); the
    // kernels instantiated with 16 are listed in dispatch()
    c.iter = (c.lpr == 32 && c.mt == 1 && row_bytes <= 4096 &&
              ((kind == WK_NBITS && ((bits == 4 && c.vec == 16) || (bits == 2 && c.vec == 8))) ||
               (kind == WK_DP4A && bits == 4 && c.vec == 16)))
                 ? 16
                 : 8;
    c.SR = c.iter * (32 / c.lpr);
    c.G = std::max(1, maxw / c.S_cta);
    c.w_pitch = c.splits > 1 ? round_up(c.S_cta * c.lpr * c.vec, 16) : row_bytes;
    // activation staging: MT rows x S_cta slices x LPR lanes x (KPL + 4) floats
    c.a_off = round_up(kLutOff + (kind == WK_CODEBOOK ? 16 * 32 * 4 : 0), 128);
    c.a_rstride = c.S_cta * c.lpr * (kpl + 4);
    c.bias_off = bias_bytes ? round_up(c.a_off + c.mt * c.a_rstride * 4, 128) : 0;
    c.stage_off = round_up(c.a_off + c.mt * c.a_rstride * 4 + (bias_bytes ? 128 + bias_bytes : 0), 1024);
    const int budget = di.max_smem_optin - c.stage_off;
    c.s_off = round_up(c.SR * c.w_pitch, 128);
    c.z_off = c.s_off + round_up(c.SR * nb * pb, 128);
    c.stage_bytes = c.z_off + (zrow ? round_up(c.SR * zrow, 128) : 0);
    // each stage also has a reduction slot: S_cta slices x iter x MT x H sums
    const int red_slot = c.S_cta * c.iter * c.mt * (32 / c.lpr) * 4;
    const int nfit = std::min(kMaxStages, budget / (c.stage_bytes + 2 * red_slot));
    if (nfit < 2) return false;
    // Ring slots are owned by row groups: slot s serves group s % G only, so
    // NST is a multiple of G.  A group then waits on a slot's phase k only
    // after it has itself consumed phase k - 1 of that slot.  (If slots were
    // shared, stage fills that land out of order could let a group wait on
    // phase k while phase k - 1 is still pending, whose parity the barrier
    // reports as complete.)  At least two stages per group when possible.
    c.G = std::max(1, std::min(c.G, nfit / 2));
    c.NST = nfit - nfit % c.G;
    c.red_off = c.stage_off + c.NST * c.stage_bytes;
    c.smem = c.red_off + 2 * c.NST * red_slot;  // reduction slots double-buffered by fill parity
    c.ntiles = (N + c.SR - 1) / c.SR;
    c.grid_x = std::min(c.ntiles, di.sm_count);
    (void)M;
    return true;
}

template <int BITS, int VEC, int MT, int BPL, int WK, int LPR, int AM, int IT = 8>
cudaError_t launch_one(const GemvArgs &a, const Cfg &c, cudaStream_t s) {
    auto kern = gemv_kernel<BITS, VEC, MT, BPL, WK, LPR, AM, IT>;
    static std::atomic<unsigned> configured{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned bit = 1u << (dev & 31);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             device_info().max_smem_optin);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    dim3 grid(c.grid_x, c.splits);
    dim3 block((c.S_cta * c.G + 1) * 32);
    const cudaError_t e = launch_pdl(kern, grid, block, c.smem, s, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t dispatch(const GemvArgs &a, const Cfg &c, int bits, int kind, cudaStream_t s) {
#define QG_CASE(B, V, MT_, BPL_, WK_, L_)                                                                 \
    if (bits == B && c.vec == V && c.mt == MT_ && c.bpl == BPL_ && kind == WK_ && c.lpr == L_) \
        return a.a_mode == A_ROWS ? launch_one<B, V, MT_, BPL_, WK_, L_, A_ROWS>(a, c, s) : cudaErrorNotSupported;
#define QG_CASE_SW(B, V, BPL_, L_)                                                                    \
    if (bits == B && c.vec == V && c.mt == 1 && c.bpl == BPL_ && kind == WK_NBITS && c.lpr == L_ && \
        a.a_mode == A_SWIGLU)                                                                      \
        return launch_one<B, V, 1, BPL_, WK_NBITS, L_, A_SWIGLU>(a, c, s);
    // 16 rows per tile (see choose_cfg): full-warp lane groups holding 32 activations
    if (c.iter == 16) {
        if (kind == WK_DP4A) {
            if (c.mt == 1 && c.lpr == 32 && c.bpl == 1 && bits == 4 && c.vec == 16)
                return a.a_mode == A_ROWS ? launch_one<4, 16, 1, 1, WK_DP4A, 32, A_ROWS, 16>(a, c, s)
                                          : launch_one<4, 16, 1, 1, WK_DP4A, 32, A_SWIGLU, 16>(a, c, s);
            return cudaErrorNotSupported;
        }
        if (c.mt == 1 && c.lpr == 32 && c.bpl == 1) {
            if (bits == 4 && c.vec == 16 && kind == WK_NBITS)
                return a.a_mode == A_ROWS ? launch_one<4, 16, 1, 1, WK_NBITS, 32, A_ROWS, 16>(a, c, s)
                                          : launch_one<4, 16, 1, 1, WK_NBITS, 32, A_SWIGLU, 16>(a, c, s);
            if (bits == 2 && c.vec == 8 && kind == WK_NBITS)
                return a.a_mode == A_ROWS ? launch_one<2, 8, 1, 1, WK_NBITS, 32, A_ROWS, 16>(a, c, s)
                                          : launch_one<2, 8, 1, 1, WK_NBITS, 32, A_SWIGLU, 16>(a, c, s);
        }
        return cudaErrorNotSupported;
    }
    // int8-activation QMoE (fc1 rows of x, fc2 SwiGLU rows)
#define QG_CASE_D4(B, BPL_, L_)                                                                        \
    if (kind == WK_DP4A && bits == B && c.vec == 16 && c.mt == 1 && c.bpl == BPL_ && c.lpr == L_)     \
        return a.a_mode == A_ROWS ? launch_one<B, 16, 1, BPL_, WK_DP4A, L_, A_ROWS>(a, c, s)           \
                                  : launch_one<B, 16, 1, BPL_, WK_DP4A, L_, A_SWIGLU>(a, c, s);
    QG_CASE_D4(4, 1, 32)
    QG_CASE_D4(4, 1, 16)
    QG_CASE_D4(2, 1, 32)
    QG_CASE_D4(2, 2, 32)
    QG_CASE_D4(2, 1, 16)
    QG_CASE_D4(2, 2, 16)
#undef QG_CASE_D4
    if (kind == WK_DP4A) return cudaErrorNotSupported;
    // fused QMoE fc2 (activations = SwiGLU of fc1's output)
    QG_CASE_SW(4, 16, 1, 32)
    QG_CASE_SW(4, 16, 1, 16)
    QG_CASE_SW(4, 8, 1, 32)
    QG_CASE_SW(2, 16, 1, 32)
    QG_CASE_SW(2, 16, 1, 16)
    QG_CASE_SW(2, 16, 2, 32)
    QG_CASE_SW(2, 16, 2, 16)
    QG_CASE_SW(2, 8, 1, 32)
    // MatMulNBits u2
    QG_CASE(2, 16, 1, 1, WK_NBITS, 32)
    QG_CASE(2, 16, 1, 1, WK_NBITS, 16)
    QG_CASE(2, 16, 1, 2, WK_NBITS, 32)
    QG_CASE(2, 16, 1, 2, WK_NBITS, 16)
    QG_CASE(2, 8, 1, 1, WK_NBITS, 32)
    QG_CASE(2, 8, 2, 1, WK_NBITS, 32)
    QG_CASE(2, 8, 2, 1, WK_NBITS, 16)
    QG_CASE(2, 4, 2, 1, WK_NBITS, 32)
    QG_CASE(2, 4, 4, 1, WK_NBITS, 32)
    // MatMulNBits u3
    QG_CASE(3, 24, 1, 1, WK_NBITS, 32)
    QG_CASE(3, 24, 1, 1, WK_NBITS, 16)
    QG_CASE(3, 24, 1, 2, WK_NBITS, 32)
    QG_CASE(3, 24, 1, 2, WK_NBITS, 16)
    QG_CASE(3, 12, 1, 1, WK_NBITS, 32)
    QG_CASE(3, 12, 2, 1, WK_NBITS, 32)
    QG_CASE(3, 12, 2, 1, WK_NBITS, 16)
    // MatMulNBits u8
    QG_CASE(8, 16, 1, 1, WK_NBITS, 32)
    QG_CASE(8, 16, 1, 1, WK_NBITS, 16)
    QG_CASE(8, 16, 2, 1, WK_NBITS, 32)
    QG_CASE(8, 16, 2, 1, WK_NBITS, 16)
    QG_CASE(8, 16, 4, 1, WK_NBITS, 32)
    // MatMulNBits u4
    QG_CASE(4, 16, 1, 1, WK_NBITS, 32)
    QG_CASE(4, 16, 1, 1, WK_NBITS, 16)
    QG_CASE(4, 8, 1, 1, WK_NBITS, 32)
    QG_CASE(4, 16, 2, 1, WK_NBITS, 32)
    QG_CASE(4, 16, 2, 1, WK_NBITS, 16)
    QG_CASE(4, 8, 2, 1, WK_NBITS, 32)
    QG_CASE(4, 8, 4, 1, WK_NBITS, 32)
    QG_CASE(4, 4, 4, 1, WK_NBITS, 32)
    // codebook (NF4 / FP4)
    QG_CASE(4, 16, 1, 1, WK_CODEBOOK, 32)
    QG_CASE(4, 16, 1, 1, WK_CODEBOOK, 16)
    QG_CASE(4, 8, 1, 1, WK_CODEBOOK, 32)
    QG_CASE(4, 16, 2, 1, WK_CODEBOOK, 32)
    QG_CASE(4, 16, 2, 1, WK_CODEBOOK, 16)
    QG_CASE(4, 8, 2, 1, WK_CODEBOOK, 32)
    QG_CASE(4, 8, 4, 1, WK_CODEBOOK, 32)
    QG_CASE(4, 4, 4, 1, WK_CODEBOOK, 32)
#undef QG_CASE
#undef QG_CASE_SW
    return cudaErrorNotSupported;
}

// Whole-stage byte count for the producer's fast path, or 0 when a whole
// stage's copies are not all multiples of 16 bytes (then every stage takes the
// general path).  Base pointers and expert strides must be 16-byte multiples.
int fast_stage_tx(const GemvArgs &a, const Cfg &c, int pb) {
    if (c.splits > 1) return 0;
    const long long code = static_cast<long long>(c.SR) * a.row_bytes;
    const long long par = static_cast<long long>(c.SR) * a.nb * pb;
    const long long zp = static_cast<long long>(c.SR) * a.zrow;
    if (a.zp_mode == ZP_PACKED && (reinterpret_cast<uintptr_t>(a.zpk) & 15u)) return 0;
    if (code % 16 || par % 16 || zp % 16) return 0;
    if (a.ids && (a.w_slot_stride % 16 || a.p_slot_stride % 16 || a.z_slot_stride % 16)) return 0;
    return static_cast<int>(code + par + zp);
}

void fill_args(GemvArgs &a, const Cfg &c) {
    a.S_total = c.S_total;
    a.S_cta = c.S_cta;
    a.G = c.G;
    a.SR = c.SR;
    a.NST = c.NST;
    a.w_pitch = c.w_pitch;
    a.stage_bytes = c.stage_bytes;
    a.s_off = c.s_off;
    a.z_off = c.z_off;
    a.red_off = c.red_off;
    a.a_off = c.a_off;
    a.a_rstride = c.a_rstride;
    a.bias_off = c.bias_off;
    a.stage_off = c.stage_off;
    a.fault = fault_word();
}

}  // namespace

size_t simt_workspace_bytes(int M, int N, int K, int bits, int bs) {
    Cfg c;
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    // the zero-point mode and the weight kind do not change the split count
    if (!choose_cfg(M, N, K, bits, bs, WK_NBITS, (K / bs) * 2, c)) return 0;
    return c.splits > 1 ? static_cast<size_t>(c.splits) * M * N * sizeof(float) : 0;
}

// Staged zero-point bytes per weight row of a request.
static int zp_row_bytes(const GemmProblem &p) {
    const int nb = p.K / p.bs;
    return p.zp_mode == ZP_TENSOR ? nb * 2 : (p.zp_mode == ZP_PACKED ? (nb * p.bits + 7) / 8 : 0);
}

bool simt_packed_zp_ok(const GemmProblem &p) {
    Cfg c;
    return p.kind == WK_NBITS && p.zp_mode == ZP_PACKED && p.zp_packed &&
           choose_cfg(p.M, p.N, p.K, p.bits, p.bs, p.kind, zp_row_bytes(p), c);
}

cudaError_t simt_gemm(const GemmProblem &p, void *ws, size_t ws_bytes, cudaStream_t s) {
    Cfg c;
    if (p.zp_mode == ZP_PACKED && (p.kind != WK_NBITS || !p.zp_packed)) return cudaErrorNotSupported;
    if (!choose_cfg(p.M, p.N, p.K, p.bits, p.bs, p.kind, zp_row_bytes(p), c)) return cudaErrorNotSupported;
    GemvArgs a{};
    a.A = p.A;
    a.a_dtype = p.a_dtype;
    a.W = p.W;
    a.params = p.kind == WK_CODEBOOK ? reinterpret_cast<const unsigned char *>(p.absmax)
                                     : reinterpret_cast<const unsigned char *>(p.scales);
    a.zp = p.zp;
    a.zpk = p.zp_packed;
    a.zp_mode = p.zp_mode;
    a.zrow = zp_row_bytes(p);
    a.zpv = p.uniform_zp;
    a.codebook = p.codebook;
    a.Y = p.Y;
    a.y_dtype = p.y_dtype;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.bs = p.bs;
    a.nb = p.K / p.bs;
    a.row_bytes = p.K * p.bits / 8;
    fill_args(a, c);
    a.ntiles = c.ntiles;
    a.tiles_per_slot = c.ntiles;
    a.ids = nullptr;
    a.num_experts = 1;
    a.a_mode = A_ROWS;
    if (c.splits > 1) {
        const size_t need = static_cast<size_t>(c.splits) * p.M * p.N * sizeof(float);
        if (!ws || ws_bytes < need) return cudaErrorInvalidValue;  // checked by the caller first
        a.partial = static_cast<float *>(ws);
    }
    a.fast_tx = fast_stage_tx(a, c, p.kind == WK_CODEBOOK ? 4 : 2);
    for (int m0 = 0; m0 < p.M; m0 += c.mt) {
        a.m0 = m0;
        cudaError_t e = dispatch(a, c, p.bits, p.kind, s);
        if (e != cudaSuccess) return e;
    }
    if (c.splits > 1) {
        const size_t MN = static_cast<size_t>(p.M) * p.N;
        const int threads = 256;
        const int blocks = static_cast<int>(std::min<size_t>((MN + threads - 1) / threads, 4096));
        const cudaError_t e = launch_pdl(splitk_reduce_kernel, dim3(blocks), dim3(threads), 0, s,
                                         static_cast<const float *>(a.partial), c.splits, MN, p.Y, p.y_dtype);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    return cudaSuccess;
}

size_t qmoe_workspace_bytes(int k, int hidden, int inter) {
    if (k <= 0 || hidden <= 0 || inter <= 0) return 0;
    const size_t g = (static_cast<size_t>(k) * 2 * inter * sizeof(float) + 255) / 256 * 256;
    const size_t o = (static_cast<size_t>(k) * hidden * sizeof(float) + 255) / 256 * 256;
    return g + o;
}

// The int8-activation configurations dispatch() has a kernel for.
static bool dp4a_dispatchable(const Cfg &c, int bits) {
    if (c.mt != 1 || c.vec != 16) return false;
    if (c.iter == 16) return bits == 4 && c.lpr == 32 && c.bpl == 1;
    return (c.lpr == 32 || c.lpr == 16) && (bits == 4 ? c.bpl == 1 : (c.bpl == 1 || c.bpl == 2));
}

// The stage plan of one of the decode's two GEMVs (fc1 or fc2).
static bool qmoe_cfg(const QmoeProblem &q, bool fc1, int kind, Cfg &c) {
    const int N = fc1 ? 2 * q.inter : q.hidden;
    const int K = fc1 ? q.hidden : q.inter;
    const uint16_t *zp = fc1 ? q.fc1_zp : q.fc2_zp;
    // the expert's bias row is staged in shared memory when it is small enough
    const uint16_t *bias = fc1 ? q.fc1_bias : q.fc2_bias;
    const int bias_bytes = bias && N <= 16384 ? (N * 2 + 15) / 16 * 16 : 0;
    return choose_cfg(1, N, K, q.bits, q.bs, kind, zp ? (K / q.bs) * 2 : 0, c, bias_bytes) && c.splits == 1;
}

bool qmoe_dp4a_simt_ok(const QmoeProblem &q) {
    Cfg c1, c2;
    return qmoe_cfg(q, true, WK_DP4A, c1) && dp4a_dispatchable(c1, q.bits) && qmoe_cfg(q, false, WK_DP4A, c2) &&
           dp4a_dispatchable(c2, q.bits);
}

cudaError_t qmoe_decode(const QmoeProblem &q, void *ws, cudaStream_t s, bool dp4a) {
    const DeviceInfo &di = device_info();
    const int kind = dp4a ? WK_DP4A : WK_NBITS;
    float *g = static_cast<float *>(ws);
    float *o = reinterpret_cast<float *>(static_cast<char *>(ws) +
                                         (static_cast<size_t>(q.k) * 2 * q.inter * sizeof(float) + 255) / 256 * 256);
    const int mid = 1 << (q.bits - 1);
    for (int stage = 0; stage < 2; ++stage) {
        const bool fc1 = stage == 0;
        const int N = fc1 ? 2 * q.inter : q.hidden;
        const int K = fc1 ? q.hidden : q.inter;
        const uint16_t *zp = fc1 ? q.fc1_zp : q.fc2_zp;
        Cfg c;
        if (!qmoe_cfg(q, fc1, kind, c)) return cudaErrorNotSupported;
        GemvArgs a{};
        a.A = q.x;
        a.a_dtype = 1;  // fp16 token
        a.W = fc1 ? q.fc1_w : q.fc2_w;
        a.params = reinterpret_cast<const unsigned char *>(fc1 ? q.fc1_scales : q.fc2_scales);
        a.zp = zp;
        a.zp_mode = zp ? ZP_TENSOR : ZP_NONE;
        a.zrow = zp ? (K / q.bs) * 2 : 0;
        a.zpv = static_cast<float>(mid);
        a.M = 1;
        a.N = N;
        a.K = K;
        a.bs = q.bs;
        a.nb = K / q.bs;
        a.row_bytes = K * q.bits / 8;
        a.m0 = 0;
        fill_args(a, c);
        a.tiles_per_slot = c.ntiles;
        a.ntiles = c.ntiles * q.k;
        a.ids = q.ids;
        a.num_experts = q.num_experts;
        a.w_slot_stride = static_cast<size_t>(N) * a.row_bytes;
        a.p_slot_stride = static_cast<size_t>(N) * a.nb * 2;
        a.z_slot_stride = static_cast<size_t>(N) * a.nb * 2;
        a.a_mode = fc1 ? A_ROWS : A_SWIGLU;
        a.gbuf = g;
        a.swiglu_interleaved = q.swiglu_interleaved;
        a.out_f32 = fc1 ? g : o;
        a.bias = fc1 ? q.fc1_bias : q.fc2_bias;
        // one bulk copy of the expert's bias row when its rows are 16-byte runs
        a.bias_bulk = a.bias && (N * 2) % 16 == 0 && (reinterpret_cast<uintptr_t>(a.bias) & 15u) == 0;
        // each expert slot owns an equal share of the SMs (its activation row is staged once per CTA)
        a.cps = std::max(1, di.sm_count / q.k);
        c.grid_x = q.k * a.cps;
        a.fast_tx = fast_stage_tx(a, c, 2);
        cudaError_t e = dispatch(a, c, q.bits, kind, s);
        if (e != cudaSuccess) return e;
    }
    const int threads = 256;
    const cudaError_t e = launch_pdl(qmoe_combine_kernel, dim3((q.hidden + threads - 1) / threads), dim3(threads), 0, s,
                                     static_cast<const float *>(o), q.ids, q.weights, q.k, q.num_experts, q.hidden,
                                     q.y, q.status);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qg
