// qg_qmoe_dp4a.cu -- fused single-token QMoE decode with int8 activations.
//
// hip-ep pull request #1328 ("Summary": a dp4a form of the fused decode sits beside the fp one;
// "Test plan": fp and dp4a x block size x zero points x bias).  The
// activation vector of each GEMV (x before fc1, h = silu(gate) * up before
// fc2) is quantized per block of bs values to int8 (largest magnitude -> 127,
// fp32 steps, ties to even); each output is then
//     sum over blocks b of  s[r,b] * sx[b] * ( sum q8 * q  -  zp[r,b] * sum q8 )
// with the integer sums formed by dp4a (four 8-bit products per instruction).
//
// This file holds the decode for the shapes the SIMT GEMV's int8-activation
// kind (qg_simt.cu) has no plan for -- rows that are not a multiple of 16
// bytes, or whose stages do not fit.  Kernels: two GEMVs (fc1 with the
// quantization of x in its prologue, fc2 with SwiGLU and the quantization of
// h in its prologue) and a combine that sums the slots in slot order.  Each
// GEMV CTA serves one expert slot: it quantizes the slot's activation vector
// into shared memory, then its warps stream weight rows with coalesced vector
// loads (lane l takes the row's units l, l + 32, ...), two rows at a time so
// that their loads overlap.
// The quantized activations are stored in the byte order that pairs them with
// the codes as they come out of one AND of a code word: for u4, lanes of
// (w & 0x0f0f0f0f) hold codes 0, 2, 4, 6 of the word and (w >> 4) & ... codes
// 1, 3, 5, 7; for u2, (w >> 2t) & 0x03030303 holds codes t, t+4, t+8, t+12.
#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr int kDThreads = 512;
constexpr int kDWarps = kDThreads / 32;
struct Dp4aGemv {
    const uint16_t *x;        // fc1: fp16 activations [K]
    const float *g;           // fc2: fc1 outputs [slots][2K] (gate/up), or null
    int swiglu_interleaved;
    const int32_t *ids;
    int num_experts;
    const uint8_t *w;         // [E][N][K*bits/8]
    const uint16_t *scales;   // [E][N][K/bs]
    const uint16_t *zp;       // same, or null (midpoint)
    const uint16_t *bias;     // [E][N], or null
    int N, K, bs, cps;
    float *out;               // [slots][N]
};

__device__ __forceinline__ int dp4a_us(uint32_t codes, uint32_t acts, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(codes), "r"(acts), "r"(c));
    return d;
}

// Byte offset of activation k in the permuted shared-memory layout.
template <int BITS>
__device__ __forceinline__ int perm_offset(int k) {
    constexpr int CPW = 32 / BITS;  // codes per code word
    constexpr int NW = CPW / 4;     // dp4a words per code word
    const int i = k % CPW;
    return (k - i) + 4 * (i % NW) + i / NW;
}

// Dot of one code word with its activation words (CPW codes).
template <int BITS>
__device__ __forceinline__ int dot_word(uint32_t w, const uint32_t *a, int acc) {
    if constexpr (BITS == 4) {
        acc = dp4a_us(w & 0x0f0f0f0fu, a[0], acc);
        acc = dp4a_us((w >> 4) & 0x0f0f0f0fu, a[1], acc);
    } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) acc = dp4a_us((w >> (2 * t)) & 0x03030303u, a[t], acc);
    }
    return acc;
}

// Activation k of the slot's vector: x, or silu(gate) * up of the slot's fc1 output.
template <int BITS, bool FC2>
__device__ __forceinline__ float act_value(const Dp4aGemv &p, int slot, int k) {
    if constexpr (FC2) {
        const int K = p.K;
        const float *gs = p.g + static_cast<size_t>(slot) * 2 * K;
        const float gate = p.swiglu_interleaved ? gs[2 * k] : gs[k];
        const float up = p.swiglu_interleaved ? gs[2 * k + 1] : gs[K + k];
        return gate / (1.f + expf(-gate)) * up;
    } else {
        return h2f(__ldg(p.x + k));
    }
}

// Quantizes the slot's activation vector per block of bs values into the
// permuted int8 layout x8, the sums of 16-value granules s16 and the block
// scales sxs; warps `warp`, `warp + nwarps`, ... take one block each.
template <int BITS, bool FC2>
__device__ __forceinline__ void quantize_acts(const Dp4aGemv &p, int slot, int warp, int nwarps, int lane,
                                              unsigned char *x8, int *s16, float *sxs) {
    const int K = p.K, bs = p.bs, nb = K / bs;
    for (int b = warp; b < nb; b += nwarps) {
        float v[8];  // bs / 32 <= 8 values per lane
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[j] = 0.f;
            if (j >= bs / 32) continue;
            const int k = b * bs + 32 * j + lane;
            const float val = act_value<BITS, FC2>(p, slot, k);
            v[j] = val;
            a = fmaxf(a, fabsf(val));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        const float sx = a > 0.f ? __fdiv_rn(a, 127.f) : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j >= bs / 32) break;  // warp-uniform
            const int k = b * bs + 32 * j + lane;
            int q = 0;
            if (a > 0.f) q = max(-127, min(127, __float2int_rn(__fdiv_rn(v[j], sx))));
            x8[perm_offset<BITS>(k)] = static_cast<unsigned char>(static_cast<signed char>(q));
            // sums over 16-value granules (lanes 0-15 and 16-31)
            int sq = q;
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
            if ((lane & 15) == 0) s16[k / 16] = sq;
        }
        if (lane == 0) sxs[b] = sx;
    }
}

// UPL: units per lane held in registers (1..4), or 0: units read from shared
// memory on every row (long rows).
template <int BITS, int VEC, bool FC2, int UPL>
__global__ void __launch_bounds__(kDThreads, 1) dp4a_gemv_kernel(Dp4aGemv p) {
    constexpr int CPW = 32 / BITS;
    constexpr int WPU = VEC / 4;            // code words per unit
    constexpr int CPU = VEC * 8 / BITS;     // codes per unit
    extern __shared__ __align__(16) unsigned char dsm[];
    const int K = p.K, bs = p.bs, nb = K / bs;
    unsigned char *x8 = dsm;                                             // [K] int8, permuted
    int *s16 = reinterpret_cast<int *>(dsm + ((K + 15) / 16) * 16);      // [K/16] sums of q8
    float *sxs = reinterpret_cast<float *>(s16 + K / 16);                // [K/bs] activation scales
    const int slot = blockIdx.x / p.cps, c = blockIdx.x % p.cps;
    const int e = __ldg(p.ids + slot);
    if (e < 0 || e >= p.num_experts) return;  // CTA-uniform: the slot adds nothing
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    quantize_acts<BITS, FC2>(p, slot, warp, kDWarps, lane, x8, s16, sxs);
    __syncthreads();

    // ---- rows of this CTA's share of the slot's matrix, two per warp at a time.
    // Lane l owns the row units l, l + 32, ... (VEC bytes, CPU codes each) of
    // every row; its activation words, 16-value sums and scales for those
    // units are fixed, so they are read from shared memory once.  The
    // integer sum is flushed every SEGC codes (a divisor of every block size).
    constexpr int SEGC = CPU < 32 ? CPU : 32;  // codes per flush
    constexpr int SPU = CPU / SEGC;            // flushes per unit
    constexpr int WPS = SEGC / CPW;            // code words per flush
    constexpr int AW = CPW / 4;                // activation words per code word
    constexpr int UR = UPL > 0 ? UPL : 1;      // unit slots held in registers
    const int row_bytes = K * BITS / 8;
    const int units = row_bytes / VEC;
    int bs_log2 = 5;
    while ((1 << bs_log2) < bs) ++bs_log2;
    const int rows_per = (p.N + p.cps - 1) / p.cps;
    const int r_lo = c * rows_per, r_hi = min(p.N, r_lo + rows_per);
    const uint8_t *we = p.w + static_cast<size_t>(e) * p.N * row_bytes;
    const uint16_t *se = p.scales + static_cast<size_t>(e) * p.N * nb;
    const uint16_t *ze = p.zp ? p.zp + static_cast<size_t>(e) * p.N * nb : nullptr;
    const float zdef = static_cast<float>(1 << (BITS - 1));

    uint32_t act[UR][WPU * AW];
    int sq[UR][SPU], blk[UR][SPU];
    float sx[UR][SPU];
    auto load_unit_consts = [&](int i, int u) {
#pragma unroll
        for (int j = 0; j < WPU * AW; ++j) act[i][j] = reinterpret_cast<const uint32_t *>(x8 + u * CPU)[j];
#pragma unroll
        for (int sgi = 0; sgi < SPU; ++sgi) {
            const int ks = u * CPU + sgi * SEGC;
            int S = 0;
#pragma unroll
            for (int gi = 0; gi < SEGC / 16; ++gi) S += s16[ks / 16 + gi];
            sq[i][sgi] = S;
            blk[i][sgi] = ks >> bs_log2;
            sx[i][sgi] = sxs[ks >> bs_log2];
        }
    };
    if constexpr (UPL > 0) {
#pragma unroll
        for (int i = 0; i < UPL; ++i)
            if (lane + 32 * i < units) load_unit_consts(i, lane + 32 * i);
    }

    for (int r0 = r_lo + 2 * warp; r0 < r_hi; r0 += 2 * kDWarps) {
        const int rr1 = min(r0 + 1, r_hi - 1);  // a missing second row re-reads the first (in bounds)
        float part[2] = {0.f, 0.f};
        for (int ub = 0; ub < units; ub += 32 * UR) {  // one pass when the units fit in registers
            uint32_t cw[2][UR][WPU];
            uint16_t sb[2][UR][SPU], zb[2][UR][SPU];
#pragma unroll
            for (int i = 0; i < UR; ++i) {
                const int u = ub + lane + 32 * i;
                if (u >= units) continue;
                if constexpr (UPL == 0) load_unit_consts(i, u);
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int r = rr ? rr1 : r0;
                    const uint8_t *src = we + static_cast<size_t>(r) * row_bytes + static_cast<size_t>(u) * VEC;
                    if constexpr (VEC == 16) {
                        const uint4 t = __ldg(reinterpret_cast<const uint4 *>(src));
                        cw[rr][i][0] = t.x;
                        cw[rr][i][1] = t.y;
                        cw[rr][i][2] = t.z;
                        cw[rr][i][3] = t.w;
                    } else {
                        const uint2 t = __ldg(reinterpret_cast<const uint2 *>(src));
                        cw[rr][i][0] = t.x;
                        cw[rr][i][1] = t.y;
                    }
#pragma unroll
                    for (int sgi = 0; sgi < SPU; ++sgi) {
                        const size_t pi = static_cast<size_t>(r) * nb + blk[i][sgi];
                        sb[rr][i][sgi] = __ldg(se + pi);
                        zb[rr][i][sgi] = ze ? __ldg(ze + pi) : uint16_t(0);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < UR; ++i) {
                if (ub + lane + 32 * i >= units) continue;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
                    for (int sgi = 0; sgi < SPU; ++sgi) {
                        int acc = 0;
#pragma unroll
                        for (int wi = sgi * WPS; wi < (sgi + 1) * WPS; ++wi)
                            acc = dot_word<BITS>(cw[rr][i][wi], &act[i][wi * AW], acc);
                        const float z = ze ? h2f(zb[rr][i][sgi]) : zdef;
                        part[rr] = fmaf(h2f(sb[rr][i][sgi]) * sx[i][sgi],
                                        static_cast<float>(acc) - z * static_cast<float>(sq[i][sgi]), part[rr]);
                    }
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            float t = part[rr];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
            const int r = r0 + rr;
            if (lane == 0 && r < r_hi) {
                if (p.bias) t += h2f(__ldg(p.bias + static_cast<size_t>(e) * p.N + r));
                p.out[static_cast<size_t>(slot) * p.N + r] = t;
            }
        }
    }
}

// y[r] = fp16( sum_j w_j * o_j[r] ) in slot order; out-of-range ids add
// nothing and set *status to 1.
__global__ void dp4a_combine_kernel(const float *__restrict__ o, const int32_t *__restrict__ ids,
                                    const float *__restrict__ w, int k, int num_experts, int H, uint16_t *y,
                                    int *status) {
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

size_t dp4a_smem(int K, int bs) { return static_cast<size_t>((K + 15) / 16) * 16 + (K / 16) * 4 + (K / bs) * 4; }

template <int BITS, int VEC, bool FC2, int UPL>
cudaError_t launch_gemv(const Dp4aGemv &a, int slots, cudaStream_t s) {
    auto kern = dp4a_gemv_kernel<BITS, VEC, FC2, UPL>;
    const size_t smem = dp4a_smem(a.K, a.bs);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    kern<<<slots * a.cps, kDThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int BITS, int VEC, bool FC2>
cudaError_t launch_upl(const Dp4aGemv &a, int slots, cudaStream_t s) {
    const int units = a.K * BITS / 8 / VEC;
    const int upl = (units + 31) / 32;
    if (BITS == 2 && VEC == 16 && upl > 2) return launch_gemv<BITS, VEC, FC2, 0>(a, slots, s);  // would spill
    switch (upl) {
    case 1: return launch_gemv<BITS, VEC, FC2, 1>(a, slots, s);
    case 2: return launch_gemv<BITS, VEC, FC2, 2>(a, slots, s);
    case 3: return launch_gemv<BITS, VEC, FC2, 3>(a, slots, s);
    case 4: return launch_gemv<BITS, VEC, FC2, 4>(a, slots, s);
    default: return launch_gemv<BITS, VEC, FC2, 0>(a, slots, s);
    }
}

template <bool FC2>
cudaError_t launch_bits(const Dp4aGemv &a, int bits, int slots, cudaStream_t s) {
    const bool v16 = (a.K * bits / 8) % 16 == 0;
    if (bits == 4) return v16 ? launch_upl<4, 16, FC2>(a, slots, s) : launch_upl<4, 8, FC2>(a, slots, s);
    return v16 ? launch_upl<2, 16, FC2>(a, slots, s) : launch_upl<2, 8, FC2>(a, slots, s);
}

}  // namespace

cudaError_t qmoe_decode_dp4a(const QmoeProblem &q, void *ws, cudaStream_t s) {
    const int H = q.hidden, I = q.inter, k = q.k;
    float *g = static_cast<float *>(ws);
    float *o = reinterpret_cast<float *>(static_cast<char *>(ws) +
                                         (static_cast<size_t>(k) * 2 * I * sizeof(float) + 255) / 256 * 256);
    // CTAs per slot: one wave of one 512-thread CTA per SM over all slots (the
    // register-resident units allow one such CTA per SM)
    const int cps = std::max(1, device_info().sm_count / k);
    Dp4aGemv a{};
    a.x = q.x;
    a.ids = q.ids;
    a.num_experts = q.num_experts;
    a.bs = q.bs;
    a.swiglu_interleaved = q.swiglu_interleaved;
    // fc1: [2I][H] per expert
    a.w = q.fc1_w;
    a.scales = q.fc1_scales;
    a.zp = q.fc1_zp;
    a.bias = q.fc1_bias;
    a.N = 2 * I;
    a.K = H;
    a.cps = std::min(cps, (a.N + 1) / 2);
    a.out = g;
    cudaError_t e = launch_bits<false>(a, q.bits, k, s);
    if (e != cudaSuccess) return e;
    // fc2: [H][I] per expert, activations silu(gate) * up of the slot's fc1 output
    a.x = nullptr;
    a.g = g;
    a.w = q.fc2_w;
    a.scales = q.fc2_scales;
    a.zp = q.fc2_zp;
    a.bias = q.fc2_bias;
    a.N = H;
    a.K = I;
    a.cps = std::min(cps, (a.N + 1) / 2);
    a.out = o;
    e = launch_bits<true>(a, q.bits, k, s);
    if (e != cudaSuccess) return e;
    dp4a_combine_kernel<<<(H + 255) / 256, 256, 0, s>>>(o, q.ids, q.weights, k, q.num_experts, H, q.y, q.status);
    return cudaGetLastError();
}

}  // namespace qg
