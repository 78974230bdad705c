// qg_gather.cu -- block-quantized embedding gather.
//
// Y[i][:] = dequant(table[idx[i]][:]) for a [V][D] table quantized along D in
// blocks (hip-ep pull request #1318, kernel test table: gather_block_quantized
// leaves Xi64_Wu4_Yfp16, Xi64_Wu8_Yfp16, Xi64_Wfp8_Yfp16; "Summary", Commit 3:
// embedding lookups through a gather).  Integer codes use the MatMulNBits
// layout and rule w = (q - zp) * s (codes LSB-first, scales and zero points
// [V][D/bs]); E4M3 bytes give w = e4m3(q) * s.  Every w is computed with the
// same two (or one) fp32 round-to-nearest operations as the dequantize
// export, then rounded to the output type.
//
// The op moves bytes only: a row of D outputs reads D*bits/8 code bytes and
// D/bs scales (and zero points) and writes D * sizeof(Y) bytes.  One thread
// handles 8 consecutive outputs of a row per unit (a 2-, 4- or 8-byte code
// load, 16 or 32 bytes of output), so a warp reads and writes contiguous
// runs.  A CTA takes one index at a time, loads it once, and its threads
// issue the loads of all their units of that row before any arithmetic.
#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr int kUnits = 4;  // 8-output units per thread per row

// Two E4M3 bytes (low byte first) -> fp16x2 (exact: every E4M3 value is an
// fp16 value; NaN stays NaN).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<unsigned short>(two)));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
    return r;
}

// Integer codes of one unit: code j of the unit, masked in place inside its
// 32-bit word and OR-ed into the fp32 pattern of 2^23, is 2^23 + q*2^p
// exactly (p = its bit position, p + bits <= 23); subtracting 2^23 and
// scaling by 2^-p gives q exactly, and the fused multiply-add
// (q*2^p)*2^-p - z rounds q - z once.  Codes above bit 23 are taken from the
// word shifted right by 16 (u8) or 20 (u4).
template <int BITS>
__device__ __forceinline__ void dequant_unit(uint32_t lo, uint32_t hi, float z, float s, float (&w)[8]) {
    constexpr uint32_t MASK = (1u << BITS) - 1u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t word;
        int pos;
        if constexpr (BITS == 2) {
            word = lo;
            pos = 2 * j;
        } else if constexpr (BITS == 4) {
            word = j < 5 ? lo : lo >> 20;
            pos = j < 5 ? 4 * j : 4 * (j - 5);
        } else {
            const uint32_t src = j < 4 ? lo : hi;
            word = (j & 3) < 2 ? src : src >> 16;
            pos = 8 * ((j & 3) & 1);
        }
        const float x = __uint_as_float((word & (MASK << pos)) | 0x4b000000u) - 8388608.f;  // q * 2^pos
        const float d = fmaf(x, __uint_as_float(static_cast<uint32_t>(127 - pos) << 23), -z);  // RN(q - z)
        w[j] = __fmul_rn(d, s);
    }
}

template <int YT>
__device__ __forceinline__ void store8(void *Y, size_t off, const float (&w)[8]) {
    if constexpr (YT == 0) {
        float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(Y) + off);
        p[0] = make_float4(w[0], w[1], w[2], w[3]);
        p[1] = make_float4(w[4], w[5], w[6], w[7]);
    } else {
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) h[j] = YT == 1 ? pack_f16x2(w[2 * j], w[2 * j + 1]) : pack_bf16x2(w[2 * j], w[2 * j + 1]);
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(Y) + off) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// FMT: 0 u2, 1 u4, 2 u8, 3 E4M3.  YT: 0 fp32, 1 fp16, 2 bf16.
// grid.y strides over the indices, grid.x over chunks of blockDim.x * kUnits
// units of a row.  Each thread first issues the loads of its (up to) kUnits
// units, then dequantizes and stores them.
template <int FMT, int YT>
__global__ void __launch_bounds__(256) gather_kernel(const int64_t *__restrict__ idx, long long n,
                                                     const uint8_t *__restrict__ W,
                                                     const uint16_t *__restrict__ scales,
                                                     const uint16_t *__restrict__ zp, float zdef, long long V, int D,
                                                     int bs_log2, void *__restrict__ Y, int *status) {
    constexpr int BITS = FMT == 0 ? 2 : (FMT == 1 ? 4 : 8);
    const int upr = D / 8;  // 8-output units per row (D is a multiple of bs >= 32)
    const long long nb = D >> bs_log2;
    const long long row_bytes = static_cast<long long>(D) * BITS / 8;
    const int u0 = blockIdx.x * blockDim.x * kUnits + threadIdx.x;
    for (long long i = blockIdx.y; i < n; i += gridDim.y) {
        long long row = __ldg(idx + i);
        if (row < 0) row += V;
        const bool ok = row >= 0 && row < V;
        if (!ok && status && u0 == 0) *status = 1;  // every writer stores the same value
        uint32_t lo[kUnits], hi[kUnits];
        float s[kUnits], z[kUnits];
#pragma unroll
        for (int k = 0; k < kUnits; ++k) {
            const int u = u0 + k * blockDim.x;
            lo[k] = hi[k] = 0;
            s[k] = z[k] = 0.f;
            if (ok && u < upr) {
                const long long b = row * nb + ((8 * u) >> bs_log2);
                const uint8_t *src = W + row * row_bytes + static_cast<long long>(u) * BITS;  // 8 codes per unit
                if constexpr (BITS == 2) lo[k] = __ldg(reinterpret_cast<const unsigned short *>(src));
                else if constexpr (BITS == 4) lo[k] = __ldg(reinterpret_cast<const unsigned int *>(src));
                else {
                    const uint2 x = __ldg(reinterpret_cast<const uint2 *>(src));
                    lo[k] = x.x;
                    hi[k] = x.y;
                }
                const uint16_t sb = __ldg(scales + b);
                if constexpr (FMT == 3 && YT == 1) {
                    s[k] = __uint_as_float(static_cast<uint32_t>(sb));  // raw fp16 bits, used as fp16x2 below
                } else {
                    s[k] = h2f(sb);
                    if constexpr (FMT != 3) z[k] = zp ? h2f(__ldg(zp + b)) : zdef;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kUnits; ++k) {
            const int u = u0 + k * blockDim.x;
            if (u >= upr) break;
            const size_t off = static_cast<size_t>(i) * D + 8 * u;
            if constexpr (FMT == 3 && YT == 1) {
                // fp16 out: RN16(e4m3 * s) directly; the exact product has at most 15 significant bits,
                // so this equals rounding the fp32 product (which is exact) to fp16.
                const uint32_t sb = __float_as_uint(s[k]);
                const uint32_t s2 = sb | (sb << 16);
                uint32_t h[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t e2 = e4m3x2_to_f16x2((j < 2 ? lo[k] : hi[k]) >> (16 * (j & 1)));
                    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(h[j]) : "r"(e2), "r"(s2));
                }
                if (!ok) h[0] = h[1] = h[2] = h[3] = 0u;
                *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(Y) + off) = make_uint4(h[0], h[1], h[2], h[3]);
            } else {
                float w[8];
                if constexpr (FMT == 3) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t e2 = e4m3x2_to_f16x2((j < 2 ? lo[k] : hi[k]) >> (16 * (j & 1)));
                        w[2 * j] = __fmul_rn(__half2float(__ushort_as_half(static_cast<unsigned short>(e2 & 0xffffu))), s[k]);
                        w[2 * j + 1] = __fmul_rn(__half2float(__ushort_as_half(static_cast<unsigned short>(e2 >> 16))), s[k]);
                    }
                } else {
                    dequant_unit<BITS>(lo[k], hi[k], z[k], s[k], w);
                }
                if (!ok) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) w[j] = 0.f;
                }
                store8<YT>(Y, off, w);
            }
        }
    }
}

template <int FMT>
cudaError_t launch_fmt(const GatherProblem &g, int bs_log2, dim3 grid, int threads, cudaStream_t s) {
    const float zdef = FMT == 3 ? 0.f : static_cast<float>(1 << ((FMT == 0 ? 2 : (FMT == 1 ? 4 : 8)) - 1));
    switch (g.y_dtype) {
    case 0:
        gather_kernel<FMT, 0><<<grid, threads, 0, s>>>(g.idx, g.n, g.W, g.scales, g.zp, zdef, g.V, g.D, bs_log2,
                                                       g.Y, g.status);
        break;
    case 1:
        gather_kernel<FMT, 1><<<grid, threads, 0, s>>>(g.idx, g.n, g.W, g.scales, g.zp, zdef, g.V, g.D, bs_log2,
                                                       g.Y, g.status);
        break;
    default:
        gather_kernel<FMT, 2><<<grid, threads, 0, s>>>(g.idx, g.n, g.W, g.scales, g.zp, zdef, g.V, g.D, bs_log2,
                                                       g.Y, g.status);
        break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather(const GatherProblem &g, cudaStream_t s) {
    int bs_log2 = 0;
    while ((1 << bs_log2) < g.bs) ++bs_log2;
    const int upr = g.D / 8;
    // threads per CTA: enough for kUnits units each over the row (a multiple of 32, at most 256)
    const int threads = std::min(256, std::max(32, ((upr + kUnits - 1) / kUnits + 31) / 32 * 32));
    dim3 grid((upr + threads * kUnits - 1) / (threads * kUnits),
              static_cast<unsigned>(std::min<long long>(g.n, 65535)));
    switch (g.fmt) {
    case 0: return launch_fmt<0>(g, bs_log2, grid, threads, s);
    case 1: return launch_fmt<1>(g, bs_log2, grid, threads, s);
    case 2: return launch_fmt<2>(g, bs_log2, grid, threads, s);
    default: return launch_fmt<3>(g, bs_log2, grid, threads, s);
    }
}

}  // namespace qg
