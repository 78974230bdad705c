// qg_util.cu -- dequantize-to-fp32 export and the fp16 uniform-value check.
//
// The export writes w[n][k] exactly as the GEMM kernels define it (two fp32
// round-to-nearest operations for MatMulNBits, one for the codebook), so the
// unpacking and dequantization can be checked bit for bit in isolation.
// The uniform check backs the scalar zero-point path of hip-ep #1318
// ("What", Commit 1: an all-equal fp16 zero-point tensor is detected once
// per buffer and then passed as a scalar).
#include "qg_device.cuh"
#include "qg_internal.h"

#include <algorithm>

namespace qg {
namespace {

// One thread per 32-bit word of codes (16 u2, 8 u4 or 4 u8 codes).
template <int BITS, int WK>
__global__ void dequant_kernel(const uint8_t *__restrict__ W, const unsigned char *__restrict__ params,
                               const uint16_t *__restrict__ zp, int zp_mode, float zpv,
                               const float *__restrict__ codebook, float *__restrict__ out, int N, int K, int bs) {
    constexpr int CPW = 32 / BITS;
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    const int wpr = K / CPW;  // words per row
    const int nb = K / bs;
    const size_t total = static_cast<size_t>(N) * wpr;
    for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(t / wpr);
        const int wi = static_cast<int>(t % wpr);
        const uint32_t x = __ldg(reinterpret_cast<const uint32_t *>(W + static_cast<size_t>(n) * (K * BITS / 8)) + wi);
        const int kbase = wi * CPW;
        const int b = kbase / bs;  // a word never straddles a block (bs >= 32 >= codes per word)
        float *o = out + static_cast<size_t>(n) * K + kbase;
        if constexpr (WK == WK_NBITS) {
            const float s = h2f(__ldg(reinterpret_cast<const unsigned short *>(params) + static_cast<size_t>(n) * nb + b));
            const float z = zp_mode == ZP_TENSOR ? h2f(__ldg(reinterpret_cast<const unsigned short *>(zp) + static_cast<size_t>(n) * nb + b)) : zpv;
#pragma unroll
            for (int i = 0; i < CPW; ++i) {
                const float d = __fsub_rn(static_cast<float>((x >> (BITS * i)) & MASK), z);
                o[i] = __fmul_rn(d, s);
            }
        } else {
            const float am = __ldg(reinterpret_cast<const float *>(params) + static_cast<size_t>(n) * nb + b);
#pragma unroll
            for (int i = 0; i < CPW; ++i) o[i] = __fmul_rn(__ldg(codebook + ((x >> (4 * i)) & 15u)), am);
        }
    }
}

// u3: one thread per weight; code k is the 3 bits at bit 3k of the row,
// which may continue into the next byte.
__global__ void dequant_u3_kernel(const uint8_t *__restrict__ W, const uint16_t *__restrict__ scales,
                                  const uint16_t *__restrict__ zp, int zp_mode, float zpv, float *__restrict__ out, int N,
                                  int K, int bs) {
    const int nb = K / bs, row_bytes = K * 3 / 8;
    const size_t total = static_cast<size_t>(N) * K;
    for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(t / K), k = static_cast<int>(t % K);
        const uint8_t *row = W + static_cast<size_t>(n) * row_bytes;
        const int bit = 3 * k;
        uint32_t v = __ldg(row + bit / 8);
        if (bit % 8 > 5) v |= static_cast<uint32_t>(__ldg(row + bit / 8 + 1)) << 8;
        const float q = static_cast<float>((v >> (bit % 8)) & 7u);
        const int b = k / bs;
        const float s = h2f(__ldg(scales + static_cast<size_t>(n) * nb + b));
        const float z = zp_mode == ZP_TENSOR ? h2f(__ldg(zp + static_cast<size_t>(n) * nb + b)) : zpv;
        out[t] = __fmul_rn(__fsub_rn(q, z), s);
    }
}

// Packed unsigned-integer zero points -> fp16 [N][nb]: zero point b of row n
// is the `bits`-wide field at bit b*bits of row n's bit string (least
// significant bit first, the codes' own packing rule; a field may continue
// into the next byte), rows padded to row_bytes = ceil(nb*bits/8).  The
// integers (at most 255) are exact in fp16.
__global__ void unpack_zero_points_kernel(const uint8_t *__restrict__ zp, int bits, int nb, int row_bytes,
                                          size_t total, uint16_t *__restrict__ out) {
    for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t n = t / nb;
        const int b = static_cast<int>(t - n * nb);
        const int bit = b * bits;
        const uint8_t *row = zp + n * row_bytes;
        uint32_t v = __ldg(row + bit / 8);
        if (bit % 8 + bits > 8) v |= static_cast<uint32_t>(__ldg(row + bit / 8 + 1)) << 8;
        const unsigned q = (v >> (bit % 8)) & ((1u << bits) - 1u);
        out[t] = __half_as_ushort(__uint2half_rn(q));
    }
}

// The same when rows need no padding (nb*bits a multiple of 8) and bits is
// 2, 4 or 8: the packed bytes form one flat stream, byte i holding zero points
// i*8/bits onwards; one thread per byte, one store of its 8/bits values.
template <int BITS>
__global__ void unpack_zero_points_flat_kernel(const uint8_t *__restrict__ zp, size_t nbytes,
                                               uint16_t *__restrict__ out) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < nbytes;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const unsigned v = __ldg(zp + i);
        if constexpr (BITS == 8) {
            out[i] = __half_as_ushort(__uint2half_rn(v));
        } else if constexpr (BITS == 4) {
            const uint32_t lo = __half_as_ushort(__uint2half_rn(v & 15u)), hi = __half_as_ushort(__uint2half_rn(v >> 4));
            reinterpret_cast<uint32_t *>(out)[i] = lo | (hi << 16);
        } else {
            uint32_t h[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) h[j] = __half_as_ushort(__uint2half_rn((v >> (2 * j)) & 3u));
            reinterpret_cast<uint2 *>(out)[i] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        }
    }
}

// Nested absmax: absmax[i] = (table[qa[i]] * absmax2[i / nested]) + offset,
// two fp32 round-to-nearest operations (bitsandbytes #1979 "Testing plan":
// nested / non-nested absmax; the layout is this library's reading).
__global__ void nested_absmax_kernel(const uint8_t *__restrict__ qa, const float *__restrict__ table,
                                     const float *__restrict__ absmax2, float offset, int nested, size_t n,
                                     float *__restrict__ out) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        out[i] = __fadd_rn(__fmul_rn(__ldg(table + __ldg(qa + i)), __ldg(absmax2 + i / nested)), offset);
}

// ws[0] <- 1 if some element's bit pattern differs from t[0].  Every writer
// stores the same value, so the result does not depend on the order.
__global__ void uniform_kernel(const uint16_t *__restrict__ t, size_t n, unsigned *ws) {
    const uint16_t v0 = __ldg(reinterpret_cast<const unsigned short *>(t));
    bool diff = false;
    const size_t n8 = n / 8;
    const uint4 *t4 = reinterpret_cast<const uint4 *>(t);
    const uint32_t pair = static_cast<uint32_t>(v0) | (static_cast<uint32_t>(v0) << 16);
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const uint4 v = __ldg(t4 + i);
        diff |= (v.x != pair) | (v.y != pair) | (v.z != pair) | (v.w != pair);
    }
    for (size_t i = n8 * 8 + blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        diff |= __ldg(reinterpret_cast<const unsigned short *>(t) + i) != v0;
    if (__syncthreads_or(diff) && threadIdx.x == 0) ws[0] = 1u;
}

}  // namespace

cudaError_t launch_dequant(const GemmProblem &p, float *out, cudaStream_t s) {
    if (p.kind == WK_NBITS && p.bits == 3) {
        const size_t total = static_cast<size_t>(p.N) * p.K;
        if (total == 0) return cudaSuccess;
        const int threads = 256;
        const int blocks = static_cast<int>(std::min<size_t>((total + threads - 1) / threads, 65536));
        dequant_u3_kernel<<<blocks, threads, 0, s>>>(p.W, p.scales, p.zp, p.zp_mode, p.uniform_zp, out, p.N, p.K, p.bs);
        return cudaGetLastError();
    }
    const int cpw = 32 / p.bits;
    const size_t total = static_cast<size_t>(p.N) * (p.K / cpw);
    const int threads = 256;
    const int blocks = static_cast<int>(std::min<size_t>((total + threads - 1) / threads, 65536));
    if (total == 0) return cudaSuccess;
    if (p.kind == WK_CODEBOOK)
        dequant_kernel<4, WK_CODEBOOK><<<blocks, threads, 0, s>>>(
            p.W, reinterpret_cast<const unsigned char *>(p.absmax), nullptr, 0, 0.f, p.codebook, out, p.N, p.K, p.bs);
    else if (p.bits == 2)
        dequant_kernel<2, WK_NBITS><<<blocks, threads, 0, s>>>(p.W, reinterpret_cast<const unsigned char *>(p.scales),
                                                                p.zp, p.zp_mode, p.uniform_zp, nullptr, out, p.N,
                                                                p.K, p.bs);
    else if (p.bits == 8)
        dequant_kernel<8, WK_NBITS><<<blocks, threads, 0, s>>>(p.W, reinterpret_cast<const unsigned char *>(p.scales),
                                                                p.zp, p.zp_mode, p.uniform_zp, nullptr, out, p.N,
                                                                p.K, p.bs);
    else
        dequant_kernel<4, WK_NBITS><<<blocks, threads, 0, s>>>(p.W, reinterpret_cast<const unsigned char *>(p.scales),
                                                                p.zp, p.zp_mode, p.uniform_zp, nullptr, out, p.N,
                                                                p.K, p.bs);
    return cudaGetLastError();
}

cudaError_t launch_nested_absmax(const uint8_t *qa, const float *table, const float *absmax2, float offset,
                                 int nested, size_t n, float *out, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = static_cast<int>(std::min<size_t>((n + threads - 1) / threads, 4096));
    nested_absmax_kernel<<<blocks, threads, 0, s>>>(qa, table, absmax2, offset, nested, n, out);
    return cudaGetLastError();
}

cudaError_t launch_unpack_zero_points(const uint8_t *zp, int bits, int N, int nb, uint16_t *out, cudaStream_t s) {
    const size_t total = static_cast<size_t>(N) * nb;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    if ((static_cast<size_t>(nb) * bits) % 8 == 0 && bits != 3) {  // out is 16-byte aligned (workspace front)
        const size_t nbytes = total * bits / 8;
        const int blocks = static_cast<int>(std::min<size_t>((nbytes + threads - 1) / threads, 65536));
        if (bits == 8) unpack_zero_points_flat_kernel<8><<<blocks, threads, 0, s>>>(zp, nbytes, out);
        else if (bits == 4) unpack_zero_points_flat_kernel<4><<<blocks, threads, 0, s>>>(zp, nbytes, out);
        else unpack_zero_points_flat_kernel<2><<<blocks, threads, 0, s>>>(zp, nbytes, out);
        return cudaGetLastError();
    }
    const int blocks = static_cast<int>(std::min<size_t>((total + threads - 1) / threads, 4096));
    unpack_zero_points_kernel<<<blocks, threads, 0, s>>>(zp, bits, nb, (nb * bits + 7) / 8, total, out);
    return cudaGetLastError();
}

cudaError_t launch_uniform_check(const uint16_t *t, size_t n, unsigned *ws, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    const int threads = 256;
    const int blocks = static_cast<int>(std::min<size_t>((n / 8 + threads - 1) / threads + 1, 1024));
    uniform_kernel<<<blocks, threads, 0, s>>>(t, n, ws);
    return cudaGetLastError();
}

}  // namespace qg
