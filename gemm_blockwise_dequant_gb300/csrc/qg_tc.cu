// qg_tc.cu -- tensor-core blockwise-dequant GEMM for M >= 16 on sm_103a
// (tcgen05 MMA, accumulator in tensor memory, TMA-fed activations).
//
//   Y[m][n] = sum_k A[m][k] * w[n][k],   A fp16 / bf16,   w rounded to A's type
//
// hip-ep #1318, "What" (Commit 1): the prefill-sized 2-bit MatMulNBits runs
// on the matrix units, with 16-bit activations and an fp32 epilogue; the
// codebook weights of bitsandbytes #1979 take the same path for M >= 16.
// The pages' WMMA tiling (gfx1151) is prior art only; this kernel is built
// for the fifth-generation tensor cores:
//
//  * Tile: 128 activation rows (MMA M) x BN weight rows (MMA N), K in steps of
//    64 (one 128-byte swizzle row of 16-bit values).  The accumulator lives in
//    tensor memory (BN fp32 columns x 128 lanes).
//  * Warp 0: TMA producer.  Per stage it loads the activation tile (2-D tiled
//    copy, 128-byte swizzle, rows past M zero-filled) and the packed weight
//    codes of the BN rows (2-D tiled copy, rows past N zero-filled).
//  * Warp 1: allocates tensor memory; one elected lane issues the four
//    K=16 MMAs of each stage and commits them to the stage's "empty"
//    barrier, which releases the stage to the producer and to the dequant
//    warps.
//  * Warps 2-5: dequantize the stage's codes into the 128-byte-swizzled
//    K-major operand layout (one 16-byte store per 8 weights, bank-conflict
//    free), fence the generic-proxy writes for the tensor core and signal the
//    stage; after the last stage they read the accumulator back (tcgen05.ld;
//    the four warps cover the four tensor-memory sub-partitions) and write Y.
//  * Dequantization of u2/u4 codes uses the fp16 magic-number form: one LOP3
//    turns two codes into an fp16 pair 1024 + c*q, an HFMA2 removes the
//    offset exactly, then the zero point and the scale are applied with
//    packed fp16 arithmetic (the weight is rounded to 16 bits, as the MMA
//    needs).  Codebook weights use a per-lane replicated table in shared
//    memory and fp32 products rounded to the activation type.
//  * Every wait is bounded; a stuck pipeline records a fault bit and the CTA
//    still releases its tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
// pipeline depth: 4 stages, 3 for the widest tile (shared-memory budget)
__host__ __device__ constexpr int stages_for(int bn) { return bn >= 256 ? 3 : 4; }
constexpr int kThreads = 320;         // warp 0 TMA, warp 1 MMA, warps 2-9 dequant + epilogue
constexpr int kDequantThreads = 256;
constexpr int kParamBox = 16;         // bytes of block parameters per weight row per stage (one TMA box column)

struct TcArgs {
    const uint16_t *scales;  // nbits, [N][nb] fp16
    const uint16_t *zp;      // nbits, [N][nb] fp16 (ZP_TENSOR)
    int zp_mode;
    float zpv;
    const float *codebook;   // codebook, [16]
    const float *absmax;     // codebook, [N][nb]
    void *Y;
    int y_dtype;
    float *partial;          // split-K partials [splits][M][N] or nullptr
    int M, N, K, bs, lbs, nb, nk, ks_per_split;  // lbs = log2(bs)
    unsigned *fault;
};

// --- tcgen05 / TMA primitives -------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (start address, leading / stride byte offsets in
// 16-byte units, descriptor version 1, swizzle mode 2 = 128B).
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, A/B fp16 or bf16,
// both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// 128-byte swizzle: 16-byte chunk c of row r (8 rows per 1024-byte atom)
__device__ __forceinline__ uint32_t swz128(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Convert an fp16 pair to the MMA operand type (identity for fp16).
template <bool BF16>
__device__ __forceinline__ uint32_t to_operand(__half2 h) {
    if constexpr (BF16) {
        const float2 f = __half22float2(h);
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
        return *reinterpret_cast<const uint32_t *>(&b);
    } else {
        return h2_as_u32(h);
    }
}

// 8 weights (k = 8c .. 8c+7 of one row) from their packed codes, as four
// operand pairs.  nbits: w = (q - zp) * s in fp16 (zp2, s2: fp16 pairs).
template <int BITS, bool BF16>
__device__ __forceinline__ uint4 dequant8_nbits(uint32_t codes, uint32_t zp2u, uint32_t s2u) {
    const __half2 zp2 = u32_as_h2(zp2u), s2 = u32_as_h2(s2u);
    uint32_t out[4];
    if constexpr (BITS == 2) {
        // codes: 16 bits, 8 codes; byte j holds codes 4j .. 4j+3
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t v = __byte_perm(codes, 0u, 0x4040u | (j * 0x0101u));  // byte j into bytes 0 and 2
            const uint32_t h01 = (v & 0x000C0003u) | 0x64006400u;  // (1024 + q0, 1024 + 4 q1)
            const uint32_t h23 = (v & 0x00C00030u) | 0x64006400u;  // (1024 + 16 q2, 1024 + 64 q3)
            const __half2 q01 = __hfma2(u32_as_h2(h01), __floats2half2_rn(1.f, 0.25f), __floats2half2_rn(-1024.f, -256.f));
            const __half2 q23 = __hfma2(u32_as_h2(h23), __floats2half2_rn(0.0625f, 0.015625f), __floats2half2_rn(-64.f, -16.f));
            out[2 * j] = to_operand<BF16>(__hmul2(__hsub2(q01, zp2), s2));
            out[2 * j + 1] = to_operand<BF16>(__hmul2(__hsub2(q23, zp2), s2));
        }
    } else {
        // codes: 32 bits, 8 codes; byte j holds codes 2j, 2j+1
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t v = __byte_perm(codes, 0u, 0x4040u | (j * 0x0101u));
            const uint32_t h = (v & 0x00F0000Fu) | 0x64006400u;  // (1024 + q0, 1024 + 16 q1)
            const __half2 q = __hfma2(u32_as_h2(h), __floats2half2_rn(1.f, 0.0625f), __floats2half2_rn(-1024.f, -64.f));
            out[j] = to_operand<BF16>(__hmul2(__hsub2(q, zp2), s2));
        }
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// codebook: w = C[q] * absmax (fp32), rounded to the operand type
template <bool BF16>
__device__ __forceinline__ uint4 dequant8_codebook(uint32_t codes, float am, const float *lut_lane) {
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float w0 = lut_lane[((codes >> (8 * j)) & 15u) * 32] * am;
        const float w1 = lut_lane[((codes >> (8 * j + 4)) & 15u) * 32] * am;
        if constexpr (BF16) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(w0, w1);
            out[j] = *reinterpret_cast<const uint32_t *>(&b);
        } else {
            out[j] = h2_as_u32(__floats2half2_rn(w0, w1));
        }
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

template <int WK, int BITS, bool BF16, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap act_map, const __grid_constant__ CUtensorMap code_map,
                   const __grid_constant__ CUtensorMap par_map, const __grid_constant__ CUtensorMap zp_map,
                   const TcArgs p) {
    constexpr int kStages = stages_for(BN);
    constexpr int CB = kBK * BITS / 8;           // code bytes per row per stage
    constexpr int ACT_BYTES = kBM * kBK * 2;     // 16 KB
    constexpr int WDQ_BYTES = BN * kBK * 2;
    constexpr int CODE_BYTES = BN * CB;
    constexpr int PAR_BYTES = BN * kParamBox;
    constexpr int PE = WK == WK_CODEBOOK ? 4 : 2;  // bytes per block parameter
    constexpr int PPB = kParamBox / PE;            // parameters per box row
    constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled tiles (pointer arithmetic on the
    // shared array keeps the accesses in the shared address space)
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char *act_s = smem;
    unsigned char *wdq_s = act_s + kStages * ACT_BYTES;
    unsigned char *code_s = wdq_s + kStages * WDQ_BYTES;
    unsigned char *par_s = code_s + kStages * CODE_BYTES;
    unsigned char *zp_s = par_s + kStages * PAR_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(zp_s + kStages * PAR_BYTES);
    uint64_t *full = bars;                 // TMA landed (count 1 + tx)
    uint64_t *wfull = bars + kStages;      // dequantized weights written (count 4 warps)
    uint64_t *empty = bars + 2 * kStages;  // MMAs of the stage finished (commit)
    uint64_t *accf = bars + 3 * kStages;   // all MMAs finished
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * kStages + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *lut = reinterpret_cast<float *>(tmem_slot + 4);  // 16 x 32 floats (codebook)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * BN;
    const int ks0 = blockIdx.z * p.ks_per_split;
    const int ks1 = min(p.nk, ks0 + p.ks_per_split);
    const int nks = max(0, ks1 - ks0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&wfull[s], kDequantThreads / 32);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if constexpr (WK == WK_CODEBOOK) {
        for (int i = threadIdx.x; i < 16 * 32; i += kThreads) lut[i] = __ldg(p.codebook + (i >> 5));
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();  // the next kernel may start launching as these CTAs retire

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            pdl_wait();  // activations may come from the preceding kernel; everything else follows this producer
            for (int i = 0; i < nks; ++i) {
                const int s = i % kStages;
                if (!mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1, abort_flag, p.fault, FAULT_WAIT_TC)) break;
                const bool zt = WK == WK_NBITS && p.zp_mode == ZP_TENSOR;
                mbar_arrive_expect_tx(&full[s], ACT_BYTES + CODE_BYTES + PAR_BYTES * (zt ? 2 : 1));
                const int ks = ks0 + i;
                const int pcol = (ks * kBK / p.bs) / PPB * PPB;  // first parameter column of the box
                tma_load_2d(act_s + s * ACT_BYTES, &act_map, ks * kBK, m0, &full[s]);
                tma_load_2d(code_s + s * CODE_BYTES, &code_map, ks * CB, n0, &full[s]);
                tma_load_2d(par_s + s * PAR_BYTES, &par_map, pcol, n0, &full[s]);
                if (zt) tma_load_2d(zp_s + s * PAR_BYTES, &zp_map, pcol, n0, &full[s]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kBM, BN, BF16);
            bool ok = true;
            for (int i = 0; i < nks && ok; ++i) {
                const int s = i % kStages;
                const uint32_t par = (i / kStages) & 1;
                ok = mbar_wait(&full[s], par, abort_flag, p.fault, FAULT_WAIT_TC) &&
                     mbar_wait(&wfull[s], par, abort_flag, p.fault, FAULT_WAIT_TC);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ad = sdesc_k128(smem_u32(act_s + s * ACT_BYTES));
                const uint64_t bd = sdesc_k128(smem_u32(wdq_s + s * WDQ_BYTES));
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)  // +32 bytes per K=16 step inside the swizzle row
                    umma_f16(tmem, ad + 2 * k, bd + 2 * k, idesc, (i > 0 || k > 0) ? 1u : 0u);
                umma_commit(&empty[s]);
            }
            umma_commit(accf);  // arrives when every MMA issued above has finished
        }
    } else {
        // ------------------------------------------------------------ dequant warps
        // Thread t owns units u = t + j*kDequantThreads (j < UPT); unit u is 8
        // weights: row u/8 of the tile, 16-byte chunk u%8 of the 64-wide stage.
        // Offsets are fixed for the whole K loop; per stage every load of the
        // thread is issued before any conversion, so its UPT chains overlap.
        constexpr int UPT = BN * 8 / kDequantThreads;
        const int t = threadIdx.x - 64;  // 0 .. kDequantThreads-1
        const float *lut_lane = lut + lane;
        // Rows past N and k past K need no test: the TMA boxes zero-fill them,
        // so their codes, scales and absmax are 0 and the weight comes out 0.
        uint32_t code_off[UPT], wdq_off[UPT], par_off[UPT];
#pragma unroll
        for (int j = 0; j < UPT; ++j) {
            const int u = t + j * kDequantThreads;
            const int r = u >> 3, c = u & 7;
            code_off[j] = r * CB + c * (CB / 8);
            wdq_off[j] = swz128(r, c);
            par_off[j] = r * kParamBox + ((8 * c) >> p.lbs) * PE;  // block of this chunk within the stage
        }
        const uint32_t zpu = __half_as_ushort(__float2half_rn(p.zpv)) * 0x10001u;
        const bool zt = WK == WK_NBITS && p.zp_mode == ZP_TENSOR;
        for (int i = 0; i < nks; ++i) {
            const int s = i % kStages;
            if (!mbar_wait(&full[s], (i / kStages) & 1, abort_flag, p.fault, FAULT_WAIT_TC)) break;
            const int kb = (ks0 + i) * kBK;
            const int pc0 = ((kb >> p.lbs) % PPB) * PE;  // first block of the stage inside its parameter box
            const unsigned char *__restrict__ cs = code_s + s * CODE_BYTES;
            const unsigned char *__restrict__ ps = par_s + s * PAR_BYTES + pc0;
            const unsigned char *__restrict__ zs = zp_s + s * PAR_BYTES + pc0;
            unsigned char *__restrict__ ws = wdq_s + s * WDQ_BYTES;
            uint32_t codes[UPT], pv[UPT], zv[UPT];
#pragma unroll
            for (int j = 0; j < UPT; ++j) {
                if constexpr (WK == WK_NBITS) {
                    codes[j] = BITS == 2 ? static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(cs + code_off[j]))
                                         : *reinterpret_cast<const uint32_t *>(cs + code_off[j]);
                    pv[j] = *reinterpret_cast<const uint16_t *>(ps + par_off[j]);
                    zv[j] = zt ? *reinterpret_cast<const uint16_t *>(zs + par_off[j]) : 0u;
                } else {
                    codes[j] = *reinterpret_cast<const uint32_t *>(cs + code_off[j]);
                    pv[j] = *reinterpret_cast<const uint32_t *>(ps + par_off[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < UPT; ++j) {
                uint4 w;
                if constexpr (WK == WK_NBITS) {
                    w = dequant8_nbits<BITS, BF16>(codes[j], zt ? zv[j] * 0x10001u : zpu, pv[j] * 0x10001u);
                } else {
                    w = dequant8_codebook<BF16>(codes[j], __uint_as_float(pv[j]), lut_lane);
                }
                *reinterpret_cast<uint4 *>(ws + wdq_off[j]) = w;
            }
            fence_async_smem();  // make the generic-proxy stores visible to the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&wfull[s]);
        }
        // ------------------------------------------------------------ epilogue
        const bool ok = mbar_wait(accf, 0, abort_flag, p.fault, FAULT_WAIT_TC);
        tc_fence_after();
        const int sub = warp & 3;  // tensor-memory sub-partition this warp may read
        const int chalf = (warp - 2) >> 2;  // two warps share a sub-partition: each takes half the columns
        const int m = m0 + sub * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(sub * 32) << 16);
        constexpr int CW = BN >= 64 ? BN / 2 : BN;
#pragma unroll 1
        for (int c0 = chalf * CW; c0 < (chalf + 1) * CW && c0 < BN; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(lane_addr + c0, r);
            if (!ok || m >= p.M || nks == 0) continue;
            const int nb0 = n0 + c0;
            if (p.partial) {
                float *dst = p.partial + (static_cast<size_t>(blockIdx.z) * p.M + m) * p.N + nb0;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (nb0 + j < p.N) dst[j] = __uint_as_float(r[j]);
            } else if (p.y_dtype == 0 && (p.N & 3) == 0 && nb0 + 32 <= p.N) {
                float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.Y) + static_cast<size_t>(m) * p.N + nb0);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                         __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (nb0 + j < p.N)
                        store_y_elem(p.Y, p.y_dtype, static_cast<size_t>(m) * p.N + nb0 + j, __uint_as_float(r[j]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

__global__ void tc_splitk_reduce_kernel(const float *__restrict__ partial, int splits, size_t MN, void *Y,
                                        int y_dtype) {
    pdl_wait();
    pdl_launch_dependents();
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < MN;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float s = 0.f;
        for (int sp = 0; sp < splits; ++sp) s += partial[sp * MN + i];
        store_y_elem(Y, y_dtype, i, s);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
    if (!f) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

struct TcCfg {
    int bn, splits, ks_per_split, nk, m_tiles, n_tiles;
};

int smem_bytes(int bn, int bits) {
    const int cb = kBK * bits / 8;
    const int st = stages_for(bn);
    return 1024 + st * (kBM * kBK * 2 + bn * kBK * 2 + bn * cb + 2 * bn * kParamBox) + 4 * st * 8 + 64 + 16 * 32 * 4;
}

// Static tile choice: the weight-tile width BN and the split of K that
// minimise (waves of CTAs) x (work per CTA), preferring wide tiles.
TcCfg choose_tc(int M, int N, int K, int bits) {
    const DeviceInfo &di = device_info();
    TcCfg best{};
    double best_t = 1e300;
    const int nk = (K + kBK - 1) / kBK;
    const int mt = (M + kBM - 1) / kBM;
    for (int bn : {256, 128, 64}) {
        if (smem_bytes(bn, bits) > di.max_smem_optin) continue;
        const int nt = (N + bn - 1) / bn;
        for (int sp = 1; sp <= 16; sp *= 2) {
            const int kps = (nk + sp - 1) / sp;
            if (kps < 4 && sp > 1) break;
            const int splits = (nk + kps - 1) / kps;
            const long ctas = static_cast<long>(mt) * nt * splits;
            if (splits > 1 && static_cast<long>(mt) * nt >= di.sm_count) break;  // split K only to fill the GPU
            const long waves = (ctas + di.sm_count - 1) / di.sm_count;
            // per-CTA time ~ k-steps x max(MMA time ~ bn, fixed dequant+issue cost) + fixed epilogue/fill
            const double per_cta = kps * std::max(bn, 96) + 600.0 + (splits > 1 ? 200.0 : 0.0);
            const double t = waves * per_cta;
            if (t < best_t * 0.97) {
                best_t = t;
                best = TcCfg{bn, splits, kps, nk, mt, nt};
            }
        }
    }
    return best;
}

template <int WK, int BITS, bool BF16, int BN>
cudaError_t launch_tc(const CUtensorMap &am, const CUtensorMap &cm, const CUtensorMap &pm, const CUtensorMap &zm,
                      const TcArgs &a, const TcCfg &c, cudaStream_t s) {
    auto kern = tc_gemm_kernel<WK, BITS, BF16, BN>;
    static std::atomic<unsigned> configured{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned bit = 1u << (dev & 31);
    const int smem = smem_bytes(BN, BITS);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    dim3 grid(c.n_tiles, c.m_tiles, c.splits);
    const cudaError_t e = launch_pdl(kern, grid, dim3(kThreads), smem, s, am, cm, pm, zm, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// M >= 9 with fp16 / bf16 activations runs on the tensor cores; fp32
// activations stay on the SIMT path (rounding them to 16 bits would break the
// 1e-4 bar), and so do shapes whose packed rows or parameter rows are not a
// multiple of 16 bytes (the TMA row stride).
bool tc_eligible(int M, int K, int bits, int a_dtype, int bs) {
    if (M < 9 || a_dtype == 0) return false;
    if ((K * bits / 8) % 16 != 0) return false;
    if ((K / bs) % 8 != 0) return false;  // parameter rows (fp16 scales / zero points, fp32 absmax) in 16-byte units
    return encode_fn() != nullptr;
}

size_t tc_workspace_bytes(int M, int N, int K, int bits) {
    const TcCfg c = choose_tc(M, N, K, bits);
    return c.splits > 1 ? static_cast<size_t>(c.splits) * M * N * sizeof(float) : 0;
}

cudaError_t tc_gemm(const GemmProblem &p, void *ws, size_t ws_bytes, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const TcCfg c = choose_tc(p.M, p.N, p.K, p.bits);
    if (c.bn == 0) return cudaErrorNotSupported;
    CUtensorMap am, cm;
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(p.M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.K) * 2};
        const cuuint32_t box[2] = {kBK, kBM};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&am, p.a_dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                const_cast<void *>(p.A), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const int row_bytes = p.K * p.bits / 8;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(p.N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK * p.bits / 8), static_cast<cuuint32_t>(c.bn)};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&cm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(p.W), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // block parameters (and zero points): [N][nb] matrices read as boxes of 16
    // bytes x BN rows, one box per stage
    CUtensorMap pm, zm;
    {
        const bool cbk = p.kind == WK_CODEBOOK;
        const int pe = cbk ? 4 : 2;
        const int nb = p.K / p.bs;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nb), static_cast<cuuint64_t>(p.N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nb) * pe};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(kParamBox / pe), static_cast<cuuint32_t>(c.bn)};
        const cuuint32_t es[2] = {1, 1};
        const CUtensorMapDataType dt = cbk ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
        const void *pp = cbk ? static_cast<const void *>(p.absmax) : static_cast<const void *>(p.scales);
        if (enc(&pm, dt, 2, const_cast<void *>(pp), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        zm = pm;
        if (!cbk && p.zp_mode == ZP_TENSOR &&
            enc(&zm, dt, 2, const_cast<uint16_t *>(p.zp), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    TcArgs a{};
    a.scales = p.scales;
    a.zp = p.zp;
    a.zp_mode = p.zp_mode;
    a.zpv = p.uniform_zp;
    a.codebook = p.codebook;
    a.absmax = p.absmax;
    a.Y = p.Y;
    a.y_dtype = p.y_dtype;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.bs = p.bs;
    a.lbs = 31 - __builtin_clz(static_cast<unsigned>(p.bs));
    a.nb = p.K / p.bs;
    a.nk = c.nk;
    a.ks_per_split = c.ks_per_split;
    a.fault = fault_word();
    if (c.splits > 1) {
        const size_t need = static_cast<size_t>(c.splits) * p.M * p.N * sizeof(float);
        if (!ws || ws_bytes < need) return cudaErrorInvalidValue;
        a.partial = static_cast<float *>(ws);
    }
    const bool bf16 = p.a_dtype == 2;
    cudaError_t e = cudaErrorNotSupported;
#define QG_TC(WK_, B_, BF_, BN_)                                                                     \
    if (p.kind == WK_ && (WK_ == WK_CODEBOOK || p.bits == B_) && bf16 == BF_ && c.bn == BN_) \
        e = launch_tc<WK_, B_, BF_, BN_>(am, cm, pm, zm, a, c, s);                                \
    else
    QG_TC(WK_NBITS, 2, false, 256) QG_TC(WK_NBITS, 2, false, 128) QG_TC(WK_NBITS, 2, false, 64)
    QG_TC(WK_NBITS, 2, true, 256) QG_TC(WK_NBITS, 2, true, 128) QG_TC(WK_NBITS, 2, true, 64)
    QG_TC(WK_NBITS, 4, false, 256) QG_TC(WK_NBITS, 4, false, 128) QG_TC(WK_NBITS, 4, false, 64)
    QG_TC(WK_NBITS, 4, true, 256) QG_TC(WK_NBITS, 4, true, 128) QG_TC(WK_NBITS, 4, true, 64)
    QG_TC(WK_CODEBOOK, 4, false, 256) QG_TC(WK_CODEBOOK, 4, false, 128) QG_TC(WK_CODEBOOK, 4, false, 64)
    QG_TC(WK_CODEBOOK, 4, true, 256) QG_TC(WK_CODEBOOK, 4, true, 128) QG_TC(WK_CODEBOOK, 4, true, 64) {}
#undef QG_TC
    if (e != cudaSuccess) return e;
    if (c.splits > 1) {
        const size_t MN = static_cast<size_t>(p.M) * p.N;
        const int threads = 256;
        const int blocks = static_cast<int>(std::min<size_t>((MN + threads - 1) / threads, 8192));
        const cudaError_t e2 = launch_pdl(tc_splitk_reduce_kernel, dim3(blocks), dim3(threads), 0, s,
                                          static_cast<const float *>(a.partial), c.splits, MN, p.Y, p.y_dtype);
        return e2 != cudaSuccess ? e2 : cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace qg
