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
//    offset exactly.  For fp16 activations the zero point and the scale are
//    then applied with packed fp16 arithmetic (one rounding to fp16 of the
//    exact product); for bf16 activations the fp32 weight (q - zp) * s is
//    formed as the plain definition forms it and rounded once to bf16.
//    Codebook weights use a per-lane replicated table in shared memory and
//    fp32 products rounded once to the activation type.
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

constexpr int kBM = 256;  // activation rows per CTA tile: two MMA halves of kMH rows sharing the weight tile
constexpr int kMH = 128;
constexpr int kBK = 64;
constexpr int kDequantThreads = 512;  // 16 dequant + epilogue warps
constexpr int kThreads = 64 + kDequantThreads;  // warp 0 TMA, warp 1 MMA, warps 2-17 dequant + epilogue
constexpr int kParamBox = 16;         // bytes of block parameters per weight row per super-stage (one TMA box column)
constexpr int kCodeBox = 64;          // bytes of packed codes per weight row per super-stage
constexpr int kCodeSlots = 2;         // super-stages of codes / parameters in flight
constexpr int kSmemBudget = 227 * 1024;
constexpr int kSmemFixed = 1024 + 4096;  // alignment slack + barriers, tensor-memory slot, codebook table
// Three buffers:
//  * the activation ring: NA K steps of 128 x 64 activations (one TMA tile each),
//    released when the step's MMAs finish;
//  * the code ring: kCodeSlots super-stages of CS = kCodeBox / (64 * bits / 8)
//    K steps, holding the packed codes (kCodeBox bytes per weight row) and one
//    box of block parameters (and zero points) per weight row, released by the
//    dequant warps -- far fewer and larger TMA rows than one small box per step;
//  * two buffers of dequantized weights (the MMA's B operand).
__host__ __device__ constexpr int code_slot_bytes(int bn) { return bn * (kCodeBox + 2 * kParamBox); }
__host__ __device__ constexpr int wdq_bytes(int bn) { return bn * kBK * 2; }
__host__ __device__ constexpr int act_slots(int bn) {
    return (kSmemBudget - kSmemFixed - 2 * wdq_bytes(bn) - kCodeSlots * code_slot_bytes(bn)) / (kBM * kBK * 2) > 8
               ? 8
               : (kSmemBudget - kSmemFixed - 2 * wdq_bytes(bn) - kCodeSlots * code_slot_bytes(bn)) / (kBM * kBK * 2);
}

struct TcArgs {
    const uint16_t *scales;  // nbits, [N][nb] fp16
    const uint16_t *zp;      // nbits, [N][nb] fp16 (ZP_TENSOR)
    int zp_mode;
    float zpv;
    const float *codebook;   // codebook, [16]
    const float *absmax;     // codebook, [N][nb]
    void *Y;
    int y_dtype;
    float *partial;          // tail partials [tail tile x split][kBM][BN] (fp32)
    int M, N, K, bs, lbs, nb, nk;  // lbs = log2(bs)
    // Schedule: CTAs 0 .. full_tiles-1 compute whole tiles (whole K); the
    // remaining tiles are split along K into tail_splits pieces of tail_kps
    // steps each, one CTA per piece, summed afterwards in split order.
    int nt, full_tiles, tail_splits, tail_kps;
    int y_vec16;  // 16-bit Y with 16-byte aligned rows (N % 8 == 0, Y 16-byte aligned): packed stores
    // fp16 block parameters whose rows (nb * 2 bytes) are not a multiple of 16
    // bytes cannot be a tensor map: the producer warp copies them with 4-byte
    // cp.async instead (nb even); w_rows = rows of the weight tensors
    int par_plain, w_rows;
    // Split-precision passes (fp32 activations): wpart 1 makes the fp16 weight
    // operand the residual fp16(w - fp16(w)) of the fp32 weight w instead of
    // fp16(w); the epilogue multiplies activation row m by row_scale[m] (when
    // set) and, with acc, adds to the fp32 Y instead of writing it.
    int wpart, acc;
    const float *row_scale;
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

// 4 bytes global -> shared, asynchronous; src_bytes 0 writes zeros (nothing is read)
__device__ __forceinline__ void cp_async4(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}

// one arrival on `bar` once every cp.async this thread issued before has landed
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Block parameters of one 8-weight unit: fp16 pairs for the fp16 operand,
// fp32 values for the bf16 operand.
struct UnitPar {
    __half2 zp2, s2;  // fp16 operand
    float zpf, sf;    // bf16 operand
    bool lo;          // fp16 operand: the residual part of the weight
};

// One operand pair from two exact integer codes q (an fp16 pair).
//  fp16: (q - zp) * s with packed fp16 arithmetic.  For the integer and
//        half-integer zero points of the workloads q - zp is exact, so the
//        pair is the single fp16 rounding of the exact product.
//  bf16: the fp32 weight fl32(fl32(q - zp) * s) (two fp32 round-to-nearest
//        operations, no contraction), then one round-to-nearest to bf16.  No
//        fp16 intermediate, so products beyond fp16's range or below its
//        normal range keep bf16's.
template <bool BF16>
__device__ __forceinline__ uint32_t operand_pair(__half2 q, const UnitPar &u) {
    if constexpr (BF16) {
        const float2 qf = __half22float2(q);
        const float w0 = __fmul_rn(__fsub_rn(qf.x, u.zpf), u.sf);
        const float w1 = __fmul_rn(__fsub_rn(qf.y, u.zpf), u.sf);
        const __nv_bfloat162 b = __floats2bfloat162_rn(w0, w1);
        return *reinterpret_cast<const uint32_t *>(&b);
    } else {
        if (!u.lo) return h2_as_u32(__hmul2(__hsub2(q, u.zp2), u.s2));
        // the residual: w (exact in fp32) minus its fp16 rounding, rounded to fp16
        const float2 qf = __half22float2(q);
        const float zf = __low2float(u.zp2), sf = __low2float(u.s2);
        const float w0 = __fmul_rn(__fsub_rn(qf.x, zf), sf), w1 = __fmul_rn(__fsub_rn(qf.y, zf), sf);
        const __half2 hi = __floats2half2_rn(w0, w1);
        return h2_as_u32(__floats2half2_rn(w0 - __low2float(hi), w1 - __high2float(hi)));
    }
}

// 8 weights (k = 8c .. 8c+7 of one row) from their packed codes, as four
// operand pairs: the codes are first turned into exact fp16 integers, then
// operand_pair applies the zero point and the scale.
template <int BITS, bool BF16>
__device__ __forceinline__ uint4 dequant8_nbits(uint32_t codes, uint32_t codes_hi, const UnitPar &u) {
    uint32_t out[4];
    if constexpr (BITS == 8) {
        // codes: 8 bytes, one code each; a byte permute puts two codes under the
        // fp16 exponent of 1024 (0x64): (1024 + q0, 1024 + q1), exact for q < 1024
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t wsrc = j < 2 ? codes : codes_hi;
            const uint32_t h = __byte_perm(wsrc, 0x64646464u, (j & 1) ? 0x4342u : 0x4140u);
            const __half2 q = __hsub2(u32_as_h2(h), __floats2half2_rn(1024.f, 1024.f));
            out[j] = operand_pair<BF16>(q, u);
        }
    } else if constexpr (BITS == 2) {
        // codes: 16 bits, 8 codes; byte j holds codes 4j .. 4j+3
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t v = __byte_perm(codes, 0u, 0x4040u | (j * 0x0101u));  // byte j into bytes 0 and 2
            const uint32_t h01 = (v & 0x000C0003u) | 0x64006400u;  // (1024 + q0, 1024 + 4 q1)
            const uint32_t h23 = (v & 0x00C00030u) | 0x64006400u;  // (1024 + 16 q2, 1024 + 64 q3)
            const __half2 q01 = __hfma2(u32_as_h2(h01), __floats2half2_rn(1.f, 0.25f), __floats2half2_rn(-1024.f, -256.f));
            const __half2 q23 = __hfma2(u32_as_h2(h23), __floats2half2_rn(0.0625f, 0.015625f), __floats2half2_rn(-64.f, -16.f));
            out[2 * j] = operand_pair<BF16>(q01, u);
            out[2 * j + 1] = operand_pair<BF16>(q23, u);
        }
    } else {
        // codes: 32 bits, 8 codes; byte j holds codes 2j, 2j+1
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t v = __byte_perm(codes, 0u, 0x4040u | (j * 0x0101u));
            const uint32_t h = (v & 0x00F0000Fu) | 0x64006400u;  // (1024 + q0, 1024 + 16 q1)
            const __half2 q = __hfma2(u32_as_h2(h), __floats2half2_rn(1.f, 0.0625f), __floats2half2_rn(-1024.f, -64.f));
            out[j] = operand_pair<BF16>(q, u);
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

// Grouped (ragged expert) mode: expert e owns activation rows row_off[e] ..
// row_off[e+1]-1 and weight rows e*N .. e*N+N-1 of the stacked [E*N] weight
// tensors; its M tiles are numbered mt_prefix[e] .. mt_prefix[e+1]-1 (an
// expert the grouped launch leaves out has none).  Passed by value -- or,
// when `offs` is set, built by every CTA after the grid-dependency wait from
// those device-resident row offsets (offs[count + 1] int64); M tiles at or
// past the last prefix then have no work.
constexpr int kMaxGroups = 256;
template <bool G>
struct TcGroups {
    int unused;
};
template <>
struct TcGroups<true> {
    int count;
    const int64_t *offs;  // device offsets, or null: the tables below
    long long max_rows;   // offs[count] may not pass it
    int *status;          // set to 1 when the device offsets break the rules
    int mt_prefix[kMaxGroups + 1];
    int row_off[kMaxGroups + 1];
};

template <int WK, int BITS, bool BF16, int BN, bool GROUPED = false>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap act_map, const __grid_constant__ CUtensorMap code_map,
                   const __grid_constant__ CUtensorMap par_map, const __grid_constant__ CUtensorMap zp_map,
                   const TcArgs p, const __grid_constant__ TcGroups<GROUPED> grp) {
    constexpr int NS = act_slots(BN);
    static_assert(NS >= 3, "shared memory too small for the activation ring");
    constexpr int CB = kBK * BITS / 8;           // code bytes per row per K step
    constexpr int CS = kCodeBox / CB;            // K steps per super-stage
    constexpr int ACT_BYTES = kBM * kBK * 2;     // 32 KB: two 128-row halves, 16 KB apart
    constexpr int WDQ_BYTES = wdq_bytes(BN);
    constexpr int CODE_BYTES = BN * kCodeBox;
    constexpr int PAR_BYTES = BN * kParamBox;
    constexpr int PE = WK == WK_CODEBOOK ? 4 : 2;  // bytes per block parameter
    constexpr int PPB = kParamBox / PE;            // parameters per box row
    constexpr uint32_t TMEM_COLS = 2 * BN;       // one BN-column accumulator per 128-row half
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled tiles (pointer arithmetic on the
    // shared array keeps the accesses in the shared address space)
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char *act_s = smem;
    unsigned char *wdq_s = act_s + NS * ACT_BYTES;
    unsigned char *code_s = wdq_s + 2 * WDQ_BYTES;
    unsigned char *par_s = code_s + kCodeSlots * CODE_BYTES;
    unsigned char *zp_s = par_s + kCodeSlots * PAR_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(zp_s + kCodeSlots * PAR_BYTES);
    uint64_t *full = bars;                 // activation tile of a K step landed (count 1 + tx)
    uint64_t *empty = bars + NS;           // the step's MMAs finished: activation slot free (commit)
    uint64_t *wfull = bars + 2 * NS;       // dequantized weights written (count: dequant warps)
    uint64_t *wempty = bars + 2 * NS + 2;  // MMAs reading a dequant buffer finished (commit)
    uint64_t *accf = bars + 2 * NS + 4;    // all MMAs finished
    uint64_t *cfull = bars + 2 * NS + 5;   // codes + parameters of a super-stage landed (count 1 + tx)
    uint64_t *cempty = cfull + kCodeSlots; // the dequant warps are done with a code slot (count: dequant warps)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cempty + kCodeSlots);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *lut = reinterpret_cast<float *>(tmem_slot + 4);  // 16 x 32 floats (codebook)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int tile = blockIdx.x, ks0 = 0, nks = p.nk, pslot = -1;
    if (!GROUPED && tile >= p.full_tiles) {
        const int q = tile - p.full_tiles, r = q / p.tail_splits, z = q - r * p.tail_splits;
        tile = p.full_tiles + r;
        ks0 = z * p.tail_kps;
        nks = max(0, min(p.nk, ks0 + p.tail_kps) - ks0);
        pslot = p.tail_splits > 1 ? q : -1;  // an unsplit tail tile writes Y directly
    }
    int m0 = (tile / p.nt) * kBM, m_end = p.M, wrow = 0;
    const int n0 = (tile % p.nt) * BN;
    if constexpr (GROUPED) {
        // the expert owning M tile mt: the last e with mt_prefix[e] <= mt
        const int mt = tile / p.nt;
        int lo = 0, hi = grp.count;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (grp.mt_prefix[mid] <= mt) lo = mid;
            else hi = mid;
        }
        m0 = grp.row_off[lo] + (mt - grp.mt_prefix[lo]) * kBM;
        m_end = grp.row_off[lo + 1];
        wrow = lo * p.N;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&wfull[b], kDequantThreads / 32);
            mbar_init(&wempty[b], 1);
        }
        for (int c = 0; c < kCodeSlots; ++c) {
            mbar_init(&cfull[c], p.par_plain ? 33 : 1);  // + one cp.async arrival per producer lane
            mbar_init(&cempty[c], kDequantThreads / 32);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    // Launched as a programmatic dependent: the set-up above overlaps the
    // preceding kernel's tail and the next kernel may start launching as these
    // CTAs retire; nothing the call reads or writes is touched before
    // pdl_wait() (any buffer may have been written by the preceding kernel).
    pdl_launch_dependents();
    pdl_wait();
    if constexpr (WK == WK_CODEBOOK) {
        for (int i = threadIdx.x; i < 16 * 32; i += kThreads) lut[i] = __ldg(p.codebook + (i >> 5));
    }
    // device offsets: every CTA numbers the experts' M tiles itself (thread e
    // counts expert e's tiles, a block-wide scan adds them up) into shared
    // memory -- the codebook table's space, which the MatMulNBits grouped
    // launch does not use -- for the search below.  Offsets that do not start
    // at 0, decrease, or end past max_rows leave every tile without work.
    int *spre = reinterpret_cast<int *>(lut);
    if constexpr (GROUPED) {
        static_assert(!GROUPED || WK == WK_NBITS, "grouped launches are MatMulNBits");
        static_assert(kMaxGroups + 1 + kThreads / 32 <= 16 * 32, "the prefix fits the table's space");
        static_assert(kMaxGroups <= kThreads, "one thread per expert");
        if (grp.offs) {
            int *wsum = spre + kMaxGroups + 1;  // the warps' tile totals
            const int e = threadIdx.x, E = grp.count;
            int cnt = 0, bad = 0;
            if (e < E) {
                const long long o0 = __ldcg(grp.offs + e), o1 = __ldcg(grp.offs + e + 1);
                bad = o1 < o0 || (e == 0 && o0 != 0) || (e == E - 1 && o1 > grp.max_rows);
                cnt = o1 > o0 ? static_cast<int>((o1 - o0 + kBM - 1) / kBM) : 0;
            }
            int inc = cnt;  // inclusive scan inside the warp
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += v;
            }
            if (lane == 31) wsum[warp] = inc;
            bad = __syncthreads_or(bad);
            int base = 0;  // the earlier warps' totals
            for (int w = 0; w < warp; ++w) base += wsum[w];
            if (e < E) spre[e] = bad ? 0 : base + inc - cnt;
            if (e == E - 1) spre[E] = bad ? 0 : base + inc;
            if (bad && blockIdx.x == 0 && e == 0 && grp.status) *grp.status = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if constexpr (GROUPED) {
        if (grp.offs) {  // the tile prefix built above
            const int mt = tile / p.nt;
            if (mt >= spre[grp.count]) {
                nks = 0;  // no work: no copies, no MMAs, no rows written
                m0 = m_end = wrow = 0;
            } else {
                int lo = 0, hi = grp.count;
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (spre[mid] <= mt) lo = mid;
                    else hi = mid;
                }
                m0 = static_cast<int>(__ldcg(grp.offs + lo)) + (mt - spre[lo]) * kBM;
                m_end = static_cast<int>(__ldcg(grp.offs + lo + 1));
                wrow = lo * p.N;
            }
        }
    }

    if (warp == 0 && p.par_plain) {
        // ------------------------------------------------------------ producer, parameters by cp.async
        // Lane 0 waits and issues the tensor copies of codes and activations
        // as below; every lane copies the parameter boxes of its rows (16
        // bytes = 8 fp16 per row) in 4-byte pieces, zero past N or past nb.
        const bool zt = WK == WK_NBITS && p.zp_mode == ZP_TENSOR;
        __syncwarp();
        for (int i = 0; i < nks; ++i) {
            const int ks = ks0 + i;
            bool ok = true;
            if (i % CS == 0) {
                const int j = i / CS, c = j % kCodeSlots;
                if (lane == 0) ok = mbar_wait(&cempty[c], ((j / kCodeSlots) & 1) ^ 1, abort_flag, p.fault, FAULT_WAIT_TC);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&cfull[c], CODE_BYTES);
                    tma_load_2d(code_s + c * CODE_BYTES, &code_map, ks * CB, wrow + n0, &cfull[c]);
                }
                const int pcol = (ks * kBK / p.bs) / PPB * PPB;
                for (int r = lane; r < BN; r += 32) {
                    const int grow = wrow + n0 + r;
#pragma unroll
                    for (int q = 0; q < kParamBox / 4; ++q) {
                        const int col = pcol + 2 * q;  // two fp16 per piece; nb is even
                        const bool in = grow < p.w_rows && col < p.nb;
                        const size_t off = in ? (static_cast<size_t>(grow) * p.nb + col) : 0;
                        cp_async4(par_s + c * PAR_BYTES + r * kParamBox + 4 * q, p.scales + off, in ? 4u : 0u);
                        if (zt) cp_async4(zp_s + c * PAR_BYTES + r * kParamBox + 4 * q, p.zp + off, in ? 4u : 0u);
                    }
                }
                cp_async_arrive(&cfull[c]);
            }
            if (lane == 0) {
                const int s = i % NS;
                ok = mbar_wait(&empty[s], ((i / NS) & 1) ^ 1, abort_flag, p.fault, FAULT_WAIT_TC);
                if (ok) {
                    mbar_arrive_expect_tx(&full[s], ACT_BYTES);
                    tma_load_2d(act_s + s * ACT_BYTES, &act_map, ks * kBK, m0, &full[s]);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const bool zt = WK == WK_NBITS && p.zp_mode == ZP_TENSOR;
            for (int i = 0; i < nks; ++i) {
                const int ks = ks0 + i;
                if (i % CS == 0) {  // codes and block parameters of the next CS steps
                    const int j = i / CS, c = j % kCodeSlots;
                    if (!mbar_wait(&cempty[c], ((j / kCodeSlots) & 1) ^ 1, abort_flag, p.fault, FAULT_WAIT_TC)) break;
                    mbar_arrive_expect_tx(&cfull[c], CODE_BYTES + PAR_BYTES * (zt ? 2 : 1));
                    const int pcol = (ks * kBK / p.bs) / PPB * PPB;  // first parameter column of the box
                    tma_load_2d(code_s + c * CODE_BYTES, &code_map, ks * CB, wrow + n0, &cfull[c]);
                    tma_load_2d(par_s + c * PAR_BYTES, &par_map, pcol, wrow + n0, &cfull[c]);
                    if (zt) tma_load_2d(zp_s + c * PAR_BYTES, &zp_map, pcol, wrow + n0, &cfull[c]);
                }
                const int s = i % NS;
                if (!mbar_wait(&empty[s], ((i / NS) & 1) ^ 1, abort_flag, p.fault, FAULT_WAIT_TC)) break;
                mbar_arrive_expect_tx(&full[s], ACT_BYTES);
                tma_load_2d(act_s + s * ACT_BYTES, &act_map, ks * kBK, m0, &full[s]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kMH, BN, BF16);
            const bool two = m0 + kMH < m_end;  // the second half holds rows below M (the expert's end)
            bool ok = true;
            for (int i = 0; i < nks && ok; ++i) {
                const int s = i % NS, b = i & 1;
                ok = mbar_wait(&full[s], (i / NS) & 1, abort_flag, p.fault, FAULT_WAIT_TC) &&
                     mbar_wait(&wfull[b], (i >> 1) & 1, abort_flag, p.fault, FAULT_WAIT_TC);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ad = sdesc_k128(smem_u32(act_s + s * ACT_BYTES));
                const uint64_t ad1 = sdesc_k128(smem_u32(act_s + s * ACT_BYTES + kMH * kBK * 2));
                const uint64_t bd = sdesc_k128(smem_u32(wdq_s + b * WDQ_BYTES));
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k) {  // +32 bytes per K=16 step inside the swizzle row
                    umma_f16(tmem, ad + 2 * k, bd + 2 * k, idesc, (i > 0 || k > 0) ? 1u : 0u);
                    if (two) umma_f16(tmem + BN, ad1 + 2 * k, bd + 2 * k, idesc, (i > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(&empty[s]);   // ring slot (activations, codes) free for the next TMA fill
                umma_commit(&wempty[b]);  // dequant buffer free
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
            code_off[j] = r * kCodeBox + c * (CB / 8);
            wdq_off[j] = swz128(r, c);
            par_off[j] = r * kParamBox + ((8 * c) >> p.lbs) * PE;  // block of this chunk within the stage
        }
        const uint32_t zpu = __half_as_ushort(__float2half_rn(p.zpv)) * 0x10001u;  // fp16 operand: zp as an fp16 pair
        const bool zt = WK == WK_NBITS && p.zp_mode == ZP_TENSOR;
        for (int i = 0; i < nks; ++i) {
            const int b = i & 1, j = i / CS, cslot = j % kCodeSlots;
            if (i % CS == 0 && !mbar_wait(&cfull[cslot], (j / kCodeSlots) & 1, abort_flag, p.fault, FAULT_WAIT_TC)) break;
            if (!mbar_wait(&wempty[b], ((i >> 1) & 1) ^ 1, abort_flag, p.fault, FAULT_WAIT_TC)) break;
            const int kb = (ks0 + i) * kBK;
            const int pc0 = ((kb >> p.lbs) % PPB) * PE;  // first block of the stage inside its parameter box
            const unsigned char *__restrict__ cs = code_s + cslot * CODE_BYTES + (i % CS) * CB;
            const unsigned char *__restrict__ ps = par_s + cslot * PAR_BYTES + pc0;
            const unsigned char *__restrict__ zs = zp_s + cslot * PAR_BYTES + pc0;
            unsigned char *__restrict__ ws = wdq_s + b * WDQ_BYTES;
            uint32_t codes[UPT], codes_hi[UPT], pv[UPT], zv[UPT];
#pragma unroll
            for (int j = 0; j < UPT; ++j) {
                codes_hi[j] = 0u;
                if constexpr (WK == WK_NBITS) {
                    if constexpr (BITS == 8) {  // 8 weights = 8 bytes
                        const uint2 v = *reinterpret_cast<const uint2 *>(cs + code_off[j]);
                        codes[j] = v.x;
                        codes_hi[j] = v.y;
                    } else {
                        codes[j] = BITS == 2 ? static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(cs + code_off[j]))
                                             : *reinterpret_cast<const uint32_t *>(cs + code_off[j]);
                    }
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
                    UnitPar u;
                    u.lo = p.wpart != 0;
                    if constexpr (BF16) {
                        u.zpf = zt ? h2f(static_cast<uint16_t>(zv[j])) : p.zpv;
                        u.sf = h2f(static_cast<uint16_t>(pv[j]));
                    } else {
                        u.zp2 = u32_as_h2(zt ? zv[j] * 0x10001u : zpu);
                        u.s2 = u32_as_h2(pv[j] * 0x10001u);
                    }
                    w = dequant8_nbits<BITS, BF16>(codes[j], codes_hi[j], u);
                } else {
                    w = dequant8_codebook<BF16>(codes[j], __uint_as_float(pv[j]), lut_lane);
                }
                *reinterpret_cast<uint4 *>(ws + wdq_off[j]) = w;
            }
            fence_async_smem();  // make the generic-proxy stores visible to the tensor core
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&wfull[b]);
                if (i % CS == CS - 1 || i == nks - 1) mbar_arrive(&cempty[cslot]);  // codes of this slot consumed
            }
        }
        // ------------------------------------------------------------ epilogue
        const bool ok = mbar_wait(accf, 0, abort_flag, p.fault, FAULT_WAIT_TC);
        tc_fence_after();
        const int sub = warp & 3;  // tensor-memory sub-partition this warp may read
        constexpr int NQ = kDequantThreads / 128;  // warps sharing a sub-partition split its columns
        const int cq = (warp - 2) >> 2;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(sub * 32) << 16);
        // columns [0, BN) hold rows m0 .. m0+127, [BN, 2 BN) rows m0+128 .. m0+255
        constexpr int CW = 2 * BN / NQ >= 32 ? 2 * BN / NQ : 32;
#pragma unroll 1
        for (int cc = cq * CW; cc < (cq + 1) * CW && cc < 2 * BN; cc += 32) {
            uint32_t r[32];
            tmem_ld32(lane_addr + cc, r);
            const int h = cc / BN, c0 = cc - h * BN;
            const int row = h * kMH + sub * 32 + lane, m = m0 + row;
            if (!ok || nks == 0 || m >= m_end) continue;  // rows past M (the expert's end) are never read back
            const int nb0 = n0 + c0;
            if (pslot >= 0) {  // a tail piece: the whole 32-column row segment (columns past N are ignored)
                float4 *dst = reinterpret_cast<float4 *>(p.partial + (static_cast<size_t>(pslot) * kBM + row) * BN + c0);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                         __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            } else if (p.row_scale) {  // split-precision pass: fp32 Y = (acc ? Y : 0) + sum * row scale
                const float rs = p.row_scale[m];
                float *y = static_cast<float *>(p.Y) + static_cast<size_t>(m) * p.N + nb0;
                if ((p.N & 3) == 0 && nb0 + 32 <= p.N) {
                    float4 *dst = reinterpret_cast<float4 *>(y);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float4 v = make_float4(__uint_as_float(r[4 * j]) * rs, __uint_as_float(r[4 * j + 1]) * rs,
                                               __uint_as_float(r[4 * j + 2]) * rs, __uint_as_float(r[4 * j + 3]) * rs);
                        if (p.acc) {
                            const float4 o = dst[j];
                            v = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
                        }
                        dst[j] = v;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (nb0 + j < p.N) y[j] = (p.acc ? y[j] : 0.f) + __uint_as_float(r[j]) * rs;
                }
            } else if (p.y_dtype == 0 && (p.N & 3) == 0 && nb0 + 32 <= p.N) {
                float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.Y) + static_cast<size_t>(m) * p.N + nb0);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                         __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            } else if (p.y_vec16 && nb0 + 32 <= p.N) {  // 16-bit output: 32 values as four 16-byte stores
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.Y) + static_cast<size_t>(m) * p.N + nb0);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t h[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float lo = __uint_as_float(r[8 * j + 2 * q]), hi = __uint_as_float(r[8 * j + 2 * q + 1]);
                        if (p.y_dtype == 1) {
                            h[q] = h2_as_u32(__floats2half2_rn(lo, hi));
                        } else {
                            const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
                            h[q] = *reinterpret_cast<const uint32_t *>(&b);
                        }
                    }
                    dst[j] = make_uint4(h[0], h[1], h[2], h[3]);
                }
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

// fp32 activations for the split-precision passes: per row m, e = the exponent
// of the largest |a| (clamped to [-110, 117]), a' = a * 2^(14 - e) (largest
// magnitude in [2^14, 2^15): fp16 range), hi = fp16(a'), lo = fp16(a' - hi),
// and the row's output multiplier 2^(e - 14).  One CTA per row.
__global__ void split_rows_kernel(const float *__restrict__ A, int K, __half *__restrict__ hi,
                                  __half *__restrict__ lo, float *__restrict__ row_scale) {
    __shared__ float wmax[32];
    pdl_wait();
    pdl_launch_dependents();
    const size_t base = static_cast<size_t>(blockIdx.x) * K;
    float mx = 0.f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) mx = fmaxf(mx, fabsf(A[base + k]));
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x < 32) {
        mx = threadIdx.x < blockDim.x / 32 ? wmax[threadIdx.x] : 0.f;
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (threadIdx.x == 0) wmax[0] = mx;
    }
    __syncthreads();
    const unsigned bits = __float_as_uint(wmax[0]);
    const int ef = static_cast<int>((bits >> 23) & 0xFFu);
    const int e = (bits == 0u || ef == 255) ? 0 : min(max(ef - 127, -110), 117);
    const float up = exp2i(14 - e);
    if (threadIdx.x == 0) row_scale[blockIdx.x] = exp2i(e - 14);
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const float x = A[base + k] * up;
        const __half h = __float2half_rn(x);
        hi[base + k] = h;
        lo[base + k] = __float2half_rn(x - __half2float(h));
    }
}

// Y for the tail tiles: the sum of each tile's K pieces in split order.
__global__ void tc_tail_reduce_kernel(const float *__restrict__ partial, int tail_tiles, int splits, int bn,
                                      int full_tiles, int nt, int M, int N, void *Y, int y_dtype) {
    pdl_wait();
    pdl_launch_dependents();
    const size_t per_tile = static_cast<size_t>(kBM) * bn;
    const size_t total = static_cast<size_t>(tail_tiles) * per_tile;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(i / per_tile);
        const int e = static_cast<int>(i - r * per_tile), row = e / bn, col = e - row * bn;
        const int tile = full_tiles + r;
        const int m = (tile / nt) * kBM + row, n = (tile % nt) * bn + col;
        if (m >= M || n >= N) continue;
        float s = 0.f;
        for (int z = 0; z < splits; ++z) s += partial[(static_cast<size_t>(r) * splits + z) * per_tile + e];
        store_y_elem(Y, y_dtype, static_cast<size_t>(m) * N + n, s);
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
    int bn, nk, mt, nt, full_tiles, tail_tiles, tail_splits, tail_kps;
    int grid() const { return full_tiles + tail_tiles * tail_splits; }
    size_t partial_bytes() const {
        return tail_splits > 1 ? static_cast<size_t>(tail_tiles) * tail_splits * kBM * bn * sizeof(float) : 0;
    }
};

int smem_bytes(int bn, int bits) {
    (void)bits;
    return kSmemFixed + act_slots(bn) * kBM * kBK * 2 + 2 * wdq_bytes(bn) + kCodeSlots * code_slot_bytes(bn);
}

// Static tile choice (no timing, no tuning): the weight-tile width BN, and the
// schedule -- whole tiles fill complete waves of CTAs, the tiles left over are
// split along K over the SMs (their pieces summed afterwards) -- that minimise
// a cost model in units of about 1.4 ns:
//  * per K step, the MMAs (~halves x BN; N=256 MMAs run at full rate, narrower
//    ones lose about a third to shared-memory bandwidth) or the dequant
//    (~1.4 BN + a fixed cost), whichever is larger;
//  * per CTA, the pipeline fill and the epilogue;
//  * for split tail tiles, writing and reducing their fp32 pieces through HBM.
TcCfg choose_tc(int M, int N, int K, int bits) {
    const DeviceInfo &di = device_info();
    const int sms = di.sm_count;
    TcCfg best{};
    double best_t = 1e300;
    const int nk = (K + kBK - 1) / kBK;
    const int mt = (M + kBM - 1) / kBM;
    const int halves = M > kMH ? 2 : 1;
    for (int bn : {256, 128, 64}) {
        if (smem_bytes(bn, bits) > di.max_smem_optin) continue;
        const int nt = (N + bn - 1) / bn;
        const long tiles = static_cast<long>(mt) * nt;
        const double step = std::max(halves * bn * (bn >= 256 ? 1.0 : 1.45), 1.4 * bn + 100.0);
        const long full_waves = tiles / sms;
        TcCfg c{bn, nk, mt, nt, static_cast<int>(full_waves * sms), static_cast<int>(tiles - full_waves * sms), 1, nk};
        double t = full_waves * (nk * step + 800.0);
        if (c.tail_tiles > 0) {
            // split the tail over the SMs, in whole 4-step code super-stages
            int sp = std::max(1, std::min(sms / c.tail_tiles, nk / 4));
            int kps = ((nk + sp - 1) / sp + 3) / 4 * 4;
            sp = (nk + kps - 1) / kps;
            if (sp > 1) {
                c.tail_splits = sp;
                c.tail_kps = kps;
                t += kps * step + 800.0 + (sp + 1.0) * c.tail_tiles * kBM * bn * 4.0 / 9520.0;
            } else {
                t += nk * step + 800.0;
            }
        }
        if (t < best_t * 0.97) {
            best_t = t;
            best = c;
        }
    }
    return best;
}

template <int WK, int BITS, bool BF16, int BN, bool GROUPED = false>
cudaError_t launch_tc(const CUtensorMap &am, const CUtensorMap &cm, const CUtensorMap &pm, const CUtensorMap &zm,
                      const TcArgs &a, int grid_x, const TcGroups<GROUPED> &grp, cudaStream_t s) {
    auto kern = tc_gemm_kernel<WK, BITS, BF16, BN, GROUPED>;
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
    const cudaError_t e = launch_pdl(kern, dim3(grid_x), dim3(kThreads), smem, s, am, cm, pm, zm, a, grp);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Tensor maps of one problem: activations [M][K] (128-byte swizzled boxes of
// 64 x 256), codes [w_rows][K*bits/8] and block parameters (and zero points)
// [w_rows][K/bs] in boxes of BN rows.  w_rows is N, or E*N for the stacked
// experts of a grouped launch.
cudaError_t build_maps(PFN_cuTensorMapEncodeTiled_v12000 enc, const GemmProblem &p, int bn, long long w_rows,
                       CUtensorMap &am, CUtensorMap &cm, CUtensorMap &pm, CUtensorMap &zm) {
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
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(w_rows)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(kCodeBox), static_cast<cuuint32_t>(bn)};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&cm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(p.W), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // block parameters (and zero points): [rows][nb] matrices read as boxes of
    // 16 bytes x BN rows, one box per stage -- unless their rows are not a
    // multiple of 16 bytes (then the kernel copies them without a map)
    if (p.kind == WK_NBITS && (p.K / p.bs) % 8 != 0) {
        pm = cm;
        zm = cm;
        return cudaSuccess;
    }
    const bool cbk = p.kind == WK_CODEBOOK;
    const int pe = cbk ? 4 : 2;
    const int nb = p.K / p.bs;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nb), static_cast<cuuint64_t>(w_rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nb) * pe};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kParamBox / pe), static_cast<cuuint32_t>(bn)};
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
    return cudaSuccess;
}

TcArgs make_args(const GemmProblem &p, const TcCfg &c) {
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
    a.nt = c.nt;
    a.full_tiles = c.full_tiles;
    a.tail_splits = c.tail_splits;
    a.tail_kps = c.tail_kps;
    a.y_vec16 = p.y_dtype != 0 && (p.N & 7) == 0 && (reinterpret_cast<uintptr_t>(p.Y) & 15u) == 0;
    a.par_plain = p.kind == WK_NBITS && (p.K / p.bs) % 8 != 0;
    a.w_rows = p.N;
    a.wpart = p.tc_wpart;
    a.acc = p.tc_acc;
    a.row_scale = p.tc_row_scale;
    a.fault = fault_word();
    return a;
}

}  // namespace

// M >= 9 with fp16 / bf16 activations runs on the tensor cores; fp32
// activations stay on the SIMT path (rounding them to 16 bits would break the
// 1e-4 bar), and so do shapes whose packed rows or parameter rows are not a
// multiple of 16 bytes (the TMA row stride).
bool tc_eligible(int M, int K, int bits, int a_dtype, int bs, int kind) {
    if (M < 9 || a_dtype == 0) return false;
    if (bits == 3) return false;  // 3-bit codes (8 per 3 bytes) run on the SIMT path
    if ((K * bits / 8) % 16 != 0) return false;
    // parameter rows: a tensor map needs 16-byte rows (nb % 8 == 0); otherwise
    // the fp16 scales / zero points of MatMulNBits are copied in 4-byte pieces
    // (nb even).  The codebook's fp32 absmax always uses the map.
    if ((K / bs) % 8 != 0 && (kind != WK_NBITS || (K / bs) % 2 != 0)) return false;
    return encode_fn() != nullptr;
}

size_t tc_workspace_bytes(int M, int N, int K, int bits) {
    const TcCfg c = choose_tc(M, N, K, bits);
    return c.partial_bytes();
}

cudaError_t tc_gemm(const GemmProblem &p, void *ws, size_t ws_bytes, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    TcCfg c = choose_tc(p.M, p.N, p.K, p.bits);
    if (c.bn == 0) return cudaErrorNotSupported;
    if (p.tc_row_scale) {  // split-precision passes write (or add to) Y directly: every tile takes the whole K
        c.full_tiles += c.tail_tiles;
        c.tail_tiles = 0;
        c.tail_splits = 1;
        c.tail_kps = c.nk;
    }
    CUtensorMap am, cm, pm, zm;
    const cudaError_t me = build_maps(enc, p, c.bn, p.N, am, cm, pm, zm);
    if (me != cudaSuccess) return me;
    TcArgs a = make_args(p, c);
    if (c.partial_bytes()) {
        if (!ws || ws_bytes < c.partial_bytes()) return cudaErrorInvalidValue;
        a.partial = static_cast<float *>(ws);
    }
    const bool bf16 = p.a_dtype == 2;
    cudaError_t e = cudaErrorNotSupported;
#define QG_TC(WK_, B_, BF_, BN_)                                                                     \
    if (p.kind == WK_ && (WK_ == WK_CODEBOOK || p.bits == B_) && bf16 == BF_ && c.bn == BN_) \
        e = launch_tc<WK_, B_, BF_, BN_>(am, cm, pm, zm, a, c.grid(), TcGroups<false>{}, s);       \
    else
    QG_TC(WK_NBITS, 2, false, 256) QG_TC(WK_NBITS, 2, false, 128) QG_TC(WK_NBITS, 2, false, 64)
    QG_TC(WK_NBITS, 2, true, 256) QG_TC(WK_NBITS, 2, true, 128) QG_TC(WK_NBITS, 2, true, 64)
    QG_TC(WK_NBITS, 4, false, 256) QG_TC(WK_NBITS, 4, false, 128) QG_TC(WK_NBITS, 4, false, 64)
    QG_TC(WK_NBITS, 4, true, 256) QG_TC(WK_NBITS, 4, true, 128) QG_TC(WK_NBITS, 4, true, 64)
    QG_TC(WK_NBITS, 8, false, 256) QG_TC(WK_NBITS, 8, false, 128) QG_TC(WK_NBITS, 8, false, 64)
    QG_TC(WK_NBITS, 8, true, 256) QG_TC(WK_NBITS, 8, true, 128) QG_TC(WK_NBITS, 8, true, 64)
    QG_TC(WK_CODEBOOK, 4, false, 256) QG_TC(WK_CODEBOOK, 4, false, 128) QG_TC(WK_CODEBOOK, 4, false, 64)
    QG_TC(WK_CODEBOOK, 4, true, 256) QG_TC(WK_CODEBOOK, 4, true, 128) QG_TC(WK_CODEBOOK, 4, true, 64) {}
#undef QG_TC
    if (e != cudaSuccess) return e;
    if (c.partial_bytes()) {
        const size_t total = static_cast<size_t>(c.tail_tiles) * kBM * c.bn;
        const int threads = 256;
        const int blocks = static_cast<int>(std::min<size_t>((total + threads - 1) / threads, 8192));
        const cudaError_t e2 = launch_pdl(tc_tail_reduce_kernel, dim3(blocks), dim3(threads), 0, s,
                                          static_cast<const float *>(a.partial), c.tail_tiles, c.tail_splits, c.bn,
                                          c.full_tiles, c.nt, p.M, p.N, p.Y, p.y_dtype);
        return e2 != cudaSuccess ? e2 : cudaGetLastError();
    }
    return cudaSuccess;
}

// Ragged expert GEMM on the tensor cores: one launch over the M tiles of every
// expert with at least min_rows rows (the others are left to the caller);
// p.M is the total row count, p.N the rows of one expert, p.W / p.scales /
// p.zp the stacked [E][N][...] tensors.  No K split.
cudaError_t tc_gemm_grouped(const GemmProblem &p, const int64_t *offsets, int E, int min_rows, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc || E > kMaxGroups || p.kind != WK_NBITS) return cudaErrorNotSupported;
    TcGroups<true> g{};
    g.count = E;
    int tiles_m = 0, big = 0, rows_big = 0;
    for (int e = 0; e < E; ++e) {
        const int64_t c = offsets[e + 1] - offsets[e];
        g.mt_prefix[e] = tiles_m;
        g.row_off[e] = static_cast<int>(offsets[e]);
        if (c >= min_rows) {
            tiles_m += static_cast<int>((c + kBM - 1) / kBM);
            ++big;
            rows_big += static_cast<int>(c);
        }
    }
    g.mt_prefix[E] = tiles_m;
    g.row_off[E] = static_cast<int>(offsets[E]);
    if (tiles_m == 0) return cudaSuccess;
    // tile width from the static model at the experts' mean row count
    TcCfg c = choose_tc(std::max(min_rows, rows_big / big), p.N, p.K, p.bits);
    if (c.bn == 0) return cudaErrorNotSupported;
    // Each M tile is used by one expert only, so a tile's fixed costs (tensor
    // memory, barriers, pipeline fill, epilogue) are spread over few K steps:
    // take the widest tile that fits the experts' N (grouped launches are
    // instantiated for 128- and 256-wide tiles).
    const int bn = (p.N >= 256 && smem_bytes(256, p.bits) <= device_info().max_smem_optin) ? 256 : 128;
    if (c.bn != bn) {
        c.bn = bn;
        c.nt = (p.N + bn - 1) / bn;
    }
    c.mt = tiles_m;
    c.full_tiles = tiles_m * c.nt;
    c.tail_tiles = 0;
    c.tail_splits = 1;
    c.tail_kps = c.nk;
    CUtensorMap am, cm, pm, zm;
    const cudaError_t me = build_maps(enc, p, c.bn, static_cast<long long>(E) * p.N, am, cm, pm, zm);
    if (me != cudaSuccess) return me;
    TcArgs a = make_args(p, c);
    a.w_rows = E * p.N;
    const bool bf16 = p.a_dtype == 2;
    const int grid = c.full_tiles;
#define QG_TCG(B_, BF_, BN_) \
    if (p.bits == B_ && bf16 == BF_ && c.bn == BN_) return launch_tc<WK_NBITS, B_, BF_, BN_, true>(am, cm, pm, zm, a, grid, g, s);
    QG_TCG(4, false, 256) QG_TCG(4, false, 128) QG_TCG(4, true, 256) QG_TCG(4, true, 128)
    QG_TCG(2, false, 256) QG_TCG(2, false, 128) QG_TCG(2, true, 256) QG_TCG(2, true, 128)
    QG_TCG(8, false, 256) QG_TCG(8, false, 128) QG_TCG(8, true, 256) QG_TCG(8, true, 128)
#undef QG_TCG
    return cudaErrorNotSupported;
}

// The same grouped launch from device-resident offsets (no host copy of them):
// the grid covers the most M tiles any offsets within max_rows rows can need,
// ceil(max_rows / kBM) + E; every CTA numbers the tiles from the offsets
// itself and tiles past the real count exit.  Every expert with rows takes
// the tensor cores.  p.M = max_rows.
cudaError_t tc_gemm_grouped_dev(const GemmProblem &p, const int64_t *offsets_dev, int E, int *status, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc || E > kMaxGroups || p.kind != WK_NBITS) return cudaErrorNotSupported;
    TcGroups<true> g{};
    g.count = E;
    g.offs = offsets_dev;
    g.max_rows = p.M;
    g.status = status;
    const int tiles_m = (p.M + kBM - 1) / kBM + E;
    TcCfg c = choose_tc(std::max(kBM, p.M / E), p.N, p.K, p.bits);
    if (c.bn == 0) return cudaErrorNotSupported;
    const int bn = (p.N >= 256 && smem_bytes(256, p.bits) <= device_info().max_smem_optin) ? 256 : 128;
    c.bn = bn;
    c.nt = (p.N + bn - 1) / bn;
    c.mt = tiles_m;
    c.full_tiles = tiles_m * c.nt;
    c.tail_tiles = 0;
    c.tail_splits = 1;
    c.tail_kps = c.nk;
    CUtensorMap am, cm, pm, zm;
    const cudaError_t e = build_maps(enc, p, c.bn, static_cast<long long>(E) * p.N, am, cm, pm, zm);
    if (e != cudaSuccess) return e;
    TcArgs a = make_args(p, c);
    a.w_rows = E * p.N;
    const bool bf16 = p.a_dtype == 2;
    const int grid = c.full_tiles;
#define QG_TCG(B_, BF_, BN_) \
    if (p.bits == B_ && bf16 == BF_ && c.bn == BN_) return launch_tc<WK_NBITS, B_, BF_, BN_, true>(am, cm, pm, zm, a, grid, g, s);
    QG_TCG(4, false, 256) QG_TCG(4, false, 128) QG_TCG(4, true, 256) QG_TCG(4, true, 128)
    QG_TCG(2, false, 256) QG_TCG(2, false, 128) QG_TCG(2, true, 256) QG_TCG(2, true, 128)
    QG_TCG(8, false, 256) QG_TCG(8, false, 128) QG_TCG(8, true, 256) QG_TCG(8, true, 128)
#undef QG_TCG
    return cudaErrorNotSupported;
}

size_t split_workspace_bytes(int M, int K) {
    const size_t part = (static_cast<size_t>(M) * K * 2 + 255) / 256 * 256;
    return 2 * part + (static_cast<size_t>(M) * 4 + 255) / 256 * 256;
}

bool split_eligible(const GemmProblem &p) {
    return p.a_dtype == 0 && p.y_dtype == 0 && p.kind == WK_NBITS && p.zp_mode != ZP_PACKED && p.M >= kSplitMinRows &&
           tc_eligible(p.M, p.K, p.bits, 1, p.bs, p.kind);
}

// Y = rs (A_hi w_hi + A_hi w_lo + A_lo w_hi): three tensor-core passes over the
// activations split by split_rows_kernel, in that fixed order (the first
// writes Y, the others add to it).  A_lo w_lo (below 2^-22 of each product)
// is left out.
cudaError_t split_gemm(const GemmProblem &p, void *ws, size_t ws_bytes, cudaStream_t s) {
    if (!ws || ws_bytes < split_workspace_bytes(p.M, p.K)) return cudaErrorInvalidValue;
    const size_t part = (static_cast<size_t>(p.M) * p.K * 2 + 255) / 256 * 256;
    __half *hi = static_cast<__half *>(ws);
    __half *lo = reinterpret_cast<__half *>(static_cast<char *>(ws) + part);
    float *rs = reinterpret_cast<float *>(static_cast<char *>(ws) + 2 * part);
    cudaError_t e = launch_pdl(split_rows_kernel, dim3(p.M), dim3(256), 0, s, static_cast<const float *>(p.A), p.K, hi,
                               lo, rs);
    if (e != cudaSuccess) return e;
    GemmProblem q = p;
    q.a_dtype = 1;
    q.tc_row_scale = rs;
    const void *a_of[3] = {hi, hi, lo};
    for (int pass = 0; pass < 3; ++pass) {
        q.A = a_of[pass];
        q.tc_wpart = pass == 1 ? 1 : 0;
        q.tc_acc = pass > 0 ? 1 : 0;
        e = tc_gemm(q, nullptr, 0, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace qg
