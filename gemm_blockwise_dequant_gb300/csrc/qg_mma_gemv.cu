// qg_mma_gemv.cu -- 2-bit MatMulNBits GEMV / small-M GEMM on the tensor
// cores through warp-level MMAs (mma.sync m16n8k16, fp16 operands, fp32
// accumulation), for sm_103a.
//
//   Y[m][n] = sum_k A[m][k] * (q[n][k] - zp[n][b]) * s[n][b],   b = k / 64
//
// hip-ep #1318, "What" (Commit 1): the u2 GEMV reads fp32 A and writes fp32 Y
// directly, with the uniform fp16 zero point passed as a scalar; "Performance":
// the phi4-14B export (block 64, zero points 1.5) it is measured on.
//
// Why the matrix unit for a GEMV: at M = 1 a u2 weight byte carries four
// codes, and a SIMT kernel that turns each code into a float needs at least
// one integer operation per code on the half-rate integer pipe -- a ceiling
// near 5 TB/s of weights on this GPU, below the HBM roofline.  Here:
//  * A code masked in place inside a 16-bit half IS an fp16 subnormal:
//    (word & (3 << p)) per half = q * 2^(p - 24), exactly.  One AND of a
//    32-bit word of 16 codes yields an fp16 pair (codes i and i + 8), so a
//    word costs one shift and eight ANDs (0.56 integer operations per code)
//    and the multiply-add runs on the tensor pipe, fed from registers.
//  * The four code positions p in {0, 2, 4, 6} inside a byte are folded into
//    the activations: the MMA's B operand holds a' * 2^-p, so every product
//    is q * a' * 2^-24 whatever p is.  a' = a * 2^(14 - e), e the exponent of
//    the row's largest |a|, so that a' * 2^-p fits fp16.
//  * fp32 activations are split into two fp16 terms (hi = fp16(x), lo =
//    fp16(x - hi)), each its own B column; fp16 / bf16 activations need one.
//  * The scale and zero point are applied per block of 64 codes in fp32,
//    outside the MMA: sum a (q - zp) s = s (sum a q - zp sum a).  To keep a
//    block's sum separate from its neighbours' without reading the
//    accumulator back after every block, the B columns are block-diagonal:
//    column (block, row m, term) holds the activations of that block only, so
//    one accumulator fragment carries up to eight blocks' sums side by side.
//  * Weights stream through an mbarrier ring of shared-memory stages, each
//    filled by one producer warp with one 1-D bulk copy of whole weight rows
//    (one contiguous run of HBM) and one of their block parameters.  Consumer
//    warp w owns the 512-code spans w, w + W, ... of every row; the producer
//    adds the warps' span sums of a tile in span order and writes Y.  Fixed
//    order everywhere: repeated calls are bit-identical (hip-ep #1328, "Why").
//  * Every wait is bounded (qg_device.cuh).
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr int kSpanBytes = 128;    // u2 code bytes of one row in a span: 512 codes, 8 blocks of 64
constexpr int kSpanCodes = 512;
constexpr int kMaxStages = 16;
constexpr int kMaxWarps = 11;      // consumer warps (warp w owns spans w, w + W, ...)
constexpr int kHeader = 512;       // barriers, abort flag, row exponents
constexpr int kPqBytes = 2 * 16 * 16;  // two buffers of 16 rows x 8 fp16 block parameters

struct MgArgs {
    const void *A;
    int a_dtype;
    const uint8_t *W;
    const uint16_t *scales, *zp;
    int row_bytes;    // K / 4
    float zpv;        // scalar zero point (uniform, or the midpoint when absent)
    void *Y;
    int y_dtype;
    int M, N, K, nb;
    int spans;        // K / 512
    int W_;           // consumer warps: warp w owns spans w, w + W_, ...
    int NST, ntiles;  // ring stages (16-row fills), 32-row tiles
    int b_off, sp_off, om_off, zero_off, stage_off, stage_bytes, par_off, zp_off, red_off, pq_off;
    int bov;          // first ring stage that holds the B fragments until every warp has them in registers (NST: none)
    int ast;          // first ring stage that receives the activations (one bulk copy) for the prologue, or -1
    unsigned *fault;
};

// 16-byte global -> shared copy that completes asynchronously (cp.async,
// bypassing L1), and the wait for every such copy this thread issued
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- the column layout, per MNT = (activation rows) x (fp16 terms) columns per block.
// BPG = 8 / MNT blocks share one accumulator fragment (a "D-group"); a span of
// 8 blocks has MNT D-groups of 4 * BPG MMAs.  Thread c of a row quad supplies
// BPG words (16 codes each) per D-group; block_of / word_of give which, and
// beta_of the block's column slot inside the D-group.  The assignments keep
// every code load of a quarter-warp on distinct banks of the swizzled box.
template <int BPG>
__host__ __device__ constexpr int block_of(int j, int c, int w) {
    return BPG == 8 ? 2 * c + (w >> 2) : (BPG == 4 ? 2 * c + j : (BPG == 2 ? ((c >> 1) ? j + 4 : j) : j));
}
template <int BPG>
__host__ __device__ constexpr int word_of(int c, int w) {
    return BPG == 8 ? (w & 3) : (BPG == 4 ? w : (BPG == 2 ? 2 * (c & 1) + w : c));
}
template <int BPG>
__host__ __device__ constexpr int beta_of(int c, int w) {
    return BPG == 8 ? 2 * c + (w >> 2) : (BPG == 4 ? c : (BPG == 2 ? (c >> 1) : 0));
}
// block of column slot beta in D-group j
template <int BPG>
__host__ __device__ constexpr int block_of_beta(int j, int beta) {
    return BPG == 8 ? beta : (BPG == 4 ? 2 * beta + j : (BPG == 2 ? j + 4 * beta : j));
}

// B-fragment entries: 16 bytes (the b0, b1 registers of two MMAs) per
// (span, D-group j, word w, half h, slot); slot = (column within block) * 4 + c.
template <int MNT>
__host__ __device__ constexpr int b_entry(int sp, int j, int w, int h, int slot) {
    return (((sp * MNT + j) * (8 / MNT) + w) * 2 + h) * (4 * MNT) + slot;
}

// (j, c, w) of the thread word that holds code word wd of block blk of a span:
// the inverse of block_of / word_of.
template <int BPG>
__device__ __forceinline__ void owner_of(int blk, int wd, int &j, int &c, int &w) {
    if constexpr (BPG == 8) {
        j = 0; c = blk >> 1; w = ((blk & 1) << 2) | wd;
    } else if constexpr (BPG == 4) {
        j = blk & 1; c = blk >> 1; w = wd;
    } else if constexpr (BPG == 2) {
        j = blk & 3; c = ((blk >> 2) << 1) | (wd >> 1); w = wd & 1;
    } else {
        j = blk; c = wd; w = 0;
    }
}

// One warp prepares span sp: lane L owns code word L (block L / 4, word L % 4,
// codes k = 512 sp + 16 L .. + 15).  Lane L's 16 activations of span sp,
// activation row m: zeros for rows m >= M.
// A is the activation matrix in global memory, or its copy in shared memory.
__device__ __forceinline__ void load_span_act(const MgArgs &p, const void *A, int sp, int m, int lane, float (&a)[16]) {
    const size_t k0 = static_cast<size_t>(sp) * kSpanCodes + 16 * lane;
    if (m >= p.M) {
#pragma unroll
        for (int i = 0; i < 16; ++i) a[i] = 0.f;
    } else if (p.a_dtype == 0) {
        const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(A) + m * static_cast<size_t>(p.K) + k0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v = src[q];
            a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
        }
    } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(A) + m * static_cast<size_t>(p.K) + k0);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint4 v = src[q];
            const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint16_t lo = static_cast<uint16_t>(ww[r] & 0xFFFFu), hi = static_cast<uint16_t>(ww[r] >> 16);
                a[8 * q + 2 * r] = p.a_dtype == 1 ? h2f(lo) : bf2f(lo);
                a[8 * q + 2 * r + 1] = p.a_dtype == 1 ? h2f(hi) : bf2f(hi);
            }
        }
    }
}

// One activation row m of span sp (its activations `a`, loaded by
// load_span_act): the span's largest magnitude |a| gives e and
// a' = a * 2^(14 - e); the lane writes the B entries of its word (fp16
// a' * 2^-p, split into hi / lo terms for fp32 activations); the block's four
// lanes add the sum of a' in a fixed order (2^-24 sum stored in spart); lane 0
// stores the span's output multiplier 2^(10 + e).
template <int MP, int NT>
__device__ __forceinline__ void build_span_row(int sp, int m, int lane, float (&a)[16], unsigned char *bfrag,
                                               float *spart, float *somul) {
    constexpr int MNT = MP * NT;
    constexpr int BPG = 8 / MNT;
    const int blk = lane >> 2, wd = lane & 3;
    int j, c, w;
    owner_of<BPG>(blk, wd, j, c, w);
    // the span's largest magnitude: a lane's 16 in a tree, then one warp-wide
    // integer max (non-negative floats order as their bit patterns)
    float m8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = fmaxf(fabsf(a[i]), fabsf(a[i + 8]));
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m8[i] = fmaxf(m8[i], m8[i + w]);
    // e clamped to [-110, 117]: both 2^(14 - e) and 2^(10 + e) stay normal
    const unsigned bits = __reduce_max_sync(0xffffffffu, __float_as_uint(m8[0]));
    const int ef = static_cast<int>((bits >> 23) & 0xFFu);
    const int e = (bits == 0u || ef == 255) ? 0 : min(max(ef - 127, -110), 117);
    const float asc = exp2i(14 - e);
    float bs = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        a[i] *= asc;
        bs += a[i];
    }
    bs += __shfl_xor_sync(0xffffffffu, bs, 1);
    bs += __shfl_xor_sync(0xffffffffu, bs, 2);
    if (wd == 0) spart[(sp * 8 + blk) * MP + m] = bs * 5.9604644775390625e-08f;  // 2^-24
    if (lane == 0) somul[sp * MP + m] = exp2i(10 + e);
    // (codes i, i + 8) pairs: hi = fp16(x) rounded to nearest, lo = fp16(x - hi),
    // two values per packed conversion
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float pinv = exp2i(-2 * (i & 3));  // 2^-p
        const float x0 = a[i] * pinv, x1 = a[i + 8] * pinv;
        const __half2 h = __floats2half2_rn(x0, x1);
        hi[i] = *reinterpret_cast<const uint32_t *>(&h);
        if (NT == 2) {
            const __half2 l = __floats2half2_rn(x0 - __low2float(h), x1 - __high2float(h));
            lo[i] = *reinterpret_cast<const uint32_t *>(&l);
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int slot = (m * NT + t) * 4 + c;
        const uint32_t *v = t == 0 ? hi : lo;
#pragma unroll
        for (int h = 0; h < 2; ++h)  // entry h: codes (4h, 4h+8), (4h+1, 4h+9), (4h+2, ..), (4h+3, ..)
            *reinterpret_cast<uint4 *>(bfrag + static_cast<size_t>(b_entry<MNT>(sp, j, w, h, slot)) * 16) =
                make_uint4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]);
    }
}

// Lanes of a row quad that hold partial sums of the same (weight row,
// activation row) add them with xor shuffles over the lane bits that keep the
// activation row (a fixed order) before the lowest of them leaves the sum in
// the reduction slot [row][m]: all four lanes for one activation row, else
// the lanes c with c % MP == m for fp32 activations (one row per lane), or
// with (2c, 2c + 1) % MP holding m for 16-bit ones (two rows per lane).
template <int MP, int NT>
__host__ __device__ constexpr int quad_first_offset() {
    return NT == 2 ? MP : (MP == 1 ? 1 : MP / 2);  // the xor offsets are this one, doubled, below 4
}

// At most kMaxWarps + 1 = 12 warps: three per SM sub-partition, whose 16 K
// registers hold three warps of 152 registers (the B fragments a warp may keep
// take 64 of them).
constexpr int kMaxRegs = 152;
static_assert((kMaxWarps + 1 + 3) / 4 * 32 * kMaxRegs <= 16384, "registers of one SM sub-partition");

// TR: MMA row tiles per tile.  TR = 2: 32-row tiles of two 16-row fills, the
// block parameters copied into the stage with the codes.  TR = 1 (long K,
// where the B fragments leave room for 8-row stages only): 16-row tiles of two
// 8-row fills, the block parameters copied by each warp (cp.async).
template <int MP, int NT, bool ZPT, int TR>
__global__ void __maxnreg__(kMaxRegs)
    mma_gemv_kernel(const MgArgs p) {
    constexpr int MNT = MP * NT;
    constexpr int BPG = 8 / MNT;
    constexpr int FR = 8 * TR;       // weight rows per fill
    constexpr int TROWS = 16 * TR;   // weight rows per tile
    constexpr bool PSMEM = TR == 2;  // block parameters in the stage
    static_assert(MNT >= 1 && MNT <= 8 && (8 % MNT) == 0, "columns per block");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 2 * kMaxStages * 8);
    uint64_t *bfree = reinterpret_cast<uint64_t *>(smem + 2 * kMaxStages * 8 + 8);  // every consumer holds its B
    uint64_t *afull = bfree + 1;  // the activations' copy has landed
    uint64_t *afree = bfree + 2;  // every consumer has read them
    unsigned char *bfrag_w = smem + p.b_off;                    // B-fragment entries of every span
    float *spart = reinterpret_cast<float *>(smem + p.sp_off);  // [blocks][MP]: 2^-24 sum of a' per block
    float *somul = reinterpret_cast<float *>(smem + p.om_off);  // [spans][MP]: each span's output multiplier
    unsigned char *stages = smem + p.stage_off;
    float *red = reinterpret_cast<float *>(smem + p.red_off);   // [stage / 2][warp][rows][MP]

    const int W = p.W_;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], W);
        }
        mbar_init(bfree, W * 32);
        mbar_init(afull, 1);
        mbar_init(afree, W * 32);
        *abort_flag = 0;
        mbar_fence_init();
    }
    // the zero slab that lanes without a B column of a word read instead
    for (int i = threadIdx.x; i < 64 * MNT; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem + p.zero_off)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    // A programmatic dependent: the set-up above overlaps the preceding
    // kernel's tail; no buffer of the call is touched before pdl_wait().
    pdl_launch_dependents();
    pdl_wait();

    // A tile is two fills of FR weight rows (TR 16-row MMA row tiles); fill f of
    // this CTA is fill f % 2 of its tile f / 2 -- whole rows: their codes are one
    // contiguous run of HBM, copied by ONE bulk copy, and (TR = 2) their block
    // parameters by one more (a copy instruction costs the TMA engine a fixed
    // time, so few large copies keep HBM busy).  Whole rounds of 2 G fills go
    // out by tile, round-robin (tile b + i G: rows (b + i G) TROWS ..); the
    // fills left over (fewer than 2 G) are dealt one per CTA, then a second
    // per CTA, so no CTA takes more than one fill beyond another.  A CTA's last
    // tile may hold one fill: its second fill's rows lie at or past N.
    const int G = static_cast<int>(gridDim.x), bx = static_cast<int>(blockIdx.x);
    const int nfills = (p.N + FR - 1) / FR;
    const int rounds = nfills / (2 * G);
    const int rem = nfills - 2 * G * rounds;
    const int ntl = rounds + (bx < rem ? 1 : 0);  // tiles of this CTA
    const int total = 2 * ntl;                    // fills of this CTA
    auto fill_row0 = [&](int i, int h) -> int {   // first row of fill h of this CTA's tile i
        return (i < rounds ? (bx + i * G) * 2 + h : 2 * G * rounds + bx + h * G) * FR;
    };
    if (warp == W) {
        // ------------------------------------------------------------ producer
        auto finish = [&](int tl, int rslot) {  // add the warps' sums of tile tl of this CTA, write Y
            const int rb0 = fill_row0(tl, 0), rb1 = fill_row0(tl, 1);
            const float *r = red + (rslot >> 1) * (W * TROWS * MP);
            for (int v = lane; v < TROWS * MP; v += 32) {
                const int row = v / MP, m = v - row * MP;
                const int n = (row < FR ? rb0 : rb1 - FR) + row;
                if (m >= p.M || n >= p.N) continue;
                float s = 0.f;
                for (int w = 0; w < W; ++w) {  // warp (span) order, then lane order
                    s += r[w * TROWS * MP + v];
                }
                store_y_elem(p.Y, p.y_dtype, static_cast<size_t>(m) * p.N + n, s);
            }
        };
        const uint32_t a_bytes = static_cast<uint32_t>(p.M) * p.K * (p.a_dtype == 0 ? 4 : 2);
        if (p.ast >= 0 && lane == 0) {  // the activations, for the consumers' prologue, ahead of the weights
            mbar_arrive_expect_tx(afull, a_bytes);
            bulk_g2s(stages + static_cast<size_t>(p.ast) * p.stage_bytes, p.A, a_bytes, afull);
        }
        bool alive = true;
        int slot = 0;
        uint32_t par = 1;  // parity of the empty phase to wait for before refilling `slot`
        // the weights are read once: evicted from L2 first, they do not push
        // out the code and operands of the launches that follow
        const uint64_t wpol = l2_evict_first();
        for (int f = 0; f < total; ++f) {
            // the first fill into the stages that hold the activations waits
            // until every consumer thread has read them
            if (f == p.ast && !__all_sync(0xffffffffu, mbar_wait(afree, 0, abort_flag, p.fault, FAULT_WAIT_EMPTY))) {
                alive = false;
                break;
            }
            // the first fill into the stages that held the B fragments waits
            // until every consumer thread has its fragments in registers
            if (f == p.bov && p.bov < p.NST &&
                !__all_sync(0xffffffffu, mbar_wait(bfree, 0, abort_flag, p.fault, FAULT_WAIT_EMPTY))) {
                alive = false;
                break;
            }
            if (f >= p.NST) {
                if (!mbar_wait(&empty[slot], par, abort_flag, p.fault, FAULT_WAIT_EMPTY)) {
                    alive = false;
                    break;
                }
                __syncwarp();
                if ((f - p.NST) & 1) finish((f - p.NST) >> 1, slot);
                __syncwarp();
            }
            if (lane == 0) {
                const int row0 = fill_row0(f >> 1, f & 1);
                const int valid = max(0, min(FR, p.N - row0));
                unsigned char *st = stages + static_cast<size_t>(slot) * p.stage_bytes;
                const uint32_t cb = valid * p.row_bytes, pb = PSMEM ? valid * p.nb * 2 : 0;
                mbar_arrive_expect_tx(&full[slot], cb + pb * (ZPT ? 2 : 1));
                if (valid) {
                    bulk_g2s_hint(st, p.W + static_cast<size_t>(row0) * p.row_bytes, cb, &full[slot], wpol);
                    if (PSMEM) {
                        bulk_g2s_hint(st + p.par_off, p.scales + static_cast<size_t>(row0) * p.nb, pb, &full[slot],
                                      wpol);
                        if (ZPT)
                            bulk_g2s_hint(st + p.zp_off, p.zp + static_cast<size_t>(row0) * p.nb, pb, &full[slot], wpol);
                    }
                }
            }
            if (++slot == p.NST) {
                slot = 0;
                par ^= 1u;
            }
        }
        if (alive) {  // the last tiles, once their fills come back
            for (int f = max(0, total - p.NST); f < total; ++f) {
                if (!(f & 1)) continue;
                const int sj = f % p.NST;
                if (!mbar_wait(&empty[sj], (f / p.NST) & 1, abort_flag, p.fault, FAULT_WAIT_EMPTY)) break;
                __syncwarp();
                finish(f >> 1, sj);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers: prologue
    // Each warp prepares its own spans (sl, sl + W, ...) with no CTA-wide
    // synchronisation: lane L holds the 16 activations of code word L of the
    // span (per activation row), normalises the span by its own largest
    // magnitude, writes the B-fragment entries of its word, and the four
    // lanes of a block add its activation sum in a fixed order.
    const int g = lane >> 2, c = lane & 3;
    const int sl = warp;
    // The warp's (span, activation row) items in batches of four: the loads of
    // a batch are all in flight together (one memory latency per batch, which
    // the weight stream started by the producer makes long).
    {
        // the activations' copy in the ring (one bulk copy by the producer), or global memory
        const void *asrc = p.A;
        if (p.ast >= 0) {
            mbar_wait(afull, 0, abort_flag, p.fault, FAULT_WAIT_FULL);
            asrc = stages + static_cast<size_t>(p.ast) * p.stage_bytes;
        }
        const int items = (p.spans - sl + W - 1) / W * MP;
#pragma unroll 1
        for (int b = 0; b < items; b += 4) {
            float a[4][16];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (b + q < items) load_span_act(p, asrc, sl + (b + q) / MP * W, (b + q) % MP, lane, a[q]);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (b + q < items)
                    build_span_row<MP, NT>(sl + (b + q) / MP * W, (b + q) % MP, lane, a[q], bfrag_w, spart, somul);
        }
        if (p.ast >= 0) mbar_arrive(afree);  // this thread's reads of the copy are done
    }
    __syncwarp();

    // ------------------------------------------------------------ consumers: tiles
    // per-thread constants: code offsets inside a span (row g of a fill; row
    // g + 8 is 8 rows further), the B lane slot
    constexpr int NCO = BPG == 8 ? 2 : MNT;
    uint32_t coff[NCO];
#pragma unroll
    for (int j = 0; j < NCO; ++j) {
        const int blk = BPG == 8 ? 2 * c + j : block_of<BPG>(j, c, 0);
        coff[j] = g * p.row_bytes + 16 * blk + (BPG == 2 ? 8 * (c & 1) : (BPG == 1 ? 4 * c : 0));
    }
    const int r8 = 8 * p.row_bytes;
    const int slot_b = (g % MNT) * 4 + c;
    const bool nz0 = (g / MNT) == beta_of<BPG>(c, 0);
    const bool nz1 = (g / MNT) == beta_of<BPG>(c, BPG - 1);  // BPG = 8: the second block of the thread
    const unsigned char *zero_slab = smem + p.zero_off;
    const int m0 = NT == 2 ? c % MP : (2 * c) % MP;
    const int m1 = NT == 2 ? m0 : (2 * c + 1) % MP;
    const int pw = p.nb;  // parameters per row in a stage
    // A warp's B fragments for one span fit in 64 registers (eight 16-byte
    // entries per lane whatever the column layout): a warp that owns a single
    // span loads them once, here, instead of from shared memory for every tile,
    // and the shared memory that held them becomes ring stages.
    constexpr bool BREG = true;
    const bool one_span = p.spans <= W;
    uint4 breg[BREG ? 8 : 1][2];  // [j * BPG + w][h]
    auto load_breg = [&](int sp) {
        const unsigned char *span_b = bfrag_w + static_cast<size_t>(sp) * 1024 * MNT + slot_b * 16;
        const unsigned char *bb0 = nz0 ? span_b : zero_slab;
        const unsigned char *bb1 = nz1 ? span_b : zero_slab;
#pragma unroll
        for (int jw = 0; jw < (BREG ? 8 : 1); ++jw) {
            const int w = jw % BPG;
            const unsigned char *bb = (BPG == 8 && w >= 4) ? bb1 : bb0;
            const int eo = jw * 2 * 64 * MNT;
            breg[jw][0] = *reinterpret_cast<const uint4 *>(bb + eo);
            breg[jw][1] = *reinterpret_cast<const uint4 *>(bb + eo + 64 * MNT);
        }
    };
    if (BREG && one_span) load_breg(sl);
    if (p.bov < p.NST) {  // the B fragments' stages go back to the ring
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // this thread's B stores before the copies
        mbar_arrive(bfree);
    }
    // TR = 1: the block parameters stay in global memory; the warp copies the
    // ones of its next (tile, span) item -- 16 rows x the span's 8 blocks, a
    // 16-byte run per row -- into one of its two buffers while it works on the
    // current item (lanes 0-15 the scales, 16-31 the zero points)
    unsigned char *pq = smem + p.pq_off + sl * kPqBytes * (ZPT ? 2 : 1);
    auto fetch_params = [&](int tl, int spn, int buf) {  // tile tl's rows: FR of each fill
        const int rr = lane & 15;
        if (ZPT || lane < 16) {
            const int n = min(fill_row0(tl, rr / FR) + rr % FR, p.N - 1);  // rows past N: any row
            const uint16_t *src = (lane < 16 ? p.scales : p.zp) + static_cast<size_t>(n) * p.nb + spn * 8;
            cp_async16(pq + (buf * (ZPT ? 2 : 1) + (lane >> 4)) * (kPqBytes / 2) + rr * 16, src);
        }
        cp_async_commit();
    };
    int pqb = 0;
    if (!PSMEM && ntl > 0) fetch_params(0, sl, 0);
    int sa_ = 0, sb_ = 1 % p.NST;
    uint32_t pa = 0, pbp = p.NST == 1 ? 1u : 0u;
    for (int i = 0; i < ntl; ++i) {
        const bool ok = mbar_wait(&full[sa_], pa, abort_flag, p.fault, FAULT_WAIT_FULL) &&
                        mbar_wait(&full[sb_], pbp, abort_flag, p.fault, FAULT_WAIT_FULL);
        // the thread's rows: rr = 0 .. 2 TR - 1 is row g + 8 (rr % TR) of fill rr / TR,
        // i.e. tile row (rr / TR) FR + g + 8 (rr % TR); MMA row tile t takes rr = 2t, 2t + 1
        float acc[2 * TR][2];
#pragma unroll
        for (int r = 0; r < 2 * TR; ++r) acc[r][0] = acc[r][1] = 0.f;
        // a tile whose second fill is empty: TR = 2 skips that fill's MMA row tile;
        // TR = 1 (one MMA row tile over both fills) reads the first fill twice
        const bool two = i < rounds || bx + G < rem;  // (fill_row0(i, 1) < N)
        // the tile body, compiled twice: TWO = false is a TR = 2 tile whose second
        // fill is empty (no loads, MMAs or epilogue for it); one straight-line body
        // each, so no branch splits the unrolled MMA sequence
        auto tile_body = [&](auto two_c) {
            constexpr bool TWO = decltype(two_c)::value;
            const unsigned char *sta = stages + static_cast<size_t>(sa_) * p.stage_bytes;  // the tile's first fill
            const unsigned char *stb = stages + static_cast<size_t>((TR == 1 && !two) ? sa_ : sb_) * p.stage_bytes;
            const uint16_t *psa = reinterpret_cast<const uint16_t *>(sta + p.par_off);
            const uint16_t *psb = reinterpret_cast<const uint16_t *>(stb + p.par_off);
            const uint16_t *zsa = reinterpret_cast<const uint16_t *>(sta + p.zp_off);
            const uint16_t *zsb = reinterpret_cast<const uint16_t *>(stb + p.zp_off);
#pragma unroll 1
            for (int sp = sl; sp < p.spans; sp += W) {
                const unsigned char *ca = sta + sp * kSpanBytes, *cb = stb + sp * kSpanBytes;
                const float *spw = spart + sp * 8 * MP;
                const unsigned char *span_b = bfrag_w + static_cast<size_t>(sp) * 1024 * MNT + slot_b * 16;
                const unsigned char *bb0 = nz0 ? span_b : zero_slab;
                const unsigned char *bb1 = nz1 ? span_b : zero_slab;
                (void)bb0;
                (void)bb1;
                if (BREG && !one_span) load_breg(sp);
                const int pb = sp * 8;  // first block of the span
                (void)pb;
                float accs[2 * TR][2];
#pragma unroll
                for (int r = 0; r < 2 * TR; ++r) accs[r][0] = accs[r][1] = 0.f;
                // TR = 1: this item's parameters have landed (each lane waits for its own
                // copies; the warp barrier shows them to every lane and ends every
                // lane's reads of the other buffer); start the next item's copy
                const uint16_t *pqs = reinterpret_cast<const uint16_t *>(pq + pqb * (ZPT ? 2 : 1) * (kPqBytes / 2));
                (void)pqs;
                if constexpr (!PSMEM) {
                    cp_async_wait_all();
                    __syncwarp();
                    if (sp + W < p.spans)
                        fetch_params(i, sp + W, pqb ^ 1);
                    else if (i + 1 < ntl)
                        fetch_params(i + 1, sl, pqb ^ 1);
                }
#pragma unroll
                for (int j = 0; j < MNT; ++j) {
                    float d[TR][4];  // [row tile][fragment]: the row tiles are independent chains
#pragma unroll
                    for (int t = 0; t < TR; ++t) d[t][0] = d[t][1] = d[t][2] = d[t][3] = 0.f;
                    // this thread's BPG code words of its 2 TR rows (vector loads)
                    uint32_t xw[2 * TR][BPG];
#pragma unroll
                    for (int rr = 0; rr < 2 * TR; ++rr) {
                        if (TR == 2 && rr >= 2 && !TWO) {  // the empty second fill: no loads
#pragma unroll
                            for (int w = 0; w < BPG; ++w) xw[rr][w] = 0u;
                            continue;
                        }
                        const unsigned char *base = (rr / TR ? cb : ca) + (rr % TR) * r8;
                        if constexpr (BPG == 8) {
#pragma unroll
                            for (int hb = 0; hb < 2; ++hb) {
                                const uint4 v = *reinterpret_cast<const uint4 *>(base + coff[hb]);
                                xw[rr][4 * hb] = v.x; xw[rr][4 * hb + 1] = v.y; xw[rr][4 * hb + 2] = v.z; xw[rr][4 * hb + 3] = v.w;
                            }
                        } else if constexpr (BPG == 4) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(base + coff[j]);
                            xw[rr][0] = v.x; xw[rr][1] = v.y; xw[rr][2] = v.z; xw[rr][3] = v.w;
                        } else if constexpr (BPG == 2) {
                            const uint2 v = *reinterpret_cast<const uint2 *>(base + coff[j]);
                            xw[rr][0] = v.x; xw[rr][1] = v.y;
                        } else {
                            xw[rr][0] = *reinterpret_cast<const uint32_t *>(base + coff[j]);
                        }
                    }
#pragma unroll
                    for (int w = 0; w < BPG; ++w) {
                        // B entries of (j, w, h = 0 / 1): a compile-time offset from the span base;
                        // one load serves both row tiles
                        uint4 bq0, bq1;
                        if constexpr (BREG) {
                            bq0 = breg[j * BPG + w][0];
                            bq1 = breg[j * BPG + w][1];
                        } else {
                            const unsigned char *bb = (BPG == 8 && w >= 4) ? bb1 : bb0;
                            const int eo = ((j * BPG + w) * 2) * 64 * MNT;
                            bq0 = *reinterpret_cast<const uint4 *>(bb + eo);
                            bq1 = *reinterpret_cast<const uint4 *>(bb + eo + 64 * MNT);
                        }
#pragma unroll
                        for (int t = 0; t < TR; ++t) {
                            if (TR == 2 && t == 1 && !TWO) continue;
                            const uint32_t x0 = xw[2 * t][w], x1 = xw[2 * t + 1][w];
                            const uint32_t t0 = x0 >> 8, t1 = x1 >> 8;
                            uint32_t u0[8], u1[8];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint32_t mk = 0x00030003u << (2 * q);
                                u0[q] = x0 & mk;
                                u0[4 + q] = t0 & mk;
                                u1[q] = x1 & mk;
                                u1[4 + q] = t1 & mk;
                            }
                            mma16816(d[t], u0[0], u1[0], u0[1], u1[1], bq0.x, bq0.y);
                            mma16816(d[t], u0[2], u1[2], u0[3], u1[3], bq0.z, bq0.w);
                            mma16816(d[t], u0[4], u1[4], u0[5], u1[5], bq1.x, bq1.y);
                            mma16816(d[t], u0[6], u1[6], u0[7], u1[7], bq1.z, bq1.w);
                        }
                    }
                    // columns 2c, 2c+1 -> (beta, m, term); the block's scale (and zero point)
                    // times (sum a' q - zp sum a'), both sums carrying 2^-24
#pragma unroll
                    for (int t = 0; t < TR; ++t) {
                        if (TR == 2 && t == 1 && !TWO) continue;
                        const float D0 = d[t][0], D1 = d[t][1], D2 = d[t][2], D3 = d[t][3];
                        // rows rr = 2t and 2t + 1: fill rr / TR, row g + 8 (rr % TR) of it
                        const uint16_t *ps0 = ((2 * t) / TR ? psb : psa) + (g + 8 * ((2 * t) % TR)) * pw;
                        const uint16_t *ps1 = ((2 * t + 1) / TR ? psb : psa) + (g + 8 * ((2 * t + 1) % TR)) * pw;
                        const uint16_t *zs0 = ((2 * t) / TR ? zsb : zsa) + (g + 8 * ((2 * t) % TR)) * pw;
                        const uint16_t *zs1 = ((2 * t + 1) / TR ? zsb : zsa) + (g + 8 * ((2 * t + 1) % TR)) * pw;
                        (void)ps0;
                        (void)ps1;
                        (void)zs0;
                        (void)zs1;
#pragma unroll
                        for (int e = 0; e < (NT == 2 ? 1 : 2); ++e) {
                            const int bl = block_of_beta<BPG>(j, (2 * c + e) / MNT);
                            const float sa = spw[bl * MP + (e ? m1 : m0)];
                            float s0, s1, z0, z1;
                            if constexpr (PSMEM) {
                                s0 = h2f(ps0[pb + bl]);
                                s1 = h2f(ps1[pb + bl]);
                                z0 = ZPT ? h2f(zs0[pb + bl]) : p.zpv;
                                z1 = ZPT ? h2f(zs1[pb + bl]) : p.zpv;
                            } else {
                                s0 = h2f(pqs[g * 8 + bl]);         // tile row g
                                s1 = h2f(pqs[(g + 8) * 8 + bl]);   // tile row g + 8
                                z0 = ZPT ? h2f(pqs[128 + g * 8 + bl]) : p.zpv;
                                z1 = ZPT ? h2f(pqs[128 + (g + 8) * 8 + bl]) : p.zpv;
                            }
                            // NT = 2: columns 2c, 2c + 1 are the hi / lo terms of one block and row
                            const float P0 = NT == 2 ? D0 + D1 : (e ? D1 : D0);
                            const float P1 = NT == 2 ? D2 + D3 : (e ? D3 : D2);
                            accs[2 * t][e] = fmaf(s0, P0 - z0 * sa, accs[2 * t][e]);
                            accs[2 * t + 1][e] = fmaf(s1, P1 - z1 * sa, accs[2 * t + 1][e]);
                        }
                    }
                }
                // the span's own output multiplier 2^(10 + e)
                const float om0 = somul[sp * MP + m0], om1 = somul[sp * MP + m1];
#pragma unroll
                for (int r = 0; r < 2 * TR; ++r) {
                    acc[r][0] = fmaf(accs[r][0], om0, acc[r][0]);
                    acc[r][1] = fmaf(accs[r][1], om1, acc[r][1]);
                }
                pqb ^= 1;
            }
        };
        if (ok) {
            if (TR == 1 || two) tile_body(std::true_type{});
            else tile_body(std::false_type{});
        }
        // this warp's span sums of the tile's rows, for the producer (in the
        // reduction slot of the tile's second fill): the lanes of a row quad
        // that hold the same (row, activation row) add their partials (xor
        // shuffles, a fixed order) and the first of them stores the sum in
        // [row][m]; the producer adds the warps' sums in warp order
        float *rw = red + (sb_ >> 1) * (W * TROWS * MP) + sl * TROWS * MP;
        constexpr int QO = quad_first_offset<MP, NT>();
#pragma unroll
        for (int r = 0; r < 2 * TR; ++r) {
            const int row = (r / TR) * FR + g + 8 * (r % TR);  // tile row of the thread's row r
            float v0 = NT == 1 && MP == 1 ? acc[r][0] + acc[r][1] : acc[r][0];  // one row: both columns
            float v1 = acc[r][1];
#pragma unroll
            for (int off = QO; off < 4; off <<= 1) {
                v0 += __shfl_xor_sync(0xffffffffu, v0, off);
                if (NT == 1 && MP > 1) v1 += __shfl_xor_sync(0xffffffffu, v1, off);
            }
            if (c < QO) {
                if (NT == 1 && MP == 1) {
                    rw[row] = v0;
                } else if (NT == 2) {  // one activation row per lane
                    rw[row * MP + m0] = v0;
                } else {               // two activation rows per lane
                    rw[row * MP + m0] = v0;
                    rw[row * MP + m1] = v1;
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&empty[sa_]);
            mbar_arrive(&empty[sb_]);
        }
        // the next tile's two fills
        for (int step = 0; step < 2; ++step) {
            if (++sa_ == p.NST) { sa_ = 0; pa ^= 1u; }
            if (++sb_ == p.NST) { sb_ = 0; pbp ^= 1u; }
        }
    }
    if (!PSMEM) cp_async_wait_all();  // no copy outlives the CTA (after a give-up)
}

// ---------------------------------------------------------------- host side
struct MgCfg {
    int MP, NT, TR, spans, W, NST, ntiles, grid;
    int b_off, sp_off, om_off, zero_off, stage_off, stage_bytes, par_off, zp_off, red_off, pq_off, smem;
    int bov, ast;
};

inline int rup(int x, int a) { return (x + a - 1) / a * a; }

// Shared-memory layout and ring depth for tiles of 16 TR rows.  ov: the B
// fragments live in the ring's last stages, which the producer fills only
// once every consumer warp holds its (single) span's fragments in registers.
bool layout_mg(int M, int N, int K, int a_dtype, bool zpt, int tr, bool ov, MgCfg &c) {
    c.TR = tr;
    const DeviceInfo &di = device_info();
    c.NT = a_dtype == 0 ? 2 : 1;
    c.MP = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
    if (c.MP * c.NT > 8) return false;
    c.spans = K / kSpanCodes;
    // consumer warps: the fewest that still give the smallest number of spans per warp
    const int per = (c.spans + kMaxWarps - 1) / kMaxWarps;
    c.W = (c.spans + per - 1) / per;
    const int mnt = c.MP * c.NT;
    const int nblk = c.spans * 8, nb = K / 64, row_bytes = K / 4;
    const int b_bytes = c.spans * 1024 * mnt;
    if (ov && c.spans > c.W) return false;  // only single-span warps keep B in registers
    c.sp_off = kHeader + (ov ? 0 : b_bytes);
    c.om_off = c.sp_off + nblk * c.MP * 4;
    c.zero_off = rup(c.om_off + c.spans * c.MP * 4, 16);
    c.stage_off = rup(c.zero_off + 1024 * mnt, 1024);
    // a stage: FR whole weight rows, their codes then (TR = 2) their block parameters
    const int fr = 8 * c.TR;
    c.par_off = rup(fr * row_bytes, 128);
    c.zp_off = rup(c.par_off + (c.TR == 2 ? fr * nb * 2 : 0), 128);
    c.stage_bytes = rup(c.zp_off + (zpt && c.TR == 2 ? fr * nb * 2 : 0), 128);
    const int red_stage = c.W * 16 * c.TR * c.MP * 4;  // one fp32 sum per (warp, row, activation row)
    // TR = 1: each consumer warp's two buffers of one span's block parameters of a tile
    const int pq_bytes = c.TR == 1 ? c.W * kPqBytes * (zpt ? 2 : 1) : 0;
    const int budget = di.max_smem_optin - 1024 - c.stage_off - pq_bytes;  // 1024: alignment slack
    // an even number of stages: a tile's second fill always lands in an odd
    // stage, whose reduction slot (stage / 2) it owns
    c.NST = std::min(kMaxStages, budget / (c.stage_bytes + red_stage / 2)) & ~1;
    if (c.NST < 4) return false;  // at least two 32-row tiles in flight
    if (ov) {
        const int kb = (b_bytes + c.stage_bytes - 1) / c.stage_bytes;
        if (kb > c.NST) return false;
        c.bov = c.NST - kb;
        c.b_off = c.stage_off + c.bov * c.stage_bytes;
    } else {
        c.bov = c.NST;
        c.b_off = kHeader;
    }
    // Long K (several spans per warp): the activations go through the ring's
    // stages 2, 3, ... (after the first tile's two fills, before the B
    // fragments' stages) as one bulk copy ahead of the weights, when they fit
    // there -- each warp's loads of four spans' activations otherwise queue
    // behind the weight stream (down, K = 17920: 18.0 -> 17.0 us).  With one
    // span per warp the plain loads are as fast.
    {
        const int a_bytes = M * K * (a_dtype == 0 ? 4 : 2);
        const int ka = (a_bytes + c.stage_bytes - 1) / c.stage_bytes;
        c.ast = (c.spans > c.W && 2 + ka <= c.bov) ? 2 : -1;
    }
    c.red_off = c.stage_off + c.NST * c.stage_bytes;
    c.pq_off = c.red_off + (c.NST / 2) * red_stage;
    c.smem = c.pq_off + pq_bytes + 1024;
    c.ntiles = (N + 16 * c.TR - 1) / (16 * c.TR);
    c.grid = std::min(c.ntiles, di.sm_count);
    return true;
}

bool choose_mg1(int M, int N, int K, int a_dtype, bool zpt, int tr, MgCfg &c) {
    return layout_mg(M, N, K, a_dtype, zpt, tr, true, c) || layout_mg(M, N, K, a_dtype, zpt, tr, false, c);
}

// 32-row tiles with the block parameters in the stage, or, when those stages
// do not fit beside the B fragments (long K, or eight B columns per block),
// 16-row tiles of 8-row fills.
bool choose_mg(int M, int N, int K, int a_dtype, bool zpt, MgCfg &c) {
    if (choose_mg1(M, N, K, a_dtype, zpt, 2, c)) return true;
    return choose_mg1(M, N, K, a_dtype, zpt, 1, c);
}

template <int MP, int NT, bool ZPT, int TR>
cudaError_t launch_mg(const MgArgs &a, const MgCfg &c, cudaStream_t s) {
    auto kern = mma_gemv_kernel<MP, NT, ZPT, TR>;
    static std::atomic<unsigned> configured{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned bit = 1u << (dev & 31);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, device_info().max_smem_optin);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const cudaError_t e = launch_pdl(kern, dim3(c.grid), dim3((c.W + 1) * 32), c.smem, s, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// Activation rows per launch: four with fp32 activations (hi / lo terms: eight
// B columns per block), eight with 16-bit ones.  fp32 requests with more rows
// run as one launch per group of four rows (each streams the weights once);
// 16-bit requests with more rows belong to the tcgen05 path.
int mma_rows(int a_dtype) { return a_dtype == 0 ? 4 : 8; }

// Activation rows per launch: mma_rows, or, where the B fragments of that
// many rows leave no room for the ring (long K), two launches of half as many
// rows -- 16-bit activations with 3 or 4 rows, fp32 ones with 2 -- which read
// the weights twice and still beat the SIMT kernel there.
static int launch_rows(const GemmProblem &p) {
    const bool zpt = p.zp_mode == ZP_TENSOR;
    const int half = p.a_dtype == 0 ? 1 : 2;
    MgCfg c;
    if (p.M > half && p.M <= 2 * half && !choose_mg(p.M, p.N, p.K, p.a_dtype, zpt, c) &&
        choose_mg(half, p.N, p.K, p.a_dtype, zpt, c))
        return half;
    return mma_rows(p.a_dtype);
}

bool mma_gemv_eligible(const GemmProblem &p) {
    if (p.kind != WK_NBITS || p.bits != 2 || p.bs != 64 || p.K % kSpanCodes != 0 || p.zp_mode == ZP_PACKED)
        return false;
    if (p.M < 1 || (p.M > mma_rows(p.a_dtype) && p.a_dtype != 0)) return false;
    const int g = launch_rows(p);
    MgCfg c;
    const bool zpt = p.zp_mode == ZP_TENSOR;
    if (!choose_mg(std::min(p.M, g), p.N, p.K, p.a_dtype, zpt, c)) return false;
    if (p.M > g && p.M % g != 0 && !choose_mg(p.M % g, p.N, p.K, p.a_dtype, zpt, c)) return false;
    // 16-row tiles copy each row's eight block parameters of a span as one
    // 16-byte run: the parameter tensors must start on a 16-byte boundary
    const auto a16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    return c.TR == 2 || (a16(p.scales) && (!zpt || a16(p.zp)));
}

bool mma_gemv_plan(int M, int N, int K, int a_dtype, int zp_mode, int out[4]) {
    if (K % kSpanCodes != 0 || M < 1 || (M > mma_rows(a_dtype) && a_dtype != 0)) return false;
    GemmProblem p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.a_dtype = a_dtype;
    p.zp_mode = zp_mode == 1 ? ZP_TENSOR : (zp_mode == 2 ? ZP_UNIFORM : ZP_NONE);
    const int g = launch_rows(p);
    MgCfg c;
    if (!choose_mg(std::min(M, g), N, K, a_dtype, zp_mode == ZP_TENSOR, c)) return false;
    out[0] = 16 * c.TR;
    out[1] = c.W;
    out[2] = c.grid;
    out[3] = c.NST;
    return true;
}

namespace {

cudaError_t mma_gemv_rows(const GemmProblem &p, cudaStream_t s) {
    MgCfg c;
    const bool zpt = p.zp_mode == ZP_TENSOR;
    if (!choose_mg(p.M, p.N, p.K, p.a_dtype, zpt, c)) return cudaErrorNotSupported;
    const int nb = p.K / p.bs;
    MgArgs a{};
    a.A = p.A;
    a.a_dtype = p.a_dtype;
    a.W = p.W;
    a.scales = p.scales;
    a.zp = p.zp;
    a.row_bytes = p.K / 4;
    a.zpv = p.uniform_zp;
    a.Y = p.Y;
    a.y_dtype = p.y_dtype;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.nb = nb;
    a.spans = c.spans;
    a.W_ = c.W;
    a.NST = c.NST;
    a.ntiles = c.ntiles;
    a.b_off = c.b_off;
    a.sp_off = c.sp_off;
    a.om_off = c.om_off;
    a.zero_off = c.zero_off;
    a.stage_off = c.stage_off;
    a.stage_bytes = c.stage_bytes;
    a.par_off = c.par_off;
    a.zp_off = c.zp_off;
    a.red_off = c.red_off;
    a.pq_off = c.pq_off;
    a.bov = c.bov;
    a.ast = c.ast;
    a.fault = fault_word();
#define QG_MG(MP_, NT_, TR_)                                                                        \
    if (c.MP == MP_ && c.NT == NT_ && c.TR == TR_)                                                  \
        return zpt ? launch_mg<MP_, NT_, true, TR_>(a, c, s) : launch_mg<MP_, NT_, false, TR_>(a, c, s);
    QG_MG(1, 2, 2)
    QG_MG(2, 2, 2)
    QG_MG(4, 2, 2)
    QG_MG(1, 1, 2)
    QG_MG(2, 1, 2)
    QG_MG(4, 1, 2)
    QG_MG(8, 1, 2)
    QG_MG(1, 2, 1)
    QG_MG(2, 2, 1)
    QG_MG(4, 2, 1)
    QG_MG(1, 1, 1)
    QG_MG(2, 1, 1)
    QG_MG(4, 1, 1)
    QG_MG(8, 1, 1)
#undef QG_MG
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t mma_gemv(const GemmProblem &p, cudaStream_t s) {
    const int g = launch_rows(p);
    if (p.M <= g) return mma_gemv_rows(p, s);
    const size_t asz = p.a_dtype == 0 ? 4 : 2, ysz = p.y_dtype == 0 ? 4 : 2;
    for (int m0 = 0; m0 < p.M; m0 += g) {
        GemmProblem q = p;
        q.A = static_cast<const char *>(p.A) + static_cast<size_t>(m0) * p.K * asz;
        q.Y = static_cast<char *>(p.Y) + static_cast<size_t>(m0) * p.N * ysz;
        q.M = std::min(g, p.M - m0);
        const cudaError_t e = mma_gemv_rows(q, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace qg
