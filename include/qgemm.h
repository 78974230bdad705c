/*
 * qgemm.h -- C ABI of the GB300 (sm_103a) blockwise low-bit dequantize +
 * GEMV / small-M GEMM library, and of the fused single-token QMoE decode.
 *
 *     Y[M, N] = A[M, K] . dequant(W)[N, K]^T
 *
 * Sources (web pages, cited by title and section):
 *   [hip-ep #1318]  hip-ep pull request #1318: 2-bit MatMulNBits kernels for
 *                   phi4-14B on gfx1151.
 *   [hip-ep #1328]  hip-ep pull request #1328: fused QMoE decode that picks
 *                   its tiling before computing.
 *   [bnb #1979]     bitsandbytes pull request #1979: "[ROCm] Fused 4-bit SIMT
 *                   GEMM" (NF4/FP4 codebook weights).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The library
 *    never allocates, frees or synchronises (except qg_fp16_uniform_value and
 *    qg_read_device_fault, which return a value to the host), and enqueues
 *    work on `stream` only, on the current device (`stream` must belong to
 *    it).  It keeps no per-call state between calls, so concurrent calls on
 *    different streams with disjoint outputs and workspaces are independent.
 *    One exception is device-wide: the fault word of qg_read_device_fault
 *    (below), which every call's kernels may set and which any caller's read
 *    clears.
 *  - Weight codes are packed along K, least significant bits first: element
 *    k of row n is bits [(k*bits)%8, (k*bits)%8 + bits) of byte
 *    n*(K*bits/8) + (k*bits)/8.  W is row-major [N][K*bits/8] bytes.
 *  - Per-block parameters (fp16 scales, fp16 zero points, fp32 absmax) are
 *    row-major [N][K/block_size].  fp16/bf16 tensors are passed as their
 *    16-bit patterns (uint16_t).
 *  - A is row-major and contiguous, [M][K] (the raw-pointer contract of
 *    [bnb #1979], "Technical details", raw-pointer safety).  Y is row-major
 *    [M][N] and is fully overwritten.
 *  - Alignment: A, W, scales, zero points, absmax and the workspace must be
 *    16-byte aligned; otherwise the call returns QG_ERR_INVALID_ARG.
 *  - Block sizes 32, 64, 128 and 256 are supported, with K % block_size == 0.
 *    Other block sizes (16 in particular, which [hip-ep #1328] "Notes for
 *    reviewers" reports computing every output wrongly) are refused with
 *    QG_ERR_UNSUPPORTED, never computed.
 *  - Arguments are checked on the host before anything is enqueued; a refused
 *    call launches nothing ([hip-ep #1328], "Test plan": arguments the
 *    launchers must refuse).
 *  - On entry the calling thread's pending, non-sticky CUDA error is cleared,
 *    so an earlier unrelated failure is not reported as this call's failure;
 *    after each launch the launch status is checked and returned as
 *    QG_ERR_CUDA ([hip-ep #1328], "What": clear the error state before the
 *    fused decode launches).
 *  - Results are deterministic: every reduction runs in a fixed order that
 *    depends only on the shape, never on timing, so repeated calls on the
 *    same inputs are bit-identical ([hip-ep #1328], "Why" and "Test plan":
 *    129 calls bit-identical).  Nothing is tuned or timed on live calls.
 *  - M == 0 or N == 0 is a no-op.  K == 0 writes zeros.
 *  - Kernels are launched as programmatic dependents of the preceding kernel
 *    on `stream`: their set-up (barriers, tensor memory) overlaps that
 *    kernel's tail, but no buffer of the call -- weights, block parameters,
 *    activations, expert ids, outputs -- is read or written before that kernel
 *    has completed, so stream order holds exactly as for plain launches.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *qg_stream_t;

/* Status codes returned by every entry point. */
enum {
    QG_OK = 0,
    QG_ERR_INVALID_ARG = 1,          /* null/misaligned pointer, bad size, K % block_size != 0 */
    QG_ERR_UNSUPPORTED = 2,          /* valid request this library does not implement (bits, block size, dtype combination) */
    QG_ERR_CUDA = 3,                 /* a CUDA launch or copy failed; the CUDA error stays readable via cudaGetLastError */
    QG_ERR_WORKSPACE_TOO_SMALL = 4   /* workspace_bytes below what *_workspace_bytes() returned for this shape */
};

/* Element types of A and Y. */
enum { QG_F32 = 0, QG_F16 = 1, QG_BF16 = 2 };

/*
 * qgemm_nbits -- MatMulNBits: per-block fp16 scale and fp16 zero point.
 *   [hip-ep #1318] "What", Commit 1 (u2 GEMV and WMMA kernels templated on
 *   the A/C element types, reading fp32 A and writing fp32 C directly) and
 *   "Performance", Model (block 64, fp16 scales and zero points).
 *
 *   w[n][k] = (q[n][k] - zp[n][k/bs]) * s[n][k/bs], computed exactly in fp32;
 *   Y[m][n] = sum_k A[m][k] * w[n][k], accumulated in fp32 (tensor-core path:
 *   the weight is rounded to A's 16-bit type before the product; fp32
 *   activations on the tensor cores -- M >= 16, fp32 Y -- go in split
 *   precision: A and w each as two fp16 terms, three products) and rounded
 *   once to y_dtype.
 *
 *   A            [M][K], a_dtype (QG_F32, QG_F16 or QG_BF16)
 *   W            [N][K*bits/8] packed codes, bits = 2, 3, 4 or 8 (the u2 / u3 / u4 /
 *                "Wi8" MatMulNBits leaves of the hip-ep #1318 kernel test table;
 *                3-bit codes run on the SIMT path for every M, a code may continue
 *                into the next byte; 8-bit: one code per byte, midpoint 128 by
 *                default); other widths are refused with QG_ERR_UNSUPPORTED
 *   scales_f16   [N][K/block_size] fp16 patterns
 *   zero_points_f16  [N][K/block_size] fp16 patterns, or NULL for the
 *                midpoint 2^(bits-1)
 *   Y            [M][N], y_dtype
 *   workspace    device scratch of at least
 *                qgemm_workspace_bytes(a_dtype, M, N, K, bits, block_size)
 *                bytes (NULL allowed when that is 0); its contents on entry
 *                do not matter and are garbage on return.  For fp32
 *                activations with M >= 16 that size includes room for the
 *                split-precision activations (4 M K bytes); a smaller
 *                workspace that still covers the call's other needs is
 *                accepted and takes a slower path (fp32 row groups).
 *   Returns a QG_* status.
 */
int qgemm_nbits(const void *A, int a_dtype, const uint8_t *W, const uint16_t *scales_f16,
                const uint16_t *zero_points_f16, void *Y, int y_dtype, int M, int N, int K, int bits,
                int block_size, void *workspace, size_t workspace_bytes, qg_stream_t stream);

/*
 * qgemm_nbits_uniform_zp -- as qgemm_nbits, with every zero point equal to
 * the scalar `uniform_zp` ([hip-ep #1318] "What", Commit 1:
 * hip_matmul_nbits_ex(..., float uniform_zp); "Why": fp16 zero points that
 * are all 1.5 cost as many bytes per token as the scales).  The zero-point
 * tensor is never read.  Bit-identical to qgemm_nbits with a full zero-point
 * tensor holding the fp16 value uniform_zp.
 */
int qgemm_nbits_uniform_zp(const void *A, int a_dtype, const uint8_t *W, const uint16_t *scales_f16,
                           float uniform_zp, void *Y, int y_dtype, int M, int N, int K, int bits,
                           int block_size, void *workspace, size_t workspace_bytes, qg_stream_t stream);

/*
 * qgemm_codebook4 -- NF4/FP4-style weights: a 4-bit code selects one of 16
 * fp32 codebook entries, multiplied by the block's fp32 absmax.
 *   [bnb #1979] "Summary" (NF4/FP4 weights decoded inside the GEMM, decoded
 *   values reused across the M rows) and "Technical details" (centroid
 *   lookup).
 *
 *   w[n][k] = codebook16[q[n][k]] * absmax[n][k/bs]   (fp32)
 *   codebook16  16 fp32 entries (device)
 *   absmax      [N][K/block_size] fp32
 *   Other arguments as qgemm_nbits (bits is 4).
 */
int qgemm_codebook4(const void *A, int a_dtype, const uint8_t *W, const float *codebook16, const float *absmax,
                    void *Y, int y_dtype, int M, int N, int K, int block_size, void *workspace,
                    size_t workspace_bytes, qg_stream_t stream);

/* Workspace bytes the two GEMM entry points need for this shape (same value
 * for qgemm_nbits, qgemm_nbits_uniform_zp and, with bits = 4,
 * qgemm_codebook4).  0 means no workspace is needed. */
size_t qgemm_workspace_bytes(int a_dtype, int M, int N, int K, int bits, int block_size);

/*
 * qmoe_decode_fused -- one token through the top-k experts of a quantized
 * MoE layer: fc1 GEMV, SwiGLU, fc2 GEMV, weighted sum over the k slots.
 *   [hip-ep #1328] "Summary" and "What" (hip_qmoe_decode_fused with
 *   num_experts; u4 weights; block 32/64/128; zero points and bias
 *   optional, "Test plan"); [hip-ep #1318] "Why" (the SwiGLU chain gate ->
 *   sigmoid -> multiplies -> up).
 *
 *   For slot j = 0..k-1 in order, e = expert_ids[j]:
 *     g = dequant(fc1[e]) . x + fc1_bias[e]                 (2*inter values)
 *     gate, up = g[0:inter], g[inter:2*inter]  (swiglu_interleaved = 0)
 *              = g[0::2],    g[1::2]           (swiglu_interleaved = 1)
 *     h = silu(gate) * up                                    (kept in fp32)
 *     o = dequant(fc2[e]) . h + fc2_bias[e]                  (hidden values)
 *   y = round_to_fp16( sum_j expert_weights[j] * o_j ), summed in slot order.
 *
 *   x_f16        [hidden] fp16
 *   expert_ids   [k] int32 (device); an id outside [0, num_experts) adds
 *                nothing and sets *status_dev to 1 (status_dev may be NULL)
 *   expert_weights [k] fp32 (device)
 *   fc1_w        [num_experts][2*inter][hidden*bits/8]
 *   fc1_scales   [num_experts][2*inter][hidden/block_size] fp16
 *   fc1_zp       same shape as fc1_scales, or NULL (midpoint 2^(bits-1))
 *   fc1_bias     [num_experts][2*inter] fp16, or NULL
 *   fc2_w        [num_experts][hidden][inter*bits/8]
 *   fc2_scales   [num_experts][hidden][inter/block_size] fp16
 *   fc2_zp       same shape as fc2_scales, or NULL
 *   fc2_bias     [num_experts][hidden] fp16, or NULL
 *   bits         4 (2 is accepted too)
 *   block_size   32, 64, 128 or 256; hidden and inter multiples of it
 *   y_f16        [hidden] fp16 output
 *   status_dev   device int written with 0 (all ids valid) or 1, or NULL
 *   workspace    at least qmoe_decode_workspace_bytes(k, hidden, inter) bytes
 *                of device memory, 16-byte aligned (QG_ERR_INVALID_ARG
 *                otherwise): the fc1 output g [k][2*inter] fp32 first, then,
 *                at the next multiple of 256 bytes, the slot outputs o
 *                [k][hidden] fp32.  Needs no initial contents; the call
 *                overwrites it.
 */
int qmoe_decode_fused(const uint16_t *x_f16, const int32_t *expert_ids, const float *expert_weights, int k,
                      int num_experts, const uint8_t *fc1_w, const uint16_t *fc1_scales, const uint16_t *fc1_zp,
                      const uint16_t *fc1_bias, const uint8_t *fc2_w, const uint16_t *fc2_scales,
                      const uint16_t *fc2_zp, const uint16_t *fc2_bias, int hidden, int inter, int bits,
                      int block_size, int swiglu_interleaved, uint16_t *y_f16, int *status_dev, void *workspace,
                      size_t workspace_bytes, qg_stream_t stream);

size_t qmoe_decode_workspace_bytes(int k, int hidden, int inter);

/*
 * qmoe_decode_fused_dp4a -- the same decode with int8 activations.
 * [hip-ep #1328] "Summary" (a dp4a form of the fused decode exists beside the fp one), "Test
 * plan" (fp and dp4a x block size x zero points x bias).  The pages do not
 * give the activation quantization; this library's reading: each activation
 * vector (x before fc1, h = silu(gate) * up before fc2) is quantized per block
 * of block_size values along the contraction,
 *     a = max |v|,  sx = fl32(a / 127),  q8 = clamp(rint(fl32(v / sx)), -127, 127)
 * (ties to even; an all-zero block gives sx = 0, q8 = 0), and each output is
 *     sum_b s[r][b] * sx[b] * ( sum_{k in b} q8[k] * q[r][k] - zp[r][b] * sum_{k in b} q8[k] )
 * with exact integer sums, plus the bias.  Results therefore differ from
 * qmoe_decode_fused by the activation quantization error (about 1/254 of each
 * block's largest magnitude per element).
 *
 * Arguments, layouts, statuses and the workspace size are those of
 * qmoe_decode_fused; in addition hidden and inter must be at most 65536
 * (QG_ERR_UNSUPPORTED otherwise).  Deterministic: repeated calls are
 * bit-identical.
 */
int qmoe_decode_fused_dp4a(const uint16_t *x_f16, const int32_t *expert_ids, const float *expert_weights, int k,
                           int num_experts, const uint8_t *fc1_w, const uint16_t *fc1_scales, const uint16_t *fc1_zp,
                           const uint16_t *fc1_bias, const uint8_t *fc2_w, const uint16_t *fc2_scales,
                           const uint16_t *fc2_zp, const uint16_t *fc2_bias, int hidden, int inter, int bits,
                           int block_size, int swiglu_interleaved, uint16_t *y_f16, int *status_dev, void *workspace,
                           size_t workspace_bytes, qg_stream_t stream);

/*
 * qmoe_decode_fused_noalloc -- qmoe_decode_fused for callers that cannot
 * allocate device memory (a decode loop inside a runtime that forbids
 * allocation on its hot path, an embedded host that must not allocate after
 * start-up, a C caller without an allocator).  The source pages have no
 * counterpart: this is an addition of this library.
 *
 * Same arguments and results as qmoe_decode_fused, minus the workspace: the
 * scratch is a fixed device array of QG_QMOE_NOALLOC_SCRATCH_BYTES inside the
 * library, held by every GPU that loads it until the process exits.  Shapes
 * needing more, i.e. qmoe_decode_workspace_bytes(k, hidden, inter) >
 * QG_QMOE_NOALLOC_SCRATCH_BYTES, are refused with QG_ERR_UNSUPPORTED before
 * anything is enqueued.  Calls no cudaMalloc, cudaFree or other allocator.
 *  - The first call on a device looks up the array's device address (once
 *    per device, with that device current); make that first call before any
 *    stream capture.  Like every entry point it works on the current device:
 *    `stream` must belong to it.
 *  - All calls on a device share the one array: calls that can overlap on
 *    the GPU (unordered streams) race.  The array keeps the last call's
 *    contents; no call depends on them.
 */
#define QG_QMOE_NOALLOC_SCRATCH_BYTES (1u << 20)
int qmoe_decode_fused_noalloc(const uint16_t *x_f16, const int32_t *expert_ids, const float *expert_weights, int k,
                              int num_experts, const uint8_t *fc1_w, const uint16_t *fc1_scales,
                              const uint16_t *fc1_zp, const uint16_t *fc1_bias, const uint8_t *fc2_w,
                              const uint16_t *fc2_scales, const uint16_t *fc2_zp, const uint16_t *fc2_bias,
                              int hidden, int inter, int bits, int block_size, int swiglu_interleaved,
                              uint16_t *y_f16, int *status_dev, qg_stream_t stream);

/*
 * qg_fp16_uniform_value -- detect an fp16 tensor whose elements all have the
 * same bit pattern ([hip-ep #1318] "What", Commit 1: the runtime detects an
 * all-equal fp16 zero-point tensor once per buffer and then passes it as a
 * scalar).  +0 and -0 differ; a NaN pattern is reported as not uniform; an
 * empty tensor is not uniform.  Enqueues one kernel on `stream`, then
 * synchronises the stream and writes *is_uniform (0/1) and, when uniform,
 * *value (host pointers).  workspace: at least 16 bytes of device memory.
 */
int qg_fp16_uniform_value(const uint16_t *t, size_t n, int *is_uniform, float *value, void *workspace,
                          size_t workspace_bytes, qg_stream_t stream);

/*
 * Dequantize to fp32 [N][K] (device), bit-exact with the definitions above.
 * Used to check unpacking and dequantization in isolation, and as the
 * "dequantize then dense GEMM" building block.
 *   qg_dequant_nbits: zero_points_f16 may be NULL (midpoint).
 */
int qg_dequant_nbits(const uint8_t *W, const uint16_t *scales_f16, const uint16_t *zero_points_f16, float *out,
                     int N, int K, int bits, int block_size, qg_stream_t stream);
int qg_dequant_nbits_uniform_zp(const uint8_t *W, const uint16_t *scales_f16, float uniform_zp, float *out, int N,
                                int K, int bits, int block_size, qg_stream_t stream);
int qg_dequant_codebook4(const uint8_t *W, const float *codebook16, const float *absmax, float *out, int N, int K,
                         int block_size, qg_stream_t stream);

/*
 * qgemm_codebook4_nested -- qgemm_codebook4 with a nested ("double-quantized")
 * absmax.  [bnb #1979] "Testing plan": nested / non-nested absmax; the pages
 * do not give the format, this library's reading:
 *   absmax[i] = fl32( fl32(absmax_table256[absmax_q[i]] * absmax2[i / nested_block]) + absmax_offset )
 * over the flat row-major index i = n * (K/block_size) + b; then exactly as
 * qgemm_codebook4 with that absmax.
 *
 *   absmax_q         [N][K/block_size] uint8 codes (device)
 *   absmax_table256  [256] fp32 (device, 4-byte aligned)
 *   absmax2          [ceil(N*(K/block_size) / nested_block)] fp32 (device, 4-byte aligned)
 *   absmax_offset    fp32 scalar (not NaN); nested_block >= 1 (bitsandbytes uses 256)
 *   Other arguments as qgemm_codebook4.  The expanded absmax is written to the
 *   front of the workspace (at least qgemm_codebook4_nested_workspace_bytes()).
 */
int qgemm_codebook4_nested(const void *A, int a_dtype, const uint8_t *W, const float *codebook16,
                           const uint8_t *absmax_q, const float *absmax_table256, const float *absmax2,
                           float absmax_offset, int nested_block, void *Y, int y_dtype, int M, int N, int K,
                           int block_size, void *workspace, size_t workspace_bytes, qg_stream_t stream);
size_t qgemm_codebook4_nested_workspace_bytes(int a_dtype, int M, int N, int K, int block_size);

/*
 * qgemm_nbits_packed_zp -- qgemm_nbits with unsigned integer zero points
 * packed like the codes.  [hip-ep #1318] "Notes for reviewers", kernel test
 * table (the 2-, 3-, 4- and 8-bit MatMulNBits leaves); the pages' own zero
 * points are fp16 ("What", Commit 1) and they describe no packed form, so the
 * layout is this library's reading: zero point b of row n is the unsigned
 * `bits`-wide field starting at bit b*bits of row n's bit string, least
 * significant bit first (a field may continue into the next byte), each row
 * occupying ceil((K/block_size)*bits/8) bytes.
 *
 *   zero_points_packed  [N][ceil((K/block_size)*bits/8)] uint8 (device, any
 *                alignment; NULL: QG_ERR_INVALID_ARG)
 *   Other arguments as qgemm_nbits; the workspace holds at least
 *   qgemm_nbits_packed_zp_workspace_bytes() bytes, 16-byte aligned.  A request
 *   that qgemm_nbits would serve with its SIMT GEMV kernel stages the packed
 *   bytes beside the codes and widens each field where it is used; any other
 *   (2-bit block-64 tensor-pipe GEMV, tensor cores) first widens the zero
 *   points to fp16 [N][K/block_size] at the front of the workspace with one
 *   small kernel.  Either way the result is bit-identical to qgemm_nbits
 *   given the same integers as fp16 zero points.  Every check of qgemm_nbits
 *   happens before anything is enqueued.
 */
int qgemm_nbits_packed_zp(const void *A, int a_dtype, const uint8_t *W, const uint16_t *scales_f16,
                          const uint8_t *zero_points_packed, void *Y, int y_dtype, int M, int N, int K, int bits,
                          int block_size, void *workspace, size_t workspace_bytes, qg_stream_t stream);
size_t qgemm_nbits_packed_zp_workspace_bytes(int a_dtype, int M, int N, int K, int bits, int block_size);

/*
 * qmoe_ragged_mm -- ragged expert GEMM: the rows of X are grouped by expert
 * and each group is multiplied by its expert's MatMulNBits weight.
 * [hip-ep #1318] kernel test table, qmoe_ragged_mm leaf Xfp16_Wu4_Yfp16; the
 * pages name the op and its types, the layout is this library's reading.
 *
 *   for e in 0 .. num_experts-1, r in [offs[e], offs[e+1]):
 *       Y[r][n] = sum_k X[r][k] * w_e[n][k],  w_e = (q - zp) * s as qgemm_nbits
 *
 *   X                [T][K] of x_dtype (QG_F32 / F16 / BF16), T = offs[num_experts]
 *   expert_offsets   [num_experts + 1] int64, HOST memory: offs[0] = 0, never
 *                    decreasing (an expert may own no row); read before return
 *   W                [num_experts][N][K*bits/8] codes, bits 2, 4 or 8
 *   scales_f16       [num_experts][N][K/block_size] fp16
 *   zero_points_f16  same shape, fp16, or NULL (midpoint 2^(bits-1))
 *   Y                [T][N] of y_dtype
 * X, W, scales and zero points 16-byte aligned; one expert's slice of W and of
 * the scales must be a multiple of 16 bytes (QG_ERR_UNSUPPORTED otherwise).
 * With 16-bit activations the experts with 9 or more rows run in one grouped
 * tensor-core launch (at most 256 experts); the others, and fp32 activations,
 * run as one GEMM per expert on its rows.  Workspace: at least
 * qmoe_ragged_mm_workspace_bytes(...) for the same offsets (0 when every expert
 * takes the grouped launch).
 */
int qmoe_ragged_mm(const void *X, int x_dtype, const int64_t *expert_offsets, int num_experts, const uint8_t *W,
                   const uint16_t *scales_f16, const uint16_t *zero_points_f16, void *Y, int y_dtype, int N, int K,
                   int bits, int block_size, void *workspace, size_t workspace_bytes, qg_stream_t stream);
size_t qmoe_ragged_mm_workspace_bytes(int x_dtype, const int64_t *expert_offsets, int num_experts, int N, int K,
                                      int bits, int block_size);

/*
 * qmoe_ragged_mm_device_offsets -- the ragged expert GEMM above with the
 * expert offsets in DEVICE memory, so that a router on the GPU needs no host
 * round trip: the computation and the reading of the pages are those of
 * qmoe_ragged_mm ([hip-ep #1318] kernel test table, qmoe_ragged_mm leaf;
 * [hip-ep #1328] "Summary": the QMoE op family).
 *
 *   expert_offsets_dev  [num_experts + 1] int64, device, 8-byte aligned,
 *                       read on the device after the preceding work on the
 *                       stream: offs[0] = 0, never decreasing, offs[E] <=
 *                       max_rows.  Offsets breaking that rule make the call
 *                       compute nothing and set *status_dev to 1 (status_dev
 *                       may be NULL; it is never cleared).
 *   max_rows            rows X and Y hold (host int, >= the real T); rows of
 *                       Y at or past offs[E] are left untouched
 *   X                   [max_rows][K] fp16 or bf16 (fp32: QG_ERR_UNSUPPORTED)
 *   W, scales, zero points, Y, N, K, bits, block_size as qmoe_ragged_mm
 *   num_experts         1 .. 256
 *   workspace           not used (may be NULL);
 *                       qmoe_ragged_mm_device_offsets_workspace_bytes(E)
 *                       returns 0
 * Every expert with rows runs in one grouped tensor-core launch (sized for the
 * most tiles offsets within max_rows can need; each CTA numbers the experts'
 * tiles from the offsets itself, and tiles past the real count end at once).
 * Returns QG_OK, QG_ERR_* for refused arguments (before any launch) or
 * QG_ERR_CUDA.
 */
int qmoe_ragged_mm_device_offsets(const void *X, int x_dtype, const int64_t *expert_offsets_dev, int num_experts,
                                  int max_rows, const uint8_t *W, const uint16_t *scales_f16,
                                  const uint16_t *zero_points_f16, void *Y, int y_dtype, int N, int K, int bits,
                                  int block_size, void *workspace, size_t workspace_bytes, int *status_dev,
                                  qg_stream_t stream);
size_t qmoe_ragged_mm_device_offsets_workspace_bytes(int num_experts);

/*
 * qg_gather_block_quantized -- embedding lookup in a block-quantized table.
 * [hip-ep #1318] kernel test table, gather_block_quantized leaves
 * Xi64_Wu4_Yfp16, Xi64_Wu8_Yfp16 and Xi64_Wfp8_Yfp16 ("Summary", Commit 3:
 * embedding lookups through a gather).  The pages name the op and its types;
 * the layout and rule below are this library's reading of them.
 *
 *   Y[i][d] = round_to(y_dtype, w(row_i, d)),  row_i = indices[i], or
 *             indices[i] + vocab when indices[i] < 0
 *   integer formats: w = fl32( fl32(q - zp) * s )  (as qgemm_nbits; zp the
 *                    midpoint 2^(bits-1) when zero_points_f16 is NULL)
 *   QG_WF_E4M3:      w = fl32( e4m3(q) * s )  (OCP E4M3 without infinities;
 *                    no zero point)
 *   with s = scales_f16[row_i][d / block_size], and rounding to nearest-even.
 *
 *   indices      [n_indices] int64 (device, 8-byte aligned).  An index outside
 *                [-vocab, vocab) gives a zero row and sets *status_dev to 1.
 *   W            [vocab][D*bits/8] codes packed LSB-first along D (bits 2, 4
 *                or 8 for QG_WF_U2 / U4 / U8), or [vocab][D] E4M3 bytes
 *   scales_f16   [vocab][D/block_size] fp16
 *   zero_points_f16  same shape, fp16, or NULL; must be NULL for E4M3
 *   block_size   32, 64, 128 or 256; D a multiple of it
 *   Y            [n_indices][D] of y_dtype (QG_F32, QG_F16 or QG_BF16)
 *   status_dev   device int, written with 0 (every index valid) or 1, or NULL
 * W, scales, zero points and Y must be 16-byte aligned.  Results are exact
 * (bit-identical to the definition) whenever w is exact in fp32, e.g. for
 * integer or half-integer zero points and for every E4M3 table.
 */
enum { QG_WF_U2 = 0, QG_WF_U4 = 1, QG_WF_U8 = 2, QG_WF_E4M3 = 3 };
int qg_gather_block_quantized(const int64_t *indices, int64_t n_indices, const uint8_t *W, int w_format,
                              const uint16_t *scales_f16, const uint16_t *zero_points_f16, int64_t vocab, int D,
                              int block_size, void *Y, int y_dtype, int *status_dev, qg_stream_t stream);

/*
 * qg_read_device_fault -- every wait inside the library's kernels is
 * bounded; a wait that gives up records a bit in a device-side fault word
 * instead of hanging.  This call synchronises the current device, returns
 * the word in *flags (0: no fault since the last read) and clears it.
 * The word is one per device, shared by every call of every stream and
 * thread: a read reports (and clears) the faults of all calls on the device
 * since the previous read, whoever made them.  A caller that needs to know
 * which call gave up must read the word between its own calls, with no other
 * work on the device in between.  (A wait that gives up is a library fault --
 * a kernel that did not get its data within seconds -- not an argument
 * error: arguments are checked before anything is enqueued.)
 */
int qg_read_device_fault(unsigned int *flags);

/* Human-readable name of a QG_* status. */
const char *qg_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H */
