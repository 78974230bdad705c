/*
 * qgemm_oracle.c -- the CPU oracle for blockwise low-bit dequantize + GEMM
 * and for the fused QMoE decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU library computes.  Only the test-suite, the
 * package smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no source, header, table or helper with the CUDA library, and the
 * library never calls it.
 *
 * Sources (web pages; cited by title and section):
 *   [P1] hip-ep pull request #1318, "2-bit MatMulNBits for phi4-14B on
 *        gfx1151" -- sections Summary, Why, What (Commit 1, kernels),
 *        Performance (Model), Notes for reviewers (Follow-ups).
 *   [P2] hip-ep pull request #1328, "fused QMoE decode picks its tiling
 *        before computing" -- sections Summary, Why, What, Test plan,
 *        Notes for reviewers.
 *   [P3] bitsandbytes pull request #1979, "[ROCm] Fused 4-bit SIMT GEMM" --
 *        sections Summary, Technical details, Testing plan.
 *   [P1] also carries the kernel unit-test table (Notes for reviewers) whose
 *        leaves name the 3-bit and 8-bit MatMulNBits codes, qmoe_ragged_mm and
 *        gather_block_quantized.
 *
 * Readings of points the pages leave open (each one is also listed in the
 * design notes):
 *   - codes are packed along K, LSB-first: element k of a row sits in byte
 *     (k*bits)/8 at bit offset (k*bits)%8; a row occupies K*bits/8 bytes;
 *   - scales / zero points / absmax are row-major [N][K/bs];
 *   - an absent zero-point tensor means the midpoint 2^(bits-1);
 *   - dequantization is two fp32 round-to-nearest operations,
 *     w = (q - zp) * s, with no fused multiply-add;
 *   - SwiGLU is silu(gate) * up with gate the first half of fc1's output
 *     (or the even elements when the interleaved layout is asked for);
 *   - every matmul is accumulated in fp64, ascending k, and returned
 *     unrounded, so that a GPU result can be compared against the exact
 *     product of the dequantized operands;
 *   - 3-bit codes continue into the next byte (one bit string per row);
 *   - the embedding gather wraps negative indices once (ONNX Gather rule)
 *     and gives a zero row for any other index outside the table; "fp8" is
 *     OCP E4M3 without infinities;
 *   - int8 activations (the dp4a decode) are quantized per weight block,
 *     largest magnitude to 127, every step in fp32, ties to even;
 *   - the ragged expert GEMM groups the rows of X by expert through
 *     offsets starting at 0;
 *   - a nested absmax is table[code] * second-level scale + offset over the
 *     flat row-major sequence of per-block values;
 *   - packed unsigned-integer zero points follow the codes' packing rule:
 *     zero point b of row n is the `bits`-wide field at bit b*bits of the
 *     row's bit string, a row padding to whole bytes (ceil(nb*bits/8)).
 *
 * Parity pins: every function here is pinned by CPU tests against values
 * written by hand from the pages' statement of the problem, closed forms,
 * library routines (numpy/torch fp16 and bf16 conversions, fp64 matmul) and
 * brute-force integer arithmetic.  No function here is "parity unpinned".
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (fp32 operations
 * must stay single-rounded, hence no contraction).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* a_dtype / element type codes.  The first three match the library's enum by
 * value (they name the same IEEE formats); F64 exists only here, so that a
 * chain of oracle calls can feed an fp64 intermediate forward. */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_F64 = 3 };

/* zero-point modes */
enum { OR_ZP_NONE = 0, OR_ZP_TENSOR = 1, OR_ZP_UNIFORM = 2 };

/* ------------------------------------------------------------------------ */
/* Scalar formats.                                                          */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent 0 encodes subnormals f * 2^-24; exponent 31 encodes inf
 * (f == 0) and NaN.  Every binary16 value is exact in a double. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int dtype, size_t i)
{
    switch (dtype) {
    case OR_F32: return (double)((const float *)base)[i];
    case OR_F16: return oracle_half_to_double(((const uint16_t *)base)[i]);
    case OR_BF16: return oracle_bf16_to_double(((const uint16_t *)base)[i]);
    default: return ((const double *)base)[i];
    }
}

/* ------------------------------------------------------------------------ */
/* Unpack.  [P1] Summary / What (Commit 1): MatMulNBits with bits=2 (and the  */
/* bits=4 instantiations it leaves unchanged); [P1] Kernel Unit Test Results: */
/* u2 / u3 / u4 / 8-bit leaves; [P3] Summary: 4-bit codes decoded inside the */
/* GEMM.  Packing order: LSB-first along K (reading): code k of a row is the */
/* `bits` bits starting at bit k*bits of the row's bit string, so a 3-bit    */
/* code may continue into the next byte.                                     */
/* ------------------------------------------------------------------------ */
int oracle_code(const uint8_t *W, int64_t K, int64_t n, int64_t k, int bits)
{
    int64_t row_bytes = K * bits / 8;
    int64_t bit = k * bits;
    const uint8_t *row = W + n * row_bytes;
    unsigned v = row[bit / 8];
    if (bit % 8 + bits > 8) /* the code continues into the next byte */
        v |= (unsigned)row[bit / 8 + 1] << 8;
    return (int)((v >> (bit % 8)) & ((1u << bits) - 1u));
}

/* ------------------------------------------------------------------------ */
/* Dequantize one weight.                                                    */
/* nbits ([P1] What, Commit 1; Performance, Model: block 64, fp16 scales,    */
/* fp16 zero points, all 1.5 on phi4, collapsed to a scalar when uniform):   */
/*     w = fl32( fl32(q - zp) * s )                                          */
/* codebook ([P3] Summary; Technical details, LDS centroid lookup; Testing   */
/* plan, absmax):                                                            */
/*     w = fl32( C[q] * absmax )                                             */
/* ------------------------------------------------------------------------ */
float oracle_weight_nbits(const uint8_t *W, const uint16_t *scales, const uint16_t *zp, int zp_mode,
                          float uniform_zp, int64_t N, int64_t K, int bits, int bs, int64_t n, int64_t k)
{
    (void)N;
    int64_t nb = K / bs;
    int64_t b = k / bs;
    int q = oracle_code(W, K, n, k, bits);
    float zpv;
    if (zp_mode == OR_ZP_TENSOR)
        zpv = (float)oracle_half_to_double(zp[n * nb + b]);
    else if (zp_mode == OR_ZP_UNIFORM)
        zpv = uniform_zp;
    else
        zpv = (float)(1 << (bits - 1));
    float s = (float)oracle_half_to_double(scales[n * nb + b]);
    float d = (float)q - zpv;
    float w = d * s;
    return w;
}

float oracle_weight_codebook4(const uint8_t *W, const float *codebook, const float *absmax, int64_t K,
                              int bs, int64_t n, int64_t k)
{
    int64_t nb = K / bs;
    int q = oracle_code(W, K, n, k, 4);
    float w = codebook[q] * absmax[n * nb + k / bs];
    return w;
}

/* Dequantized matrices, fp32 [N][K].  The library's dequant-export entry
 * points must reproduce these bit for bit. */
void oracle_dequant_nbits(const uint8_t *W, const uint16_t *scales, const uint16_t *zp, int zp_mode,
                          float uniform_zp, int64_t N, int64_t K, int bits, int bs, float *out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = oracle_weight_nbits(W, scales, zp, zp_mode, uniform_zp, N, K, bits, bs, n, k);
}

void oracle_dequant_codebook4(const uint8_t *W, const float *codebook, const float *absmax, int64_t N,
                              int64_t K, int bs, float *out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = oracle_weight_codebook4(W, codebook, absmax, K, bs, n, k);
}

/* ------------------------------------------------------------------------ */
/* Matmul  Y[m, n] = sum_k A[m, k] * w[n, k]   (fp64, ascending k).          */
/* [P1] What (Commit 1): GEMV reads fp32 A and writes fp32 C directly;       */
/* [P3] Summary: decoded values reused across the M rows of a small batch.   */
/* `rows` selects which weight rows n to evaluate (NULL: all N); the result  */
/* is Y[m][j] for n = rows[j], as a dense [M][n_rows] fp64 array.           */
/* ------------------------------------------------------------------------ */
void oracle_qgemm_nbits(const void *A, int a_dtype, const uint8_t *W, const uint16_t *scales,
                        const uint16_t *zp, int zp_mode, float uniform_zp, int64_t M, int64_t N, int64_t K,
                        int bits, int bs, const int64_t *rows, int64_t n_rows, double *Y)
{
    if (!rows) n_rows = N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < n_rows; ++j) {
        int64_t n = rows ? rows[j] : j;
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = load_elem(A, a_dtype, (size_t)(m * K + k));
                double w = (double)oracle_weight_nbits(W, scales, zp, zp_mode, uniform_zp, N, K, bits, bs, n, k);
                acc += a * w;
            }
            Y[m * n_rows + j] = acc;
        }
    }
}

void oracle_qgemm_codebook4(const void *A, int a_dtype, const uint8_t *W, const float *codebook,
                            const float *absmax, int64_t M, int64_t N, int64_t K, int bs, const int64_t *rows,
                            int64_t n_rows, double *Y)
{
    if (!rows) n_rows = N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < n_rows; ++j) {
        int64_t n = rows ? rows[j] : j;
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = load_elem(A, a_dtype, (size_t)(m * K + k));
                double w = (double)oracle_weight_codebook4(W, codebook, absmax, K, bs, n, k);
                acc += a * w;
            }
            Y[m * n_rows + j] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Uniform zero point.  [P1] What (Commit 1): an all-equal fp16 zero-point    */
/* tensor is detected once per buffer and then passed as a scalar.           */
/* Equality is on bit patterns: +0 and -0 differ, and a NaN pattern is never */
/* treated as a usable scalar (reading).  Returns 1 and writes the value     */
/* when uniform, else 0.  An empty tensor is not uniform.                    */
/* ------------------------------------------------------------------------ */
int oracle_fp16_uniform_value(const uint16_t *t, int64_t n, float *value)
{
    if (n <= 0) return 0;
    for (int64_t i = 1; i < n; ++i)
        if (t[i] != t[0]) return 0;
    double v = oracle_half_to_double(t[0]);
    if (isnan(v)) return 0;
    *value = (float)v;
    return 1;
}

/* ------------------------------------------------------------------------ */
/* Fused QMoE decode, one token.                                             */
/* [P2] Summary / What: fc1 GEMV -> SwiGLU -> fc2 GEMV over the top-k        */
/* experts of one token, with u4 weights, block 32/64/128, optional zero     */
/* points and optional bias ([P2] Test plan); num_experts bounds the ids.    */
/* [P1] Why: the quantized SwiGLU chain is gate -> sigmoid -> two multiplies */
/* -> up, i.e. h = gate * sigmoid(gate) * up.                                */
/* For slot j (ascending): e = ids[j]; g = W1[e] x + b1[e];                  */
/*   gate/up halves of g; h = silu(gate) * up; o = W2[e] h + b2[e];          */
/*   y += weights[j] * o.                                                    */
/* Everything after the fp32 dequantized weights is fp64.  An expert id      */
/* outside [0, num_experts) contributes nothing and is reported through the  */
/* return value (the number of such slots).                                  */
/* Weight layouts: fc1 codes [E][2I][H*bits/8], scales/zp [E][2I][H/bs],     */
/* bias [E][2I]; fc2 codes [E][H][I*bits/8], scales/zp [E][H][I/bs],         */
/* bias [E][H].  Scratch: g [2I], h [I] doubles supplied by the caller.      */
/* ------------------------------------------------------------------------ */
static double silu(double v) { return v / (1.0 + exp(-v)); }

int oracle_qmoe_decode(const uint16_t *x_f16, const int32_t *ids, const float *weights, int k,
                       int num_experts, const uint8_t *fc1_w, const uint16_t *fc1_scales,
                       const uint16_t *fc1_zp, const uint16_t *fc1_bias, const uint8_t *fc2_w,
                       const uint16_t *fc2_scales, const uint16_t *fc2_zp, const uint16_t *fc2_bias,
                       int64_t hidden, int64_t inter, int bits, int bs, int swiglu_interleaved, double *g,
                       double *h, double *y)
{
    const int64_t H = hidden, I = inter, I2 = 2 * inter;
    const int64_t fc1_row_bytes = H * bits / 8, fc2_row_bytes = I * bits / 8;
    const int64_t fc1_nb = H / bs, fc2_nb = I / bs;
    int bad = 0;
    for (int64_t i = 0; i < H; ++i) y[i] = 0.0;

    for (int j = 0; j < k; ++j) {
        int e = ids[j];
        if (e < 0 || e >= num_experts) {
            ++bad;
            continue;
        }
        const uint8_t *w1 = fc1_w + (int64_t)e * I2 * fc1_row_bytes;
        const uint16_t *s1 = fc1_scales + (int64_t)e * I2 * fc1_nb;
        const uint16_t *z1 = fc1_zp ? fc1_zp + (int64_t)e * I2 * fc1_nb : NULL;
        const uint8_t *w2 = fc2_w + (int64_t)e * H * fc2_row_bytes;
        const uint16_t *s2 = fc2_scales + (int64_t)e * H * fc2_nb;
        const uint16_t *z2 = fc2_zp ? fc2_zp + (int64_t)e * H * fc2_nb : NULL;
        int zm1 = z1 ? OR_ZP_TENSOR : OR_ZP_NONE;
        int zm2 = z2 ? OR_ZP_TENSOR : OR_ZP_NONE;

        /* fc1: g[r] = sum_c x[c] * W1[r][c] + b1[r] */
        for (int64_t r = 0; r < I2; ++r) {
            double acc = 0.0;
            for (int64_t c = 0; c < H; ++c)
                acc += oracle_half_to_double(x_f16[c]) *
                       (double)oracle_weight_nbits(w1, s1, z1, zm1, 0.0f, I2, H, bits, bs, r, c);
            if (fc1_bias) acc += oracle_half_to_double(fc1_bias[(int64_t)e * I2 + r]);
            g[r] = acc;
        }
        /* SwiGLU */
        for (int64_t i = 0; i < I; ++i) {
            double gate = swiglu_interleaved ? g[2 * i] : g[i];
            double up = swiglu_interleaved ? g[2 * i + 1] : g[I + i];
            h[i] = silu(gate) * up;
        }
        /* fc2 and the weighted sum over slots, in slot order */
        for (int64_t r = 0; r < H; ++r) {
            double acc = 0.0;
            for (int64_t c = 0; c < I; ++c)
                acc += h[c] * (double)oracle_weight_nbits(w2, s2, z2, zm2, 0.0f, H, I, bits, bs, r, c);
            if (fc2_bias) acc += oracle_half_to_double(fc2_bias[(int64_t)e * H + r]);
            y[r] += (double)weights[j] * acc;
        }
        (void)fc1_row_bytes;
        (void)fc2_row_bytes;
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* 8-bit floating point, E4M3 ([P1] Notes for reviewers, kernel test table: */
/* gather_block_quantized leaf Xi64_Wfp8_Yfp16; the format is read as the   */
/* OCP E4M3 encoding without infinities): 1 sign bit, 4 exponent bits (bias */
/* 7), 3 fraction bits.  Exponent 0 encodes subnormals f * 2^-9; the two    */
/* patterns with every exponent and fraction bit set are NaN.               */
/* ------------------------------------------------------------------------ */
double oracle_e4m3_to_double(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, f = b & 7;
    double v;
    if (e == 15 && f == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(f + 8), e - 10);
    return s ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* Block-quantized embedding gather ([P1] Notes for reviewers, kernel test  */
/* table: gather_block_quantized leaves Xi64_Wu4_Yfp16, Xi64_Wu8_Yfp16,     */
/* Xi64_Wfp8_Yfp16; [P1] Summary, Commit 3: embedding lookups through       */
/* hip.gather).  Reading: the table is [V][D], quantized along D in blocks  */
/* of bs with the MatMulNBits layout (codes LSB-first, scales and zero      */
/* points [V][D/bs]); integer codes dequantize as in oracle_weight_nbits,   */
/* E4M3 bytes as w = fl32(e4m3(q) * s).  out[i][d] = w(row, d) for          */
/* row = idx[i], a negative index counting from the end (row = idx[i] + V). */
/* An index outside [-V, V) yields a zero row and is counted in the return  */
/* value.  out is fp32 [n][D]: the exact dequantized values, before any     */
/* rounding to an output type.                                              */
/* ------------------------------------------------------------------------ */
enum { OR_W_U2 = 0, OR_W_U4 = 1, OR_W_U8 = 2, OR_W_E4M3 = 3 };

int64_t oracle_gather_block_quantized(const int64_t *idx, int64_t n, const uint8_t *W, int wfmt,
                                      const uint16_t *scales, const uint16_t *zp, int64_t V, int64_t D,
                                      int bs, float *out)
{
    int64_t bad = 0;
    int64_t nb = D / bs;
    for (int64_t i = 0; i < n; ++i) {
        int64_t row = idx[i];
        if (row < 0)
            row += V;
        if (row < 0 || row >= V) {
            ++bad;
            for (int64_t d = 0; d < D; ++d)
                out[i * D + d] = 0.0f;
            continue;
        }
        for (int64_t d = 0; d < D; ++d) {
            float w;
            if (wfmt == OR_W_E4M3) {
                float s = (float)oracle_half_to_double(scales[row * nb + d / bs]);
                float q = (float)oracle_e4m3_to_double(W[row * D + d]);
                w = q * s;
            } else {
                int bits = wfmt == OR_W_U2 ? 2 : (wfmt == OR_W_U4 ? 4 : 8);
                w = oracle_weight_nbits(W, scales, zp, zp ? OR_ZP_TENSOR : OR_ZP_NONE, 0.0f, V, D, bits, bs,
                                        row, d);
            }
            out[i * D + d] = w;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* int8-activation QMoE decode ([P2] Summary: the fused decode "and its dp4a */
/* variant"; Test plan: fp and dp4a x block size x zero points x bias, a CPU */
/* reference that quantizes where the kernels do; Why: int8 activations).    */
/* The pages do not give the activation quantization; reading: per block of  */
/* bs consecutive values along the contraction, symmetric int8 with the      */
/* block's largest magnitude mapped to 127, every step in fp32:              */
/*     a = max |v|;  sx = fl32(a / 127);                                     */
/*     q8 = clamp(rint(fl32(v / sx)), -127, 127)   (ties to even)            */
/* and a block of zeros has sx = 0 and q8 = 0.  The decision (q8) is taken   */
/* in fp32 on both sides of any comparison.                                  */
/* ------------------------------------------------------------------------ */
void oracle_quantize_i8_blocks(const float *v, int64_t n, int bs, int8_t *q8, float *sx)
{
    for (int64_t b = 0; b < n / bs; ++b) {
        float a = 0.0f;
        for (int64_t k = b * bs; k < (b + 1) * bs; ++k) {
            float m = fabsf(v[k]);
            if (m > a)
                a = m;
        }
        if (a == 0.0f) {
            sx[b] = 0.0f;
            for (int64_t k = b * bs; k < (b + 1) * bs; ++k)
                q8[k] = 0;
            continue;
        }
        float s = a / 127.0f;
        sx[b] = s;
        for (int64_t k = b * bs; k < (b + 1) * bs; ++k) {
            float r = rintf(v[k] / s);
            if (r > 127.0f)
                r = 127.0f;
            if (r < -127.0f)
                r = -127.0f;
            q8[k] = (int8_t)r;
        }
    }
}

/* One output of a dp4a GEMV: sum over blocks b of
 *     s[r,b] * sx[b] * ( sum_{k in b} q8[k] * q[r,k]  -  zp[r,b] * sum_{k in b} q8[k] )
 * with the integer sums exact and the rest in fp64 (zp: the fp16 zero point,
 * or the midpoint 2^(bits-1) when the tensor is absent). */
static double dp4a_row(const int8_t *q8, const float *sx, const uint8_t *W, const uint16_t *scales,
                       const uint16_t *zp, int64_t K, int bits, int bs, int64_t r)
{
    int64_t nb = K / bs;
    double acc = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        int64_t dot = 0, sum = 0;
        for (int64_t k = b * bs; k < (b + 1) * bs; ++k) {
            dot += (int64_t)q8[k] * oracle_code(W, K, r, k, bits);
            sum += q8[k];
        }
        double z = zp ? oracle_half_to_double(zp[r * nb + b]) : (double)(1 << (bits - 1));
        double s = oracle_half_to_double(scales[r * nb + b]);
        acc += s * (double)sx[b] * ((double)dot - z * (double)sum);
    }
    return acc;
}

/* The decode: for slot j (ascending) with e = ids[j] in range,
 *   x8 = quantize(x);  g[r] = dp4a_row(x8, fc1[e], r) + b1[e][r];
 *   h = silu(gate) * up, rounded to fp32;  h8 = quantize(h);
 *   o[r] = dp4a_row(h8, fc2[e], r) + b2[e][r];  y += w_j * o.
 * Returns the number of out-of-range ids (their slots add nothing).
 * Scratch from the caller: g [2I] doubles, h [I] floats, q8 [max(H, I)]
 * bytes, sx [max(H, I)/bs] floats. */
int oracle_qmoe_decode_dp4a(const uint16_t *x_f16, const int32_t *ids, const float *weights, int k,
                            int num_experts, const uint8_t *fc1_w, const uint16_t *fc1_scales,
                            const uint16_t *fc1_zp, const uint16_t *fc1_bias, const uint8_t *fc2_w,
                            const uint16_t *fc2_scales, const uint16_t *fc2_zp, const uint16_t *fc2_bias,
                            int64_t hidden, int64_t inter, int bits, int bs, int swiglu_interleaved, double *g,
                            float *h, int8_t *q8, float *sx, double *y)
{
    const int64_t H = hidden, I = inter, I2 = 2 * inter;
    const int64_t fc1_row_bytes = H * bits / 8, fc2_row_bytes = I * bits / 8;
    const int64_t fc1_nb = H / bs, fc2_nb = I / bs;
    int bad = 0;
    for (int64_t i = 0; i < H; ++i) y[i] = 0.0;
    for (int j = 0; j < k; ++j) {
        int e = ids[j];
        if (e < 0 || e >= num_experts) {
            ++bad;
            continue;
        }
        const uint8_t *w1 = fc1_w + (int64_t)e * I2 * fc1_row_bytes;
        const uint16_t *s1 = fc1_scales + (int64_t)e * I2 * fc1_nb;
        const uint16_t *z1 = fc1_zp ? fc1_zp + (int64_t)e * I2 * fc1_nb : NULL;
        const uint8_t *w2 = fc2_w + (int64_t)e * H * fc2_row_bytes;
        const uint16_t *s2 = fc2_scales + (int64_t)e * H * fc2_nb;
        const uint16_t *z2 = fc2_zp ? fc2_zp + (int64_t)e * H * fc2_nb : NULL;

        for (int64_t c = 0; c < H; ++c)
            h[c] = (float)oracle_half_to_double(x_f16[c]); /* x, exactly, as the quantizer's input */
        oracle_quantize_i8_blocks(h, H, bs, q8, sx);
        for (int64_t r = 0; r < I2; ++r) {
            double acc = dp4a_row(q8, sx, w1, s1, z1, H, bits, bs, r);
            if (fc1_bias) acc += oracle_half_to_double(fc1_bias[(int64_t)e * I2 + r]);
            g[r] = acc;
        }
        for (int64_t i = 0; i < I; ++i) {
            double gate = swiglu_interleaved ? g[2 * i] : g[i];
            double up = swiglu_interleaved ? g[2 * i + 1] : g[I + i];
            h[i] = (float)(silu(gate) * up);
        }
        oracle_quantize_i8_blocks(h, I, bs, q8, sx);
        for (int64_t r = 0; r < H; ++r) {
            double acc = dp4a_row(q8, sx, w2, s2, z2, I, bits, bs, r);
            if (fc2_bias) acc += oracle_half_to_double(fc2_bias[(int64_t)e * H + r]);
            y[r] += (double)weights[j] * acc;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Ragged expert GEMM ([P1] Notes for reviewers, kernel test table:          */
/* qmoe_ragged_mm leaf Xfp16_Wu4_Yfp16; [P2] Summary: the QMoE op family).   */
/* Reading: the rows of X are grouped by expert, expert e owning rows        */
/* [off[e], off[e+1]); each row is multiplied by its expert's dequantized    */
/* MatMulNBits weight:  Y[r][n] = sum_k X[r][k] * w_e(n, k)  (fp64, ascending */
/* k, unrounded).  W is [E][N][K*bits/8], scales / zero points [E][N][K/bs]. */
/* Returns 0, or -1 (nothing written) when off[0] != 0 or the offsets        */
/* decrease.                                                                 */
/* ------------------------------------------------------------------------ */
int oracle_qmoe_ragged_mm(const void *X, int x_dtype, const int64_t *off, int E, const uint8_t *W,
                          const uint16_t *scales, const uint16_t *zp, int64_t N, int64_t K, int bits, int bs,
                          double *Y)
{
    if (off[0] != 0)
        return -1;
    for (int e = 0; e < E; ++e)
        if (off[e + 1] < off[e])
            return -1;
    const int64_t row_bytes = K * bits / 8, nb = K / bs;
    for (int e = 0; e < E; ++e) {
        const uint8_t *we = W + (int64_t)e * N * row_bytes;
        const uint16_t *se = scales + (int64_t)e * N * nb;
        const uint16_t *ze = zp ? zp + (int64_t)e * N * nb : NULL;
        for (int64_t r = off[e]; r < off[e + 1]; ++r)
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += load_elem(X, x_dtype, (size_t)(r * K + k)) *
                           (double)oracle_weight_nbits(we, se, ze, ze ? OR_ZP_TENSOR : OR_ZP_NONE, 0.0f, N, K,
                                                       bits, bs, n, k);
                Y[r * N + n] = acc;
            }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Nested ("double-quantized") absmax of the codebook GEMM ([P3] Testing     */
/* plan: quantization modes, nested / non-nested absmax).  The pages do not  */
/* give the format; reading: the per-block absmax values, taken as one flat  */
/* row-major sequence i = n * nb + b, are stored as 8-bit codes qa[i] into a */
/* 256-entry fp32 table, with one fp32 second-level scale per group of       */
/* nested_bs consecutive values and one fp32 offset:                         */
/*     absmax[i] = fl32( fl32(table[qa[i]] * absmax2[i / nested_bs]) + offset ) */
/* (two fp32 round-to-nearest operations).  The GEMM then uses absmax as the */
/* plain codebook GEMM does.                                                 */
/* ------------------------------------------------------------------------ */
void oracle_nested_absmax(const uint8_t *qa, const float *table256, const float *absmax2, float offset,
                          int nested_bs, int64_t n, float *absmax)
{
    for (int64_t i = 0; i < n; ++i) {
        float v = table256[qa[i]] * absmax2[i / nested_bs];
        absmax[i] = v + offset;
    }
}

/* ------------------------------------------------------------------------ */
/* Packed unsigned-integer zero points.  [P1] Notes for reviewers, kernel    */
/* unit-test table: MatMulNBits leaves for 2-, 3-, 4- and 8-bit weights; the */
/* pages' own zero points are fp16 ([P1] What, Commit 1).  Reading: integer  */
/* zero points may also come packed like the codes -- zero point b of row n  */
/* is the unsigned `bits`-wide field starting at bit b*bits of row n's bit   */
/* string (LSB-first, a field may continue into the next byte), each row     */
/* occupying ceil(nb*bits/8) bytes.  The GEMM is then the zero-point-tensor  */
/* GEMM with these integers as zero points (exact in fp16 for bits <= 8).    */
/* ------------------------------------------------------------------------ */
void oracle_unpack_zero_points(const uint8_t *zp, int64_t N, int64_t nb, int bits, int32_t *out)
{
    int64_t row_bytes = (nb * bits + 7) / 8;
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t *row = zp + n * row_bytes;
        for (int64_t b = 0; b < nb; ++b) {
            int64_t bit = b * bits;
            unsigned v = row[bit / 8];
            if (bit % 8 + bits > 8) /* the field continues into the next byte */
                v |= (unsigned)row[bit / 8 + 1] << 8;
            out[n * nb + b] = (int32_t)((v >> (bit % 8)) & ((1u << bits) - 1u));
        }
    }
}
