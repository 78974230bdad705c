// qg_api.cu -- the C ABI (include/qgemm.h): argument checks, error-state
// hygiene and dispatch to the kernels.
//
// Argument refusal before any launch and clearing the stale CUDA error on
// entry follow hip-ep #1328 ("What": clear the error state before the fused
// decode launches; "Test plan": the arguments the launchers must refuse).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstring>

#include "../../include/qgemm.h"
#include "qg_internal.h"

namespace qg {

__device__ unsigned g_fault_word;

namespace {
DeviceInfo g_info[kMaxDevices];
std::atomic<int> g_info_ready[kMaxDevices];
unsigned *g_fault_ptr[kMaxDevices];
std::atomic<int> g_fault_ready[kMaxDevices];

DeviceInfo query_info(int dev) {
    DeviceInfo d{};
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (d.sm_count <= 0) d.sm_count = 1;
    if (d.max_smem_optin <= 0) d.max_smem_optin = 48 * 1024;
    return d;
}
}  // namespace

int device_slot() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev < 0 || dev >= kMaxDevices ? -1 : dev;
}

const DeviceInfo &device_info() {
    const int slot = device_slot();
    if (slot < 0) {  // not cached: this thread's copy, queried now
        thread_local DeviceInfo d;
        int dev = 0;
        cudaGetDevice(&dev);
        d = query_info(dev);
        return d;
    }
    if (!g_info_ready[slot].load(std::memory_order_acquire)) {
        g_info[slot] = query_info(slot);
        g_info_ready[slot].store(1, std::memory_order_release);
    }
    return g_info[slot];
}

unsigned *fault_word() {
    const int slot = device_slot();
    if (slot < 0 || !g_fault_ready[slot].load(std::memory_order_acquire)) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fault_word) != cudaSuccess) return nullptr;
        if (slot < 0) return static_cast<unsigned *>(p);
        g_fault_ptr[slot] = static_cast<unsigned *>(p);
        g_fault_ready[slot].store(1, std::memory_order_release);
    }
    return g_fault_ptr[slot];
}

}  // namespace qg

namespace {

using qg::GemmProblem;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_dtype(int d) { return d == QG_F32 || d == QG_F16 || d == QG_BF16; }
bool valid_bs(int bs) { return bs == 32 || bs == 64 || bs == 128 || bs == 256; }

// Sizes beyond these are valid in principle but not implemented (32-bit
// index arithmetic inside the kernels).
constexpr long long kMaxK = 1 << 24;
constexpr long long kMaxN = 1 << 28;
constexpr long long kMaxM = 1 << 20;

// Code widths of the GEMM entry points: MatMulNBits u2 / u3 / u4 / u8 (the codebook is 4-bit).
bool valid_bits(int bits) { return bits == 2 || bits == 3 || bits == 4 || bits == 8; }

// The workspace a GEMM call cannot do without (the SIMT split-K partials, the
// tensor-core tail pieces).
size_t gemm_workspace_min(int a_dtype, int M, int N, int K, int bits, int bs) {
    if (M <= 0 || N <= 0 || K <= 0 || !valid_bits(bits) || !valid_bs(bs) || K % bs) return 0;
    // the query has no weight kind: the larger need of MatMulNBits and codebook
    // (their tensor-core eligibility differs when K / bs is not a multiple of 8)
    size_t need = 0;
    for (int kind : {qg::WK_NBITS, qg::WK_CODEBOOK})
        need = std::max(need, qg::tc_eligible(M, K, bits, a_dtype, bs, kind) ? qg::tc_workspace_bytes(M, N, K, bits)
                                                                              : qg::simt_workspace_bytes(M, N, K, bits, bs));
    return need;
}

// The workspace the query reports: the minimum, or, for fp32 activations with
// enough rows on a tensor-core shape, room for the split-precision path (a
// call whose workspace is smaller takes the slower path instead).
size_t gemm_workspace(int a_dtype, int M, int N, int K, int bits, int bs) {
    size_t need = gemm_workspace_min(a_dtype, M, N, K, bits, bs);
    if (need == 0 && (M <= 0 || N <= 0 || K <= 0 || !valid_bits(bits) || !valid_bs(bs) || K % bs)) return 0;
    if (a_dtype == QG_F32 && M >= qg::kSplitMinRows && qg::tc_eligible(M, K, bits, QG_F16, bs, qg::WK_NBITS))
        need = std::max(need, qg::split_workspace_bytes(M, K));
    return need;
}

// Common checks of the three GEMM entry points.  `params` is the scales or
// absmax pointer.
int check_gemm(const void *A, int a_dtype, const uint8_t *W, const void *params, const void *zp, const void *Y,
               int y_dtype, int M, int N, int K, int bits, int bs, const void *ws, size_t ws_bytes) {
    if (!valid_dtype(a_dtype) || !valid_dtype(y_dtype)) return QG_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (!valid_bits(bits)) return QG_ERR_UNSUPPORTED;
    if (!valid_bs(bs)) return QG_ERR_UNSUPPORTED;
    if (K % bs) return QG_ERR_INVALID_ARG;
    if (M > kMaxM || N > kMaxN || K > kMaxK) return QG_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return QG_OK;
    if (!Y) return QG_ERR_INVALID_ARG;
    if (K > 0) {
        if (!A || !W || !params) return QG_ERR_INVALID_ARG;
        if (!aligned16(A) || !aligned16(W) || !aligned16(params)) return QG_ERR_INVALID_ARG;
        if (zp && !aligned16(zp)) return QG_ERR_INVALID_ARG;
    }
    const size_t need = gemm_workspace_min(a_dtype, M, N, K, bits, bs);
    if (need > 0) {
        if (!ws || ws_bytes < need) return QG_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned16(ws)) return QG_ERR_INVALID_ARG;
    }
    return QG_OK;
}

size_t elem_size(int dtype) { return dtype == QG_F32 ? 4 : 2; }

int run_gemm(const GemmProblem &p, void *ws, size_t ws_bytes, cudaStream_t s) {
    if (p.M == 0 || p.N == 0) return QG_OK;
    if (p.K == 0) {
        if (cudaMemsetAsync(p.Y, 0, static_cast<size_t>(p.M) * p.N * elem_size(p.y_dtype), s) != cudaSuccess)
            return QG_ERR_CUDA;
        return QG_OK;
    }
    const bool split = qg::split_eligible(p) && ws && aligned16(ws) && ws_bytes >= qg::split_workspace_bytes(p.M, p.K);
    const bool packed = p.zp_mode == qg::ZP_PACKED;  // chosen only where the SIMT kernel takes the request
    const cudaError_t e = packed                                                            ? qg::simt_gemm(p, ws, ws_bytes, s)
                          : split                                                           ? qg::split_gemm(p, ws, ws_bytes, s)
                          : qg::tc_eligible(p.M, p.K, p.bits, p.a_dtype, p.bs, p.kind) ? qg::tc_gemm(p, ws, ws_bytes, s)
                          : qg::mma_gemv_eligible(p)                                   ? qg::mma_gemv(p, s)
                                                                                       : qg::simt_gemm(p, ws, ws_bytes, s);
    if (e == cudaErrorNotSupported) return QG_ERR_UNSUPPORTED;
    return e == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

int nbits_common(const void *A, int a_dtype, const uint8_t *W, const uint16_t *scales, const uint16_t *zp,
                 int zp_mode, float uniform_zp, void *Y, int y_dtype, int M, int N, int K, int bits, int bs,
                 void *ws, size_t ws_bytes, qg_stream_t stream) {
    (void)cudaGetLastError();  // do not report an earlier, unrelated failure as ours
    const int st = check_gemm(A, a_dtype, W, scales, zp, Y, y_dtype, M, N, K, bits, bs, ws, ws_bytes);
    if (st != QG_OK) return st;
    GemmProblem p{};
    p.A = A;
    p.a_dtype = a_dtype;
    p.W = W;
    p.kind = qg::WK_NBITS;
    p.scales = scales;
    p.zp = zp;
    p.zp_mode = zp_mode;
    p.uniform_zp = zp_mode == qg::ZP_NONE ? static_cast<float>(1 << (bits - 1)) : uniform_zp;
    p.Y = Y;
    p.y_dtype = y_dtype;
    p.M = M;
    p.N = N;
    p.K = K;
    p.bits = bits;
    p.bs = bs;
    return run_gemm(p, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int qmoe_common(bool dp4a, const uint16_t *x_f16, const int32_t *expert_ids, const float *expert_weights, int k,
                int num_experts, const uint8_t *fc1_w, const uint16_t *fc1_scales, const uint16_t *fc1_zp,
                const uint16_t *fc1_bias, const uint8_t *fc2_w, const uint16_t *fc2_scales, const uint16_t *fc2_zp,
                const uint16_t *fc2_bias, int hidden, int inter, int bits, int block_size, int swiglu_interleaved,
                uint16_t *y_f16, int *status_dev, void *workspace, size_t workspace_bytes, qg_stream_t stream) {
    (void)cudaGetLastError();  // do not report an earlier, unrelated failure as ours
    if (k < 0 || num_experts < 0 || hidden <= 0 || inter <= 0) return QG_ERR_INVALID_ARG;
    if (swiglu_interleaved != 0 && swiglu_interleaved != 1) return QG_ERR_INVALID_ARG;
    if (bits != 2 && bits != 4) return QG_ERR_UNSUPPORTED;
    if (!valid_bs(block_size)) return QG_ERR_UNSUPPORTED;
    if (hidden % block_size || inter % block_size) return QG_ERR_INVALID_ARG;
    if (hidden > kMaxK || inter > kMaxK / 2 || k > 4096) return QG_ERR_UNSUPPORTED;
    if (dp4a && (hidden > 65536 || inter > 65536)) return QG_ERR_UNSUPPORTED;  // quantized vector in shared memory
    if (!x_f16 || !y_f16) return QG_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (k == 0) {
        if (cudaMemsetAsync(y_f16, 0, static_cast<size_t>(hidden) * 2, s) != cudaSuccess) return QG_ERR_CUDA;
        if (status_dev && cudaMemsetAsync(status_dev, 0, sizeof(int), s) != cudaSuccess) return QG_ERR_CUDA;
        return QG_OK;
    }
    if (num_experts < 1 || !expert_ids || !expert_weights || !fc1_w || !fc1_scales || !fc2_w || !fc2_scales)
        return QG_ERR_INVALID_ARG;
    const void *al16[] = {fc1_w, fc1_scales, fc2_w, fc2_scales};
    for (const void *q : al16)
        if (!aligned16(q)) return QG_ERR_INVALID_ARG;
    if ((fc1_zp && !aligned16(fc1_zp)) || (fc2_zp && !aligned16(fc2_zp))) return QG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(expert_ids) | reinterpret_cast<uintptr_t>(expert_weights)) & 3u)
        return QG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x_f16) | reinterpret_cast<uintptr_t>(y_f16) |
         reinterpret_cast<uintptr_t>(fc1_bias) | reinterpret_cast<uintptr_t>(fc2_bias)) & 1u)
        return QG_ERR_INVALID_ARG;
    if (status_dev && (reinterpret_cast<uintptr_t>(status_dev) & 3u)) return QG_ERR_INVALID_ARG;
    const size_t need = qg::qmoe_workspace_bytes(k, hidden, inter);
    if (!workspace || workspace_bytes < need) return QG_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return QG_ERR_INVALID_ARG;
    qg::QmoeProblem q{};
    q.x = x_f16;
    q.ids = expert_ids;
    q.weights = expert_weights;
    q.k = k;
    q.num_experts = num_experts;
    q.fc1_w = fc1_w;
    q.fc1_scales = fc1_scales;
    q.fc1_zp = fc1_zp;
    q.fc1_bias = fc1_bias;
    q.fc2_w = fc2_w;
    q.fc2_scales = fc2_scales;
    q.fc2_zp = fc2_zp;
    q.fc2_bias = fc2_bias;
    q.hidden = hidden;
    q.inter = inter;
    q.bits = bits;
    q.bs = block_size;
    q.swiglu_interleaved = swiglu_interleaved;
    q.y = y_f16;
    q.status = status_dev;
    // int8 activations: the SIMT kernel's dp4a kind where it has a plan, else the plain-load kernels
    // (rows that are not a multiple of 16 bytes)
    const cudaError_t e = !dp4a                         ? qg::qmoe_decode(q, workspace, s)
                          : qg::qmoe_dp4a_simt_ok(q) ? qg::qmoe_decode(q, workspace, s, true)
                                                     : qg::qmoe_decode_dp4a(q, workspace, s);
    if (e == cudaErrorNotSupported) return QG_ERR_UNSUPPORTED;
    return e == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

// Ragged expert GEMM: the checks and the plan.  Experts with at least
// kRaggedTcRows rows run in one grouped tensor-core launch when the shape is
// eligible; every other expert with rows is one ordinary GEMM call on its
// slice (SIMT for few rows or fp32 activations).
constexpr int kRaggedTcRows = 9;

// Offsets, types and sizes; *T_out = total rows.
int ragged_check_shape(const int64_t *off, int E, int x_dtype, int y_dtype, int N, int K, int bits, int bs,
                       long long *T_out) {
    if (!off || E < 1) return QG_ERR_INVALID_ARG;
    if (off[0] != 0) return QG_ERR_INVALID_ARG;
    for (int e = 0; e < E; ++e)
        if (off[e + 1] < off[e]) return QG_ERR_INVALID_ARG;
    const long long T = off[E];
    if (!valid_dtype(x_dtype) || !valid_dtype(y_dtype) || N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (bits != 2 && bits != 4 && bits != 8) return QG_ERR_UNSUPPORTED;
    if (!valid_bs(bs)) return QG_ERR_UNSUPPORTED;
    if (K % bs) return QG_ERR_INVALID_ARG;
    if (T > kMaxM || N > kMaxN || K > kMaxK || E > (1 << 20)) return QG_ERR_UNSUPPORTED;
    // each expert's slice of the stacked tensors must keep 16-byte alignment
    if ((static_cast<long long>(N) * K * bits / 8) % 16 || (static_cast<long long>(N) * (K / bs) * 2) % 16)
        return QG_ERR_UNSUPPORTED;
    *T_out = T;
    return QG_OK;
}

int ragged_check(const void *X, int x_dtype, const int64_t *off, int E, const uint8_t *W, const uint16_t *scales,
                 const uint16_t *zp, const void *Y, int y_dtype, int N, int K, int bits, int bs, long long *T_out) {
    const int st = ragged_check_shape(off, E, x_dtype, y_dtype, N, K, bits, bs, T_out);
    if (st != QG_OK || *T_out == 0 || N == 0) return st;
    if (!Y) return QG_ERR_INVALID_ARG;
    if (K > 0) {
        if (!X || !W || !scales) return QG_ERR_INVALID_ARG;
        if (!aligned16(X) || !aligned16(W) || !aligned16(scales) || (zp && !aligned16(zp))) return QG_ERR_INVALID_ARG;
    }
    return QG_OK;
}

bool ragged_grouped(int x_dtype, int E, int K, int bits, int bs) {
    return E <= 256 && qg::tc_eligible(kRaggedTcRows, K, bits, x_dtype, bs, qg::WK_NBITS);
}

size_t ragged_workspace(int x_dtype, const int64_t *off, int E, int N, int K, int bits, int bs) {
    const bool grouped = ragged_grouped(x_dtype, E, K, bits, bs);
    size_t need = 0;
    for (int e = 0; e < E; ++e) {
        const long long c = off[e + 1] - off[e];
        if (c <= 0 || (grouped && c >= kRaggedTcRows)) continue;
        need = std::max(need, gemm_workspace(x_dtype, static_cast<int>(c), N, K, bits, bs));
    }
    return need;
}

}  // namespace

extern "C" {

int qgemm_nbits(const void *A, int a_dtype, const uint8_t *W, const uint16_t *scales_f16,
                const uint16_t *zero_points_f16, void *Y, int y_dtype, int M, int N, int K, int bits, int block_size,
                void *workspace, size_t workspace_bytes, qg_stream_t stream) {
    return nbits_common(A, a_dtype, W, scales_f16, zero_points_f16,
                        zero_points_f16 ? qg::ZP_TENSOR : qg::ZP_NONE, 0.f, Y, y_dtype, M, N, K, bits, block_size,
                        workspace, workspace_bytes, stream);
}

int qgemm_nbits_uniform_zp(const void *A, int a_dtype, const uint8_t *W, const uint16_t *scales_f16,
                           float uniform_zp, void *Y, int y_dtype, int M, int N, int K, int bits, int block_size,
                           void *workspace, size_t workspace_bytes, qg_stream_t stream) {
    if (!(uniform_zp == uniform_zp) || uniform_zp > 65504.f || uniform_zp < -65504.f) {
        (void)cudaGetLastError();
        return QG_ERR_INVALID_ARG;  // not a finite fp16 value
    }
    return nbits_common(A, a_dtype, W, scales_f16, nullptr, qg::ZP_UNIFORM, uniform_zp, Y, y_dtype, M, N, K, bits,
                        block_size, workspace, workspace_bytes, stream);
}

int qgemm_codebook4(const void *A, int a_dtype, const uint8_t *W, const float *codebook16, const float *absmax,
                    void *Y, int y_dtype, int M, int N, int K, int block_size, void *workspace,
                    size_t workspace_bytes, qg_stream_t stream) {
    (void)cudaGetLastError();
    int st = check_gemm(A, a_dtype, W, absmax, nullptr, Y, y_dtype, M, N, K, 4, block_size, workspace,
                        workspace_bytes);
    if (st != QG_OK) return st;
    if (M > 0 && N > 0 && K > 0 && !codebook16) return QG_ERR_INVALID_ARG;
    GemmProblem p{};
    p.A = A;
    p.a_dtype = a_dtype;
    p.W = W;
    p.kind = qg::WK_CODEBOOK;
    p.codebook = codebook16;
    p.absmax = absmax;
    p.Y = Y;
    p.y_dtype = y_dtype;
    p.M = M;
    p.N = N;
    p.K = K;
    p.bits = 4;
    p.bs = block_size;
    return run_gemm(p, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t qgemm_codebook4_nested_workspace_bytes(int a_dtype, int M, int N, int K, int block_size) {
    if (M <= 0 || N <= 0 || K <= 0 || !valid_bs(block_size) || K % block_size) return 0;
    const size_t expanded = (static_cast<size_t>(N) * (K / block_size) * sizeof(float) + 255) / 256 * 256;
    return expanded + gemm_workspace(a_dtype, M, N, K, 4, block_size);
}

int qgemm_codebook4_nested(const void *A, int a_dtype, const uint8_t *W, const float *codebook16,
                           const uint8_t *absmax_q, const float *absmax_table256, const float *absmax2,
                           float absmax_offset, int nested_block, void *Y, int y_dtype, int M, int N, int K,
                           int block_size, void *workspace, size_t workspace_bytes, qg_stream_t stream) {
    (void)cudaGetLastError();
    if (!valid_dtype(a_dtype) || !valid_dtype(y_dtype) || M < 0 || N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (!valid_bs(block_size)) return QG_ERR_UNSUPPORTED;
    if (K % block_size) return QG_ERR_INVALID_ARG;
    if (M > kMaxM || N > kMaxN || K > kMaxK) return QG_ERR_UNSUPPORTED;
    if (nested_block < 1 || !(absmax_offset == absmax_offset)) return QG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return QG_OK;
    if (!Y) return QG_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {
        GemmProblem z{};
        z.Y = Y;
        z.y_dtype = y_dtype;
        z.M = M;
        z.N = N;
        return run_gemm(z, nullptr, 0, s);  // an empty sum: zeros
    }
    if (!A || !W || !codebook16 || !absmax_q || !absmax_table256 || !absmax2) return QG_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(W)) return QG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(absmax_table256) | reinterpret_cast<uintptr_t>(absmax2)) & 3u)
        return QG_ERR_INVALID_ARG;
    const size_t need = qgemm_codebook4_nested_workspace_bytes(a_dtype, M, N, K, block_size);
    if (!workspace || workspace_bytes < need) return QG_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return QG_ERR_INVALID_ARG;
    const size_t n = static_cast<size_t>(N) * (K / block_size);
    float *absmax = static_cast<float *>(workspace);
    if (qg::launch_nested_absmax(absmax_q, absmax_table256, absmax2, absmax_offset, nested_block, n, absmax, s) !=
        cudaSuccess)
        return QG_ERR_CUDA;
    const size_t expanded = (n * sizeof(float) + 255) / 256 * 256;
    GemmProblem p{};
    p.A = A;
    p.a_dtype = a_dtype;
    p.W = W;
    p.kind = qg::WK_CODEBOOK;
    p.codebook = codebook16;
    p.absmax = absmax;
    p.Y = Y;
    p.y_dtype = y_dtype;
    p.M = M;
    p.N = N;
    p.K = K;
    p.bits = 4;
    p.bs = block_size;
    return run_gemm(p, static_cast<char *>(workspace) + expanded, workspace_bytes - expanded, s);
}

size_t qgemm_workspace_bytes(int a_dtype, int M, int N, int K, int bits, int block_size) {
    return gemm_workspace(a_dtype, M, N, K, bits, block_size);
}

size_t qgemm_nbits_packed_zp_workspace_bytes(int a_dtype, int M, int N, int K, int bits, int block_size) {
    if (M <= 0 || N <= 0 || K <= 0 || !valid_bits(bits) || !valid_bs(block_size) || K % block_size) return 0;
    const size_t expanded = (static_cast<size_t>(N) * (K / block_size) * sizeof(uint16_t) + 255) / 256 * 256;
    return expanded + gemm_workspace(a_dtype, M, N, K, bits, block_size);
}

int qgemm_nbits_packed_zp(const void *A, int a_dtype, const uint8_t *W, const uint16_t *scales_f16,
                          const uint8_t *zero_points_packed, void *Y, int y_dtype, int M, int N, int K, int bits,
                          int block_size, void *workspace, size_t workspace_bytes, qg_stream_t stream) {
    (void)cudaGetLastError();
    if (!valid_dtype(a_dtype) || !valid_dtype(y_dtype) || M < 0 || N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (!valid_bits(bits) || !valid_bs(block_size)) return QG_ERR_UNSUPPORTED;
    if (K % block_size) return QG_ERR_INVALID_ARG;
    if (M > kMaxM || N > kMaxN || K > kMaxK) return QG_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return QG_OK;
    if (!Y) return QG_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {
        GemmProblem z{};
        z.Y = Y;
        z.y_dtype = y_dtype;
        z.M = M;
        z.N = N;
        return run_gemm(z, nullptr, 0, s);  // an empty sum: zeros
    }
    if (!zero_points_packed) return QG_ERR_INVALID_ARG;
    const size_t need = qgemm_nbits_packed_zp_workspace_bytes(a_dtype, M, N, K, bits, block_size);
    if (!workspace || workspace_bytes < need) return QG_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return QG_ERR_INVALID_ARG;
    const int nb = K / block_size;
    const size_t expanded = (static_cast<size_t>(N) * nb * sizeof(uint16_t) + 255) / 256 * 256;
    uint16_t *zp16 = static_cast<uint16_t *>(workspace);
    void *gws = static_cast<char *>(workspace) + expanded;
    const size_t gws_bytes = workspace_bytes - expanded;
    // everything qgemm_nbits checks, before anything is enqueued
    const int st = check_gemm(A, a_dtype, W, scales_f16, zp16, Y, y_dtype, M, N, K, bits, block_size, gws, gws_bytes);
    if (st != QG_OK) return st;
    GemmProblem p{};
    p.A = A;
    p.a_dtype = a_dtype;
    p.W = W;
    p.kind = qg::WK_NBITS;
    p.scales = scales_f16;
    p.zp = zp16;
    p.zp_mode = qg::ZP_TENSOR;
    p.Y = Y;
    p.y_dtype = y_dtype;
    p.M = M;
    p.N = N;
    p.K = K;
    p.bits = bits;
    p.bs = block_size;
    // A request the SIMT kernel takes stages the packed bytes with the codes
    // and widens each zero point where it is used; the others (tensor-pipe
    // GEMV, tensor cores) read an fp16 copy widened into the workspace first.
    const bool split = qg::split_eligible(p) && aligned16(gws) && gws_bytes >= qg::split_workspace_bytes(M, K);
    const bool simt = !split && !qg::tc_eligible(M, K, bits, a_dtype, block_size, qg::WK_NBITS) && !qg::mma_gemv_eligible(p);
    GemmProblem q = p;
    q.zp = nullptr;
    q.zp_packed = zero_points_packed;
    q.zp_mode = qg::ZP_PACKED;
    if (simt && qg::simt_packed_zp_ok(q)) return run_gemm(q, gws, gws_bytes, s);
    if (qg::launch_unpack_zero_points(zero_points_packed, bits, N, nb, zp16, s) != cudaSuccess) return QG_ERR_CUDA;
    return run_gemm(p, gws, gws_bytes, s);
}

int qmoe_decode_fused(const uint16_t *x_f16, const int32_t *expert_ids, const float *expert_weights, int k,
                      int num_experts, const uint8_t *fc1_w, const uint16_t *fc1_scales, const uint16_t *fc1_zp,
                      const uint16_t *fc1_bias, const uint8_t *fc2_w, const uint16_t *fc2_scales,
                      const uint16_t *fc2_zp, const uint16_t *fc2_bias, int hidden, int inter, int bits,
                      int block_size, int swiglu_interleaved, uint16_t *y_f16, int *status_dev, void *workspace,
                      size_t workspace_bytes, qg_stream_t stream) {
    return qmoe_common(false, x_f16, expert_ids, expert_weights, k, num_experts, fc1_w, fc1_scales, fc1_zp, fc1_bias,
                       fc2_w, fc2_scales, fc2_zp, fc2_bias, hidden, inter, bits, block_size, swiglu_interleaved, y_f16,
                       status_dev, workspace, workspace_bytes, stream);
}

int qmoe_decode_fused_dp4a(const uint16_t *x_f16, const int32_t *expert_ids, const float *expert_weights, int k,
                           int num_experts, const uint8_t *fc1_w, const uint16_t *fc1_scales, const uint16_t *fc1_zp,
                           const uint16_t *fc1_bias, const uint8_t *fc2_w, const uint16_t *fc2_scales,
                           const uint16_t *fc2_zp, const uint16_t *fc2_bias, int hidden, int inter, int bits,
                           int block_size, int swiglu_interleaved, uint16_t *y_f16, int *status_dev, void *workspace,
                           size_t workspace_bytes, qg_stream_t stream) {
    return qmoe_common(true, x_f16, expert_ids, expert_weights, k, num_experts, fc1_w, fc1_scales, fc1_zp, fc1_bias,
                       fc2_w, fc2_scales, fc2_zp, fc2_bias, hidden, inter, bits, block_size, swiglu_interleaved, y_f16,
                       status_dev, workspace, workspace_bytes, stream);
}

size_t qmoe_decode_workspace_bytes(int k, int hidden, int inter) {
    return qg::qmoe_workspace_bytes(k, hidden, inter);
}

int qg_fp16_uniform_value(const uint16_t *t, size_t n, int *is_uniform, float *value, void *workspace,
                          size_t workspace_bytes, qg_stream_t stream) {
    (void)cudaGetLastError();
    if (!is_uniform || !value) return QG_ERR_INVALID_ARG;
    if (n == 0) {
        *is_uniform = 0;
        return QG_OK;
    }
    if (!t || !aligned16(t)) return QG_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace)) return QG_ERR_INVALID_ARG;
    if (workspace_bytes < 16) return QG_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned *ws = static_cast<unsigned *>(workspace);
    if (qg::launch_uniform_check(t, n, ws, s) != cudaSuccess) return QG_ERR_CUDA;
    unsigned diff = 0;
    uint16_t first = 0;
    if (cudaMemcpyAsync(&diff, ws, sizeof diff, cudaMemcpyDeviceToHost, s) != cudaSuccess) return QG_ERR_CUDA;
    if (cudaMemcpyAsync(&first, t, sizeof first, cudaMemcpyDeviceToHost, s) != cudaSuccess) return QG_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QG_ERR_CUDA;
    const bool nan = (first & 0x7C00u) == 0x7C00u && (first & 0x03FFu) != 0u;
    if (diff || nan) {
        *is_uniform = 0;
        return QG_OK;
    }
    // binary16 -> float (exact)
    const uint32_t sign = (first >> 15) & 1u, ex = (first >> 10) & 31u, fr = first & 1023u;
    float v;
    if (ex == 0)
        v = static_cast<float>(fr) * (1.0f / 16777216.0f);
    else if (ex == 31)
        v = INFINITY;
    else {
        uint32_t bits = ((ex - 15 + 127) << 23) | (fr << 13);
        std::memcpy(&v, &bits, sizeof v);
    }
    *value = sign ? -v : v;
    *is_uniform = 1;
    return QG_OK;
}

static int dequant_common(GemmProblem &p, float *out, qg_stream_t stream) {
    (void)cudaGetLastError();
    if (p.N < 0 || p.K < 0) return QG_ERR_INVALID_ARG;
    if (!valid_bits(p.bits)) return QG_ERR_UNSUPPORTED;
    if (!valid_bs(p.bs)) return QG_ERR_UNSUPPORTED;
    if (p.K % p.bs) return QG_ERR_INVALID_ARG;
    if (p.N > kMaxN || p.K > kMaxK) return QG_ERR_UNSUPPORTED;
    if (p.N == 0 || p.K == 0) return QG_OK;
    const void *params = p.kind == qg::WK_CODEBOOK ? static_cast<const void *>(p.absmax) : p.scales;
    if (!p.W || !params || !out) return QG_ERR_INVALID_ARG;
    if (p.kind == qg::WK_CODEBOOK && !p.codebook) return QG_ERR_INVALID_ARG;
    if (!aligned16(p.W) || !aligned16(params) || !aligned16(out) || (p.zp && !aligned16(p.zp)))
        return QG_ERR_INVALID_ARG;
    return qg::launch_dequant(p, out, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

int qg_dequant_nbits(const uint8_t *W, const uint16_t *scales_f16, const uint16_t *zero_points_f16, float *out,
                     int N, int K, int bits, int block_size, qg_stream_t stream) {
    GemmProblem p{};
    p.W = W;
    p.kind = qg::WK_NBITS;
    p.scales = scales_f16;
    p.zp = zero_points_f16;
    p.zp_mode = zero_points_f16 ? qg::ZP_TENSOR : qg::ZP_NONE;
    p.uniform_zp = valid_bits(bits) ? static_cast<float>(1 << (bits - 1)) : 0.f;
    p.N = N;
    p.K = K;
    p.bits = bits;
    p.bs = block_size;
    return dequant_common(p, out, stream);
}

int qg_dequant_nbits_uniform_zp(const uint8_t *W, const uint16_t *scales_f16, float uniform_zp, float *out, int N,
                                int K, int bits, int block_size, qg_stream_t stream) {
    GemmProblem p{};
    p.W = W;
    p.kind = qg::WK_NBITS;
    p.scales = scales_f16;
    p.zp_mode = qg::ZP_UNIFORM;
    p.uniform_zp = uniform_zp;
    p.N = N;
    p.K = K;
    p.bits = bits;
    p.bs = block_size;
    return dequant_common(p, out, stream);
}

int qg_dequant_codebook4(const uint8_t *W, const float *codebook16, const float *absmax, float *out, int N, int K,
                         int block_size, qg_stream_t stream) {
    GemmProblem p{};
    p.W = W;
    p.kind = qg::WK_CODEBOOK;
    p.codebook = codebook16;
    p.absmax = absmax;
    p.N = N;
    p.K = K;
    p.bits = 4;
    p.bs = block_size;
    return dequant_common(p, out, stream);
}

int qg_gather_block_quantized(const int64_t *indices, int64_t n_indices, const uint8_t *W, int w_format,
                              const uint16_t *scales_f16, const uint16_t *zero_points_f16, int64_t vocab, int D,
                              int block_size, void *Y, int y_dtype, int *status_dev, qg_stream_t stream) {
    (void)cudaGetLastError();
    if (n_indices < 0 || vocab < 0 || D < 0) return QG_ERR_INVALID_ARG;
    if (w_format < QG_WF_U2 || w_format > QG_WF_E4M3) return QG_ERR_UNSUPPORTED;
    if (y_dtype != QG_F32 && y_dtype != QG_F16 && y_dtype != QG_BF16) return QG_ERR_UNSUPPORTED;
    if (!valid_bs(block_size)) return QG_ERR_UNSUPPORTED;
    if (D % block_size) return QG_ERR_INVALID_ARG;
    if (w_format == QG_WF_E4M3 && zero_points_f16) return QG_ERR_INVALID_ARG;
    if (D > kMaxK) return QG_ERR_UNSUPPORTED;
    if (status_dev && (reinterpret_cast<uintptr_t>(status_dev) & 3u)) return QG_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (status_dev && cudaMemsetAsync(status_dev, 0, sizeof(int), s) != cudaSuccess) return QG_ERR_CUDA;
    if (n_indices == 0 || D == 0) return QG_OK;
    if (!indices || !Y) return QG_ERR_INVALID_ARG;
    if (vocab > 0 && (!W || !scales_f16)) return QG_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(indices) & 7u) return QG_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(scales_f16) || !aligned16(Y) || (zero_points_f16 && !aligned16(zero_points_f16)))
        return QG_ERR_INVALID_ARG;
    qg::GatherProblem g{};
    g.idx = indices;
    g.n = n_indices;
    g.W = W;
    g.fmt = w_format;
    g.scales = scales_f16;
    g.zp = zero_points_f16;
    g.V = vocab;
    g.D = D;
    g.bs = block_size;
    g.Y = Y;
    g.y_dtype = y_dtype;
    g.status = status_dev;
    return qg::launch_gather(g, s) == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

size_t qmoe_ragged_mm_workspace_bytes(int x_dtype, const int64_t *expert_offsets, int num_experts, int N, int K,
                                      int bits, int block_size) {
    long long T = 0;
    if (ragged_check_shape(expert_offsets, num_experts, x_dtype, QG_F32, N, K, bits, block_size, &T) != QG_OK)
        return 0;
    return ragged_workspace(x_dtype, expert_offsets, num_experts, N, K, bits, block_size);
}

int qmoe_ragged_mm(const void *X, int x_dtype, const int64_t *expert_offsets, int num_experts, const uint8_t *W,
                   const uint16_t *scales_f16, const uint16_t *zero_points_f16, void *Y, int y_dtype, int N, int K,
                   int bits, int block_size, void *workspace, size_t workspace_bytes, qg_stream_t stream) {
    (void)cudaGetLastError();
    long long T = 0;
    int st = ragged_check(X, x_dtype, expert_offsets, num_experts, W, scales_f16, zero_points_f16, Y, y_dtype, N, K,
                          bits, block_size, &T);
    if (st != QG_OK || T == 0 || N == 0) return st;
    const size_t need = ragged_workspace(x_dtype, expert_offsets, num_experts, N, K, bits, block_size);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return QG_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned16(workspace)) return QG_ERR_INVALID_ARG;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    GemmProblem p{};
    p.A = X;
    p.a_dtype = x_dtype;
    p.W = W;
    p.kind = qg::WK_NBITS;
    p.scales = scales_f16;
    p.zp = zero_points_f16;
    p.zp_mode = zero_points_f16 ? qg::ZP_TENSOR : qg::ZP_NONE;
    p.uniform_zp = static_cast<float>(1 << (bits - 1));
    p.Y = Y;
    p.y_dtype = y_dtype;
    p.M = static_cast<int>(T);
    p.N = N;
    p.K = K;
    p.bits = bits;
    p.bs = block_size;
    const bool grouped = K > 0 && ragged_grouped(x_dtype, num_experts, K, bits, block_size);
    if (grouped) {
        const cudaError_t e = qg::tc_gemm_grouped(p, expert_offsets, num_experts, kRaggedTcRows, s);
        if (e == cudaErrorNotSupported) return QG_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return QG_ERR_CUDA;
    }
    const size_t w_stride = static_cast<size_t>(N) * K * bits / 8, p_stride = static_cast<size_t>(N) * (K / block_size);
    for (int e = 0; e < num_experts; ++e) {
        const long long r0 = expert_offsets[e], c = expert_offsets[e + 1] - r0;
        if (c == 0 || (grouped && c >= kRaggedTcRows)) continue;
        GemmProblem q = p;
        q.A = static_cast<const char *>(X) + static_cast<size_t>(r0) * K * elem_size(x_dtype);
        q.W = W + e * w_stride;
        q.scales = scales_f16 + e * p_stride;
        q.zp = zero_points_f16 ? zero_points_f16 + e * p_stride : nullptr;
        q.Y = static_cast<char *>(Y) + static_cast<size_t>(r0) * N * elem_size(y_dtype);
        q.M = static_cast<int>(c);
        st = run_gemm(q, workspace, workspace_bytes, s);
        if (st != QG_OK) return st;
    }
    return QG_OK;
}

size_t qmoe_ragged_mm_device_offsets_workspace_bytes(int num_experts) {
    (void)num_experts;
    return 0;  // the grouped launch numbers its tiles itself
}

int qmoe_ragged_mm_device_offsets(const void *X, int x_dtype, const int64_t *expert_offsets_dev, int num_experts,
                                  int max_rows, const uint8_t *W, const uint16_t *scales_f16,
                                  const uint16_t *zero_points_f16, void *Y, int y_dtype, int N, int K, int bits,
                                  int block_size, void *workspace, size_t workspace_bytes, int *status_dev,
                                  qg_stream_t stream) {
    (void)cudaGetLastError();
    if (num_experts < 1 || max_rows < 0 || N < 0 || K < 0) return QG_ERR_INVALID_ARG;
    if (!valid_dtype(x_dtype) || !valid_dtype(y_dtype)) return QG_ERR_INVALID_ARG;
    if (x_dtype == QG_F32 || num_experts > 256) return QG_ERR_UNSUPPORTED;  // the grouped tensor-core launch only
    if (bits != 2 && bits != 4 && bits != 8) return QG_ERR_UNSUPPORTED;
    if (!valid_bs(block_size)) return QG_ERR_UNSUPPORTED;
    if (K % block_size) return QG_ERR_INVALID_ARG;
    if (max_rows > kMaxM || N > kMaxN || K > kMaxK) return QG_ERR_UNSUPPORTED;
    if ((static_cast<long long>(N) * K * bits / 8) % 16 || (static_cast<long long>(N) * (K / block_size) * 2) % 16)
        return QG_ERR_UNSUPPORTED;
    if (!expert_offsets_dev || (reinterpret_cast<uintptr_t>(expert_offsets_dev) & 7u)) return QG_ERR_INVALID_ARG;
    if (max_rows == 0 || N == 0) return QG_OK;
    if (!Y) return QG_ERR_INVALID_ARG;
    if (K == 0) return QG_ERR_UNSUPPORTED;  // no contraction: the rows to zero are not known on the host
    if (!X || !W || !scales_f16) return QG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W) || !aligned16(scales_f16) || (zero_points_f16 && !aligned16(zero_points_f16)))
        return QG_ERR_INVALID_ARG;
    if (!qg::tc_eligible(kRaggedTcRows, K, bits, x_dtype, block_size, qg::WK_NBITS)) return QG_ERR_UNSUPPORTED;
    (void)workspace;  // none needed: kept for the signature
    (void)workspace_bytes;
    GemmProblem p{};
    p.A = X;
    p.a_dtype = x_dtype;
    p.W = W;
    p.kind = qg::WK_NBITS;
    p.scales = scales_f16;
    p.zp = zero_points_f16;
    p.zp_mode = zero_points_f16 ? qg::ZP_TENSOR : qg::ZP_NONE;
    p.uniform_zp = static_cast<float>(1 << (bits - 1));
    p.Y = Y;
    p.y_dtype = y_dtype;
    p.M = max_rows;
    p.N = N;
    p.K = K;
    p.bits = bits;
    p.bs = block_size;
    const cudaError_t e =
        qg::tc_gemm_grouped_dev(p, expert_offsets_dev, num_experts, status_dev, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return QG_ERR_UNSUPPORTED;
    return e == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

int qg_read_device_fault(unsigned int *flags) {
    if (!flags) return QG_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return QG_ERR_CUDA;
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, qg::g_fault_word, sizeof v) != cudaSuccess) return QG_ERR_CUDA;
    if (cudaMemcpyToSymbol(qg::g_fault_word, &zero, sizeof zero) != cudaSuccess) return QG_ERR_CUDA;
    *flags = v;
    return QG_OK;
}

const char *qg_status_string(int status) {
    switch (status) {
    case QG_OK: return "QG_OK";
    case QG_ERR_INVALID_ARG: return "QG_ERR_INVALID_ARG";
    case QG_ERR_UNSUPPORTED: return "QG_ERR_UNSUPPORTED";
    case QG_ERR_CUDA: return "QG_ERR_CUDA";
    case QG_ERR_WORKSPACE_TOO_SMALL: return "QG_ERR_WORKSPACE_TOO_SMALL";
    default: return "QG_ERR_UNKNOWN";
    }
}

}  // extern "C"
