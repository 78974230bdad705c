// qg_internal.h -- host-side declarations shared by the library's translation
// units (not part of the public ABI; see include/qgemm.h for that).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <utility>

namespace qg {

// Launch `kern` as a programmatic dependent of the preceding work on `s`: it
// may begin before the preceding kernel ends, and must itself call
// pdl_wait() before touching anything that kernel may have written.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ZP_PACKED: bits-wide unsigned zero points packed along each row, rows padded
// to whole bytes (the SIMT kernel reads them as staged; no other kernel does).
enum ZpMode { ZP_NONE = 0, ZP_TENSOR = 1, ZP_UNIFORM = 2, ZP_PACKED = 3 };
// WK_DP4A: MatMulNBits codes against int8 activations quantized per block
// (the int8-activation QMoE decode).
enum WeightKind { WK_NBITS = 0, WK_CODEBOOK = 1, WK_DP4A = 2 };

// The library's per-device caches (device attributes, symbol addresses) hold
// kMaxDevices entries.  device_slot() is the current device's index into them,
// or -1 when cudaGetDevice fails or the index is kMaxDevices or more; such a
// device is served without caching (looked up on every call), never through
// another device's entry.  Every entry point works on the current device: its
// stream must belong to that device.
constexpr int kMaxDevices = 64;
int device_slot();

// Per-device facts cached on first use.
struct DeviceInfo {
    int sm_count;
    int max_smem_optin;
};
const DeviceInfo &device_info();

// Address of the device fault word of the current device (see
// qg_read_device_fault).
unsigned *fault_word();

// One blockwise-dequant GEMM/GEMV request, already validated.
struct GemmProblem {
    const void *A;
    int a_dtype;
    const uint8_t *W;
    int kind;                 // WeightKind
    const uint16_t *scales;   // nbits
    const uint16_t *zp;       // nbits, ZP_TENSOR
    const uint8_t *zp_packed = nullptr;  // nbits, ZP_PACKED
    int zp_mode;
    float uniform_zp;         // ZP_UNIFORM (ZP_NONE: midpoint filled in by the caller)
    const float *codebook;    // codebook
    const float *absmax;      // codebook
    void *Y;
    int y_dtype;
    int M, N, K, bits, bs;
    // tensor-core split-precision pass (qg_tc.cu): weight part, accumulate, row scales
    int tc_wpart = 0;
    int tc_acc = 0;
    const float *tc_row_scale = nullptr;
};

// SIMT decode path (small M).
size_t simt_workspace_bytes(int M, int N, int K, int bits, int bs);
cudaError_t simt_gemm(const GemmProblem &p, void *ws, size_t ws_bytes, cudaStream_t s);
// The SIMT kernel has a stage plan for this request with packed zero points.
bool simt_packed_zp_ok(const GemmProblem &p);

// 2-bit MatMulNBits GEMV / small-M GEMM through warp-level MMAs (M <= 4 with
// fp32 activations, M <= 8 with 16-bit ones; block 64, K a multiple of 512).
bool mma_gemv_eligible(const GemmProblem &p);
cudaError_t mma_gemv(const GemmProblem &p, cudaStream_t s);
// The plan mma_gemv takes for a 2-bit block-64 request of this shape: rows per
// tile, consumer warps, CTAs, ring stages; false when the request does not
// take it.
bool mma_gemv_plan(int M, int N, int K, int a_dtype, int zp_mode, int out[4]);

// Tensor-core path (M >= 9 with 16-bit activations).
bool tc_eligible(int M, int K, int bits, int a_dtype, int bs, int kind);
// fp32 activations on the tensor cores by split precision (three fp16 passes:
// A_hi w_hi + A_hi w_lo + A_lo w_hi, per-row power-of-two scaling), when the
// caller's workspace holds split_workspace_bytes(M, K).
constexpr int kSplitMinRows = 16;
size_t split_workspace_bytes(int M, int K);
bool split_eligible(const GemmProblem &p);
cudaError_t split_gemm(const GemmProblem &p, void *ws, size_t ws_bytes, cudaStream_t s);
size_t tc_workspace_bytes(int M, int N, int K, int bits);
cudaError_t tc_gemm(const GemmProblem &p, void *ws, size_t ws_bytes, cudaStream_t s);
// Ragged expert GEMM (grouped tensor-core launch over the experts with at least
// min_rows rows; offsets[0..E] host values).  At most 256 experts.
cudaError_t tc_gemm_grouped(const GemmProblem &p, const int64_t *offsets, int E, int min_rows, cudaStream_t s);
// The grouped launch from device-resident offsets (p.M = the row capacity):
// every CTA numbers the M tiles from the offsets; *status is set to 1 for
// offsets it refuses.
cudaError_t tc_gemm_grouped_dev(const GemmProblem &p, const int64_t *offsets_dev, int E, int *status, cudaStream_t s);

// Fused single-token QMoE decode (fc1 -> SwiGLU -> fc2 -> weighted sum).
struct QmoeProblem {
    const uint16_t *x;
    const int32_t *ids;
    const float *weights;
    int k, num_experts;
    const uint8_t *fc1_w;
    const uint16_t *fc1_scales, *fc1_zp, *fc1_bias;
    const uint8_t *fc2_w;
    const uint16_t *fc2_scales, *fc2_zp, *fc2_bias;
    int hidden, inter, bits, bs, swiglu_interleaved;
    uint16_t *y;
    int *status;
};
size_t qmoe_workspace_bytes(int k, int hidden, int inter);
cudaError_t qmoe_decode(const QmoeProblem &q, void *ws, cudaStream_t s, bool dp4a = false);
// The SIMT kernel serves this int8-activation decode (else qmoe_decode_dp4a).
bool qmoe_dp4a_simt_ok(const QmoeProblem &q);
// Same decode with int8 activations (dp4a); hidden and inter at most 65536.
cudaError_t qmoe_decode_dp4a(const QmoeProblem &q, void *ws, cudaStream_t s);

// Block-quantized embedding gather (validated request).
struct GatherProblem {
    const int64_t *idx;
    long long n;              // number of indices
    const uint8_t *W;         // [V][D * bits / 8]
    int fmt;                  // 0 u2, 1 u4, 2 u8, 3 E4M3 (QG_WF_*)
    const uint16_t *scales;   // [V][D / bs] fp16
    const uint16_t *zp;       // [V][D / bs] fp16 or null (integer formats only)
    long long V;
    int D, bs;
    void *Y;                  // [n][D]
    int y_dtype;
    int *status;              // set to 1 when an index is out of range, or null
};
cudaError_t launch_gather(const GatherProblem &g, cudaStream_t s);

// Utility kernels.
cudaError_t launch_dequant(const GemmProblem &p, float *out, cudaStream_t s);
cudaError_t launch_uniform_check(const uint16_t *t, size_t n, unsigned *ws, cudaStream_t s);
cudaError_t launch_nested_absmax(const uint8_t *qa, const float *table, const float *absmax2, float offset,
                                 int nested, size_t n, float *out, cudaStream_t s);
cudaError_t launch_unpack_zero_points(const uint8_t *zp, int bits, int N, int nb, uint16_t *out, cudaStream_t s);

}  // namespace qg
