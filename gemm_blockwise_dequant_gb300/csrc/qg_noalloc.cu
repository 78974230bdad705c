// qg_noalloc.cu -- qmoe_decode_fused_noalloc: the fused QMoE decode for
// callers that cannot allocate device memory.
//
// qmoe_decode_fused needs a caller-provided workspace (the fc1 output and the
// per-slot fc2 outputs).  Some callers cannot provide one: a decode loop that
// runs inside a host runtime which owns all device memory and forbids
// allocation on its hot path, an embedded or real-time host that must not
// allocate after start-up, or a plain C caller with no allocator of its own
// (no torch, no caching allocator) that cannot call cudaMalloc at decode
// time.  This entry point takes the same arguments minus the workspace and
// uses a fixed scratch array that lives in this library's device image
// instead.  It computes exactly what qmoe_decode_fused computes, through the
// same kernels.
//
// The scratch array is a file-scope __device__ variable, so every GPU that
// loads the library holds its QG_QMOE_NOALLOC_SCRATCH_BYTES until the process
// exits.  Host code cannot use the array's name as a device address (on the
// host it is only a stand-in symbol); the address is obtained with
// cudaGetSymbolAddress once per device, on that device, by the first call
// made there -- so that first call must come before any stream capture.
// All calls on a device share the one array: calls that may overlap on the
// GPU (different streams without ordering) race and must not be issued.
#include <atomic>

#include "../../include/qgemm.h"
#include "qg_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_qmoe_scratch[QG_QMOE_NOALLOC_SCRATCH_BYTES];

void *g_scratch_ptr[qg::kMaxDevices];
std::atomic<int> g_scratch_ready[qg::kMaxDevices];

// Device address of the current device's scratch array: looked up on the
// first call made on that device and cached per device (the library's common
// device index: a device beyond the cache is looked up on every call).
int scratch_address(void **out) {
    const int slot = qg::device_slot();
    if (slot < 0 || !g_scratch_ready[slot].load(std::memory_order_acquire)) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_qmoe_scratch) != cudaSuccess || p == nullptr) return QG_ERR_CUDA;
        if (slot < 0) {
            *out = p;
            return QG_OK;
        }
        g_scratch_ptr[slot] = p;
        g_scratch_ready[slot].store(1, std::memory_order_release);
    }
    *out = g_scratch_ptr[slot];
    return QG_OK;
}

}  // namespace

extern "C" int qmoe_decode_fused_noalloc(const uint16_t *x_f16, const int32_t *expert_ids,
                                         const float *expert_weights, int k, int num_experts, const uint8_t *fc1_w,
                                         const uint16_t *fc1_scales, const uint16_t *fc1_zp,
                                         const uint16_t *fc1_bias, const uint8_t *fc2_w, const uint16_t *fc2_scales,
                                         const uint16_t *fc2_zp, const uint16_t *fc2_bias, int hidden, int inter,
                                         int bits, int block_size, int swiglu_interleaved, uint16_t *y_f16,
                                         int *status_dev, qg_stream_t stream) {
    // Every byte of the scratch that the kernels read is written earlier in
    // the same call (fc1 writes all of its outputs, invalid slots included,
    // before fc2 reads them; fc2 writes all of its outputs before the combine
    // reads them), so nothing has to start at zero and the contents left by
    // the previous call never matter.
    if (qmoe_decode_workspace_bytes(k, hidden, inter) > QG_QMOE_NOALLOC_SCRATCH_BYTES) {
        (void)cudaGetLastError();
        return QG_ERR_UNSUPPORTED;  // k * (2 * inter + hidden) * 4 bytes do not fit the fixed scratch
    }
    void *ws = nullptr;
    const int st = scratch_address(&ws);
    if (st != QG_OK) return st;
    return qmoe_decode_fused(x_f16, expert_ids, expert_weights, k, num_experts, fc1_w, fc1_scales, fc1_zp, fc1_bias,
                             fc2_w, fc2_scales, fc2_zp, fc2_bias, hidden, inter, bits, block_size, swiglu_interleaved,
                             y_f16, status_dev, ws, QG_QMOE_NOALLOC_SCRATCH_BYTES, stream);
}
