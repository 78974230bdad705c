// qg_testing.cu -- a hook for the failure-detection test (include/qgemm_testing.h).
//
// Every pipeline wait of the library's kernels goes through mbar_wait
// (qg_device.cuh): bounded by %globaltimer, it gives up, records a bit in the
// device fault word, raises the CTA's abort flag and returns false.  This
// kernel has the pipeline's shape -- one producer warp, consumer warps that
// wait on a stage's "full" barrier -- with a producer that can be told never
// to fill the stage, and a short bound, so that the give-up path runs on the
// GPU without any fault, trap or endless loop.
#include "../../include/qgemm.h"
#include "../../include/qgemm_testing.h"
#include "qg_device.cuh"
#include "qg_internal.h"

namespace {

constexpr int kConsumerWarps = 3;

__global__ void bounded_wait_kernel(int fill, unsigned long long limit_ns, unsigned *fault, int *out) {
    __shared__ __align__(8) uint64_t full;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        qg::mbar_init(&full, 1);
        abort_flag = 0;
        qg::mbar_fence_init();
    }
    __syncthreads();
    if (warp == 0) {  // producer: fills the stage (one arrival) only when told to
        if (fill && lane == 0) qg::mbar_arrive(&full);
        return;
    }
    const bool ok = qg::mbar_wait(&full, 0, &abort_flag, fault, qg::FAULT_WAIT_FULL, limit_ns);
    if (lane == 0) out[warp - 1] = ok ? 1 : 0;
}

}  // namespace

extern "C" int qg_test_bounded_wait(int fill, unsigned int limit_us, int *out_dev, qg_stream_t stream) {
    (void)cudaGetLastError();
    if (!out_dev || limit_us == 0 || limit_us > 2000000u) return QG_ERR_INVALID_ARG;
    unsigned *fault = qg::fault_word();
    if (!fault) return QG_ERR_CUDA;
    bounded_wait_kernel<<<1, 32 * (1 + kConsumerWarps), 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        fill ? 1 : 0, 1000ull * limit_us, fault, out_dev);
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

extern "C" int qg_test_gemv_plan(int M, int N, int K, int a_dtype, int zp_mode, int *out) {
    if (!out || M < 1 || N < 1 || K < 1) return QG_ERR_INVALID_ARG;
    return qg::mma_gemv_plan(M, N, K, a_dtype, zp_mode, out) ? QG_OK : QG_ERR_UNSUPPORTED;
}
