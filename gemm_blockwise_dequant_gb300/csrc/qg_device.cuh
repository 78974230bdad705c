// qg_device.cuh -- device helpers shared by the library's kernels (sm_103a):
// mbarriers with bounded waits, 1-D bulk copies (TMA) global -> shared,
// named barriers, fp16/bf16 conversions and the packed fp32x2 FMA.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace qg {

// Bits recorded in the device fault word when a bounded wait gives up.
enum : unsigned {
    FAULT_WAIT_FULL = 1u,     // consumer waited too long for a stage to land
    FAULT_WAIT_EMPTY = 2u,    // producer waited too long for a stage to be released
    FAULT_WAIT_TC = 4u,       // tensor-core pipeline wait gave up
};

constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// One bounded probe of the phase; a thread whose phase is not complete may
// be suspended for a system-dependent time limit instead of spinning, and
// resumes as soon as the phase completes.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// after limit_ns of %globaltimer (kWaitTimeoutNs unless a caller passes a
// shorter bound), or as soon as another warp of the CTA has given up
// (*abort != 0); on giving up it records `code` in the device fault word,
// raises *abort and returns false.  Never hangs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort, unsigned *fault,
                                          unsigned code, unsigned long long limit_ns = kWaitTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                if (fault) atomicOr(fault, code);
                *abort = 1;
                return false;
            }
        }
    }
}

// 1-D bulk copy (TMA engine) of `bytes` (multiple of 16, both addresses
// 16-byte aligned) from global memory into this CTA's shared memory;
// completion is signalled on `bar` through its transaction count.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// The same copy with an L2 eviction policy (from l2_evict_first()).
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// An L2 policy for data read once (a weight stream larger than L2): its lines
// are evicted first, so the stream leaves the kernels' code and the small
// operands that every launch reads resident in L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

// Copy `bytes` (even) from global to shared memory with the calling warp.
// The 16-byte-aligned bulk part goes through the TMA engine (lane 0 issues
// it; its byte count is returned so the caller can add it to the barrier's
// expected transaction count); the rest is copied by the warp's lanes with
// ordinary loads and stores, finished before this returns (__syncwarp).
// Lane 0 must arrive on `bar` with expect_tx of the returned byte count
// BEFORE the bulk copy is allowed to complete; the caller therefore calls
// this with `issue_bulk` = false first to get the count and the lane copies
// done, arrives, then calls bulk_issue().
struct CopyPlan {
    uint32_t bulk_bytes;  // bytes moved by the TMA engine
};

__device__ __forceinline__ CopyPlan copy_plan(const void *dst, const void *src, uint32_t bytes) {
    CopyPlan p;
    const bool aligned = ((reinterpret_cast<uintptr_t>(src) | static_cast<uintptr_t>(smem_u32(dst))) & 15u) == 0;
    p.bulk_bytes = aligned ? (bytes & ~15u) : 0u;
    return p;
}

// Lane part of a copy: everything past the bulk prefix, in 2-byte units.
__device__ __forceinline__ void copy_tail_lanes(void *dst, const void *src, uint32_t bytes, CopyPlan p, int lane) {
    const uint16_t *s = reinterpret_cast<const uint16_t *>(src);
    uint16_t *d = reinterpret_cast<uint16_t *>(dst);
    for (uint32_t i = p.bulk_bytes / 2 + lane; i < bytes / 2; i += 32) d[i] = __ldg(s + i);
}

// Programmatic dependent launch.  pdl_wait(): block until the preceding
// kernel on the stream has completed and its writes are visible (a no-op when
// the kernel was not launched as a dependent).  pdl_launch_dependents(): let
// the next kernel on the stream begin launching as this one's CTAs retire.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// 2^e as a float for integer e in [-127, 127] (exact).
__device__ __forceinline__ float exp2i(int e) {
    return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Packed fp32x2 fused multiply-add (one instruction, two IEEE fp32 FMAs with
// round-to-nearest; subnormal inputs and results are kept).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rc, rd;\n"
        " mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// Load element i of a row of A given its dtype code (0 f32, 1 f16, 2 bf16).
__device__ __forceinline__ float load_a_elem(const void *A, int dtype, size_t i) {
    if (dtype == 0) return __ldg(reinterpret_cast<const float *>(A) + i);
    const uint16_t v = __ldg(reinterpret_cast<const unsigned short *>(A) + i);
    return dtype == 1 ? h2f(v) : bf2f(v);
}

__device__ __forceinline__ void store_y_elem(void *Y, int dtype, size_t i, float v) {
    if (dtype == 0)
        reinterpret_cast<float *>(Y)[i] = v;
    else if (dtype == 1)
        reinterpret_cast<uint16_t *>(Y)[i] = f2h(v);
    else
        reinterpret_cast<uint16_t *>(Y)[i] = f2bf(v);
}

}  // namespace qg
