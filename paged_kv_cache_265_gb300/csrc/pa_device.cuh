// pa_device.cuh -- sm_103a device helpers: mbarriers with bounded waits, bulk
// (TMA engine) global->shared copies, ldmatrix, mma.sync and exp2.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// A bounded wait gives up after this long and raises PA_DEVERR_TIMEOUT; every
// legitimate wait in these kernels ends within microseconds.  Pipeline waits
// take the limit of their launch (pa_set_wait_limit_ns), this by default.
constexpr unsigned int kWaitLimitNs = 2000000000u;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe: never suspends the thread.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// A pipeline wait under a limit shorter than the default (a test setting): polls with the
// non-blocking probe and reads the timer on every turn, so the wait gives up soon after
// `limit_ns` even where a blocking probe would have slept until the phase completed.
static __device__ __noinline__ bool mbar_wait_polled(uint32_t bar, uint32_t parity, int* err, volatile int* abort_flag,
                                              unsigned int limit_ns) {
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_test_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(err, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

// Waits until the phase with the given parity has completed.  Returns false
// (and records PA_DEVERR_TIMEOUT) if that takes longer than the limit or if
// `abort_flag` (shared, may be null) becomes non-zero.  A pipeline wait (one
// given an abort flag) uses `limit_ns`, the launch's setting; a drain wait (no
// abort flag: a CTA waiting for its own copies or products before it exits)
// always uses kWaitLimitNs, so no CTA leaves with work still in flight.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err,
                                          volatile int* abort_flag,
                                          unsigned int limit_ns = kWaitLimitNs) {
    if (abort_flag && limit_ns < kWaitLimitNs) return mbar_wait_polled(bar, parity, err, abort_flag, limit_ns);
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (abort_flag && *abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                atomicOr(err, PA_DEVERR_TIMEOUT);
                if (abort_flag) *abort_flag = 1;
                return false;
            }
        }
    }
}

// L2 policy: the K/V stream is read once per kv head, so it should not evict
// data that is reused (the shared prefix, the block tables, the partials).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy global -> this CTA's shared memory, completion counted in bytes on
// `bar`.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// 16-bit element traits: the mma variant and fp32 <-> storage conversions.
template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kDtype = PA_BF16;
    __device__ __forceinline__ static void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // Packs (lo, hi) into one register, lo in the low half.
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ __forceinline__ static float round_trip(float x) {
        return __bfloat162float(__float2bfloat16_rn(x));
    }
    __device__ __forceinline__ static uint16_t to_bits(float x) {
        __nv_bfloat16 v = __float2bfloat16_rn(x);
        return *reinterpret_cast<uint16_t*>(&v);
    }
};

template <>
struct Elem<__half> {
    static constexpr int kDtype = PA_FP16;
    __device__ __forceinline__ static void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ __forceinline__ static float round_trip(float x) { return __half2float(__float2half_rn(x)); }
    __device__ __forceinline__ static uint16_t to_bits(float x) {
        __half v = __float2half_rn(x);
        return *reinterpret_cast<uint16_t*>(&v);
    }
};

// 2^x on the special-function unit (ex2.approx: relative error about 2^-22).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before its predecessor in the stream has finished;
// griddep_wait() blocks until that predecessor has completed and its memory is
// visible, griddep_launch_dependents() lets the next such kernel start early.
// Both are no-ops for kernels launched the ordinary way.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace pa
