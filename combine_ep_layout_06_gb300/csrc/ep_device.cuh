// Device-side helpers: cache-hinted 16/8-byte memory ops, release/acquire
// flag ops, a bounded wait and the sticky error word.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ep_internal.cuh"

namespace ep {

#ifndef EP_LD_L2_PREFETCH
#define EP_LD_L2_PREFETCH 0     // 0, 128 or 256: L2 prefetch size on streaming reads
#endif

// Streaming read of data used once (not allocated in L1).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
#if EP_LD_L2_PREFETCH == 256
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#elif EP_LD_L2_PREFETCH == 128
    asm volatile("ld.global.nc.L1::no_allocate.L2::128B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#else
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#endif
    return v;
}

// Streaming (evict-first) stores.
__device__ __forceinline__ void st_stream16(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_stream8(void *p, const uint2 &v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};"
                 :: "l"(p), "r"(v.x), "r"(v.y)
                 : "memory");
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v)
                 : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p,
                                                         uint32_t v) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
                 : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Two-wide fp32 add: each half is the IEEE round-to-nearest scalar add
// (subnormals kept), one instruction for the pair on this SM generation.
// Only for sums of values that no multiply produced: measured on sm_103a
// with CUDA 13.0, a two-wide round-to-nearest multiply feeding a two-wide
// add could come out fused (one rounding), even with contraction disabled,
// so products that must be rounded on their own stay scalar.
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ void set_error(uint32_t *words, uint32_t bit) {
    atomicOr(words + kWordErr, bit);
}

// Spin until *p == want, for at most timeout_ns of %globaltimer and at most
// a fixed number of polls.  Returns false on expiry (the caller records
// EP_DEVERR_TIMEOUT).  Never waits without a bound.
__device__ __forceinline__ bool wait_flag_eq(const uint32_t *p, uint32_t want,
                                             int64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    const uint32_t max_polls = 1u << 24;
    for (uint32_t it = 0;; ++it) {
        if (ld_acquire_gpu(p) == want) return true;
        if (it >= max_polls) return false;
        if ((int64_t)(globaltimer_ns() - t0) > timeout_ns) return false;
        __nanosleep(128);
    }
}

}  // namespace ep
