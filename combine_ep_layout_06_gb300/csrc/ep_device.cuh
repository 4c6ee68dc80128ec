// Device-side helpers: cache-hinted 16/8-byte memory ops, release/acquire
// flag ops, a bounded wait and the sticky error word.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ep_internal.cuh"

namespace ep {

// Read of data used once, on the non-coherent read-only path (the data is
// not written while the kernel runs).  Allocating in L1 measured faster
// than L1::no_allocate for every bandwidth-bound gather here (combine of
// 32 768 tokens: 445 against 461 us).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// The same, not allocated in L1: faster for a gather of few tokens
// (2048-token decode combine: 45.5 against 49.6 us), where the kernel is
// latency-bound.
__device__ __forceinline__ uint4 ld_stream16_na(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Streaming (evict-first) stores.
__device__ __forceinline__ void st_stream16(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// Plain (write-back) store: faster than evict-first for the FP8 dispatch's
// code stores (277 against 279 us).
__device__ __forceinline__ void st_plain16(void *p, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
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
// Measured on sm_103a with CUDA 13.0, a two-wide round-to-nearest multiply
// feeding a two-wide add could come out fused (one rounding), even with
// contraction disabled, so products that must be rounded on their own are
// scalar round-to-nearest multiplies; sums of those (the FP8 combine) and
// of plain values use this add, and the parity tests compare every bit.
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Programmatic dependent launch: the dependent grid may start once every CTA
// of this one has signalled; griddepcontrol.wait blocks until the grid it
// depends on has completed and its memory is visible (no-op otherwise).
__device__ __forceinline__ void grid_dependents_may_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
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

// ------------------------------------------------ mbarrier + bulk copies
// Shared-memory mbarriers and the Tensor Memory Accelerator's 1-D bulk
// copies (cp.async.bulk), as the bulk dispatch and the bulk grouping use them.

#ifndef EP_BULK_EVICT_FIRST
#define EP_BULK_EVICT_FIRST 1          // L2 evict-first hints on bulk copies
#endif

__device__ __forceinline__ uint32_t smem_u32(const void *ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded: gives up after timeout_ns of %globaltimer or 2^26 polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          int64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((int64_t)(globaltimer_ns() - t0) > timeout_ns) return false;
    }
    return false;
}
// L2 policy for data touched once: evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// HINT: with the L2 evict-first policy `pol` (the dispatch's rows, touched
// once), else with no cache hint (measured faster for the grouping's copies:
// 990 against 1009 us).
template <bool HINT = true>
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar, uint64_t pol) {
    if constexpr (HINT && EP_BULK_EVICT_FIRST) {
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
                     "[%0], [%1], %2, [%3], %4;"
                     :: "r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
                     : "memory");
    } else {
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                     "[%0], [%1], %2, [%3];"
                     :: "r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                     : "memory");
    }
}
template <bool HINT = true>
__device__ __forceinline__ void bulk_store(void *gdst, const void *smem_src, uint32_t bytes,
                                           uint64_t pol) {
    if constexpr (HINT && EP_BULK_EVICT_FIRST) {
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                     :: "l"(gdst), "r"(smem_u32(smem_src)), "r"(bytes), "l"(pol) : "memory");
    } else {
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                     :: "l"(gdst), "r"(smem_u32(smem_src)), "r"(bytes) : "memory");
    }
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Launch `kernel` programmatically dependent on the kernel before it on the
// stream: its CTAs may be scheduled while that kernel finishes and must call
// grid_dependency_wait() before reading anything it (or earlier work) wrote.
template <typename... Params, typename... Args>
cudaError_t launch_after_previous(void (*kernel)(Params...), unsigned blocks, unsigned threads,
                                  size_t dyn, cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace ep
