// minf_sm103.cuh -- inline-PTX wrappers for the Blackwell (sm_103a) features the kernels use:
// mbarriers with bounded waits, TMA tensor copies, proxy fences, named barriers and the
// programmatic-dependent-launch controls.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "minf_common.cuh"

namespace minf {

// Budget of one mbarrier wait.  A wait that runs out sets MINF_ERRBIT_TIMEOUT and tells every
// role of the CTA to stop waiting, so a broken pipeline returns instead of hanging the GPU.
constexpr unsigned long long kWaitBudgetNs = 200ull * 1000 * 1000;

__device__ __forceinline__ uint32_t su32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(unsigned long long *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}

// Ends an mbarrier's use (all its phases complete and no wait pending), so that its word can
// be initialized again.
__device__ __forceinline__ void mbar_inval(unsigned long long *b) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(su32(b)) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tensor cores).
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}

__device__ __forceinline__ bool mbar_try(unsigned long long *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false, without waiting, once
// the CTA is aborting; returns false and starts the abort if the budget runs out.
__device__ __forceinline__ bool mbar_wait(unsigned long long *b, uint32_t parity, volatile int *abort_flag,
                                          int32_t *err) {
    if (mbar_try(b, parity)) return true;
    if (*abort_flag) return false;
    const unsigned long long t0 = gtimer();
    while (true) {
        if (mbar_try(b, parity)) return true;
        if (*abort_flag) return false;
        if (gtimer() - t0 > kWaitBudgetNs) {
            *abort_flag = 1;
            flag_error(err, MINF_ERRBIT_TIMEOUT);
            return false;
        }
    }
}

// Brings a tensor map (a __grid_constant__ kernel parameter) into the TMA unit's descriptor
// cache ahead of its first copy.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}

// The same copy with an evict-first L2 policy: for rows streamed once per step, so that they
// leave L2 before the small operands (q, positions, partials) that other requests wait on.
__device__ __forceinline__ void tma_load_2d_stream(void *dst, const CUtensorMap *map, int x, int y,
                                                   unsigned long long *bar) {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(su32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(su32(bar)), "l"(pol)
        : "memory");
}

// 2-D tensor copy global -> shared, completion counted in bytes on the mbarrier.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(su32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(su32(bar))
        : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier generic-proxy view of global memory (writes it made or acquired
// from other CTAs) before its later async-proxy (bulk copy) reads of it.
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Contiguous global -> shared copy (cp.async.bulk), completion counted in bytes on the
// mbarrier.  Both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, unsigned long long *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(bar))
                 : "memory");
}

// Named barrier over the first `threads` threads of the CTA (barrier 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also returns whether `v` holds in every one of the `threads` threads.
__device__ __forceinline__ bool named_all(int id, int threads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// Programmatic dependent launch: wait for the preceding kernel's completion and memory, and
// allow the following kernel to be scheduled.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void gdc_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void gdc_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// Host: a 2-D tensor map over a row-major [rows, cols] matrix of `dt` elements (elem_bytes
// each) with a {box_cols, box_rows} box.  swizzle128: the 128-byte swizzle the tensor cores
// read (the box's inner extent must then be 128 bytes).
bool make_tensor_map_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint32_t elem_bytes,
                        uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows, bool swizzle128);

}  // namespace minf
