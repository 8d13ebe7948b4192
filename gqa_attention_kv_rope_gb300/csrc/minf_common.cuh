// minf_common.cuh -- device helpers shared by the library's kernels (not by the oracle).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/minf.h"

namespace minf {

constexpr int kMaxHalf = 128;  // hd <= 256: the angular-speed table holds hd/2 entries

// The RoPE angular-speed table, passed to kernels by value (512 bytes of kernel
// parameter space), so a captured graph carries it with the launch.
struct RopeTable {
    float f[kMaxHalf];
};

// Fills a RopeTable on the host ("11 . Attention, vec ops, and the KV cache",
// §2.3: freq_i = freq_scale / theta^(2i/hd), evaluated in double, rounded once).
void rope_table(RopeTable *t, int hd, float theta, float freq_scale);

// log2(e): exp(x) = 2^(x * log2 e), the change-of-base identity.
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float4 ldg_stream(const float4 *p) {
    // read-only, do not keep in L1: K/V rows are streamed once per step
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void flag_error(int32_t *err, int bit) {
    if (err) atomicOr(err, bit);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count();

}  // namespace minf
