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

// Packed fp32 pairs (sm_100 and later): two IEEE round-to-nearest operations in one
// instruction, each bit-identical to its scalar form (fmaf, __fadd_rn, __fmul_rn).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
        " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
        " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
        " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float4 cat2(float2 a, float2 b) { return make_float4(a.x, a.y, b.x, b.y); }

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

// The first 256 bytes of every attention workspace are a control block shared by the decode
// and prefill layouts: the prefill step's grid-barrier counts, the decode kernel's unit
// counters, and a tag naming the layout of the last call that used the workspace.  Every call
// that finishes leaves its counters at zero.  A call takes the workspace only when the tag is
// zero (freshly zero-filled) or one its merge tickets can follow (see each kernel); otherwise
// it sets MINF_ERRBIT_WORKSPACE and computes nothing that depends on the workspace.  A call
// whose bounded wait expired leaves the tag at kWsPoison, so the next call refuses it too.
constexpr size_t kWsCtlBytes = 256;
constexpr int kWsBarArrive = 0, kWsBarDepart = 1, kWsUnitCtr = 2, kWsUnitDone = 3, kWsTag = 4;
constexpr int kWsPoison = -1;
constexpr int kWsKindDecode = 1, kWsKindPrefill = 2;

// A layout tag: 'MI' in the high half, a hash of the layout's offsets, the kind in the low bits.
inline int ws_key(int kind, unsigned long long a, unsigned long long b, unsigned long long c,
                  unsigned long long d) {
    unsigned long long h = 1469598103934665603ull;
    for (unsigned long long x : {a, b, c, d}) {
        h ^= x;
        h *= 1099511628211ull;
    }
    const unsigned v = static_cast<unsigned>(h ^ (h >> 29) ^ (h >> 47));
    return static_cast<int>(0x4D490000u | (v & 0xFFFCu) | static_cast<unsigned>(kind));
}
__host__ __device__ __forceinline__ bool ws_key_valid(int t) {
    const unsigned u = static_cast<unsigned>(t);
    return (u & 0xFFFF0000u) == 0x4D490000u && ((u & 3u) == 1u || (u & 3u) == 2u);
}

__device__ __forceinline__ int ld_relaxed(const int *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count();

}  // namespace minf
