// minf_prologue.cuh -- row operations of a layer step's prologue (region stores, the RMSNorm of
// a row, the rotation of a pair), shared by the prologue launch and the fused prefill step.
#pragma once

#include <cuda_fp16.h>

#include "minf_common.cuh"

namespace minf {

// Region elements: fp32 as is, binary16 converted with round to nearest even ("11 . Attention,
// vec ops, and the KV cache", §2.5: the GPU backends may keep the K/V regions in f16).
__device__ __forceinline__ void put1(float *p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void put1(__half *p, size_t i, float v) { p[i] = __float2half_rn(v); }
__device__ __forceinline__ void put4(float *p, size_t i4, float4 v) { reinterpret_cast<float4 *>(p)[i4] = v; }
__device__ __forceinline__ void put4(__half *p, size_t i4, float4 v) {
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&a);
    u.y = *reinterpret_cast<const uint32_t *>(&b);
    reinterpret_cast<uint2 *>(p)[i4] = u;
}

// "11 . Attention, vec ops, and the KV cache", §3.2.1: y = x / sqrt(mean(x^2) + eps) * w for row
// `warp` of x (n values), by one warp; the sum of squares is a per-lane fp32 sum folded by a
// butterfly, and the loops are unrolled so that a lane's loads of a row are in flight together.
// Rows of at most kNormRegF4 * 128 values in float4s: a lane loads all of its float4s of the row
// and of the gain before it uses any, so that they are in flight together and x is read once
// (a store into y could alias a later load, so a loop that stores as it goes issues each load
// only after the previous store).  The same arithmetic in the same order as rms_norm_row.
constexpr int kNormRegF4 = 16;
__device__ __forceinline__ void rms_norm_row_reg(float *y, const float *x, const float *w, int row, int n, float eps) {
    const int lane = threadIdx.x & 31;
    const int n4 = n >> 2;
    const float4 *x4 = reinterpret_cast<const float4 *>(x + static_cast<size_t>(row) * n);
    const float4 *w4 = reinterpret_cast<const float4 *>(w);
    float4 v[kNormRegF4], g[kNormRegF4];
#pragma unroll
    for (int k = 0; k < kNormRegF4; ++k)
        if (lane + 32 * k < n4) {
            v[k] = x4[lane + 32 * k];
            g[k] = w ? w4[lane + 32 * k] : make_float4(1.f, 1.f, 1.f, 1.f);
        }
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < kNormRegF4; ++k)
        if (lane + 32 * k < n4) {
            ss = fmaf(v[k].x, v[k].x, ss);
            ss = fmaf(v[k].y, v[k].y, ss);
            ss = fmaf(v[k].z, v[k].z, ss);
            ss = fmaf(v[k].w, v[k].w, ss);
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float scale = 1.0f / sqrtf(ss / static_cast<float>(n) + eps);
    float4 *y4 = reinterpret_cast<float4 *>(y + static_cast<size_t>(row) * n);
#pragma unroll
    for (int k = 0; k < kNormRegF4; ++k)
        if (lane + 32 * k < n4)
            y4[lane + 32 * k] = make_float4(v[k].x * scale * g[k].x, v[k].y * scale * g[k].y,
                                            v[k].z * scale * g[k].z, v[k].w * scale * g[k].w);
}

template <bool kVec>
__device__ __forceinline__ void rms_norm_row(float *y, const float *x, const float *w, int warp, int n, float eps) {
    if (kVec && n <= kNormRegF4 * 128) {
        rms_norm_row_reg(y, x, w, warp, n, eps);
        return;
    }
    const int lane = threadIdx.x & 31;
    const float *xr = x + static_cast<size_t>(warp) * n;
    float *yr = y + static_cast<size_t>(warp) * n;
    float ss = 0.0f;
    if (kVec) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xr);
#pragma unroll 8
        for (int i = lane; i < n / 4; i += 32) {
            float4 v = x4[i];
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
        }
    } else {
#pragma unroll 8
        for (int i = lane; i < n; i += 32) ss = fmaf(xr[i], xr[i], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float mean = ss / static_cast<float>(n);
    const float scale = 1.0f / sqrtf(mean + eps);
    if (kVec) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xr);
        const float4 *w4 = reinterpret_cast<const float4 *>(w);
        float4 *y4 = reinterpret_cast<float4 *>(yr);
#pragma unroll 8
        for (int i = lane; i < n / 4; i += 32) {
            float4 v = x4[i];
            float4 g = w ? w4[i] : make_float4(1.f, 1.f, 1.f, 1.f);
            y4[i] = make_float4(v.x * scale * g.x, v.y * scale * g.y, v.z * scale * g.z,
                                v.w * scale * g.w);
        }
    } else {
#pragma unroll 8
        for (int i = lane; i < n; i += 32) {
            float v = xr[i] * scale;
            yr[i] = w ? v * w[i] : v;
        }
    }
}

// "11 . Attention, vec ops, and the KV cache", §3.2.2: the pair is rotated by +th with
// th = pos * freq_i in fp32.  Each product is rounded separately (no contraction), so
// the only difference from an exact evaluation is sincosf's own rounding.
__device__ __forceinline__ void rope_pair(float &x0, float &x1, float th) {
    float sn, cs;
    sincosf(th, &sn, &cs);
    const float a = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
    const float b = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs));
    x0 = a;
    x1 = b;
}

// rope_pair with the sine and cosine of th given (the same products and sums, rounded the same).
__device__ __forceinline__ void rope_pair_sc(float &x0, float &x1, float sn, float cs) {
    const float a = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
    const float b = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs));
    x0 = a;
    x1 = b;
}

}  // namespace minf
