// minf_q8.cuh -- Q8_0 block arithmetic shared by the store, decode and prefill kernels.
//
// "11 . Attention, vec ops, and the KV cache", §2.5: a Q8_0 block is 32 consecutive values of a
// row, kept as one binary16 scale and 32 int8 quants; the store quantizes, the attention read
// dequantizes.  Quantizer (the pages give the format, not the rounding): d = max|x|/127,
// q = round(x * (1/d)) with halves away from zero (d = 0 gives q = 0); a value reads back as
// f16(d) * q, which fp32 holds exactly.  Row layout: the W quants, then the W/32 scales, then
// zero padding to a multiple of 16 bytes.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "minf_common.cuh"

namespace minf {

struct Q8 {};  // storage tag: Q8_0 rows

// Four Q8_0 quants q (4 bytes, element order) as exact floats: each byte is placed in the
// mantissa of 2^23 (offset by 128) and the offset subtracted.
__device__ __forceinline__ float4 int8x4_to_float4(uint32_t q) {
    const uint32_t u = q ^ 0x80808080u;
    const float2 off = make_float2(-8388736.0f, -8388736.0f);
    const float2 ab = add2(make_float2(__int_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                                       __int_as_float(__byte_perm(u, 0x4B000000u, 0x7441))), off);
    const float2 cd = add2(make_float2(__int_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                                       __int_as_float(__byte_perm(u, 0x4B000000u, 0x7443))), off);
    return cat2(ab, cd);
}

// Four Q8_0 values: quants q, block scale s.
__device__ __forceinline__ float4 deq4(uint32_t q, float s) {
    const float4 x = int8x4_to_float4(q);
    const float2 ss = make_float2(s, s);
    return cat2(mul2(lo2(x), ss), mul2(hi2(x), ss));
}

// Quantization of one 32-value block held as four values by each of eight consecutive lanes
// (mask: exactly those lanes).  Returns the four quants packed in element order; d_out = d.
__device__ __forceinline__ uint32_t quant4(float4 x, unsigned mask, float &d_out) {
    float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
    amax = fmaxf(amax, __shfl_xor_sync(mask, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(mask, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(mask, amax, 4));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    const int a = static_cast<int>(roundf(__fmul_rn(x.x, id))), b = static_cast<int>(roundf(__fmul_rn(x.y, id)));
    const int c = static_cast<int>(roundf(__fmul_rn(x.z, id))), e = static_cast<int>(roundf(__fmul_rn(x.w, id)));
    d_out = d;
    return (static_cast<uint32_t>(a) & 0xffu) | ((static_cast<uint32_t>(b) & 0xffu) << 8) |
           ((static_cast<uint32_t>(c) & 0xffu) << 16) | ((static_cast<uint32_t>(e) & 0xffu) << 24);
}

// Elements 4*i4 .. 4*i4+3 of a Q8_0 row (row: its first byte; W: values in the row).
__device__ __forceinline__ float4 ld4_q8(const unsigned char *row, int W, int i4) {
    const uint32_t q = reinterpret_cast<const uint32_t *>(row)[i4];
    const float s = __half2float(reinterpret_cast<const __half *>(row + W)[i4 >> 3]);
    return deq4(q, s);
}

}  // namespace minf
