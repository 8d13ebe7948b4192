// minf_qkv.cu -- the fused QKV decode op in one launch.
//
// "13 . The decode loop and graph reuse", §2.3: for a single token a GPU build merges the three
// projection matmuls, their three biases, the two RoPEs and the two KV stores into one op.  Here
// the launch also normalizes its input ("11 . Attention, vec ops, and the KV cache", §3.2.1):
//   xn = RMSNorm(h) * gain
//   y  = W xn + b          W: [n_out, n_embd] rows = nh*hd q outputs, nk*hd_kv k, nk*hd_kv v
//   q, k rotated at pos (§3.2.2); the rotated k and v stored at row pos of the regions (§3.2.3)
// for up to kQkvMaxTok tokens of one sequence.  Each CTA normalizes every token into shared memory
// (a few KB; block 0 also writes xn out), then each warp produces one rotating pair of outputs
// (or two consecutive v outputs) for every token: it streams the pair's two weight rows once,
// with 128-bit loads, against all tokens' inputs, reduces by butterfly, and its lane 0 adds the
// biases, rotates, writes the outputs and stores k and v.  The weights dominate the bytes, so
// the launch is bound by reading W once.
#include <cmath>

#include "minf_common.cuh"
#include "minf_kernels.h"

namespace minf {

namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void rot_pair(float &x0, float &x1, float th) {
    float sn, cs;
    sincosf(th, &sn, &cs);
    const float a = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
    const float b = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs));
    x0 = a;
    x1 = b;
}

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
    acc = fmaf(a.z, b.z, acc);
    return fmaf(a.w, b.w, acc);
}

__global__ void __launch_bounds__(kWarps * 32) fused_qkv_kernel(QkvArgs a, const RopeTable tq, const RopeTable tk) {
    extern __shared__ float4 xs4[];  // [nt][n_embd / 4] normalized inputs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n4 = a.n_embd >> 2;
    for (int t = warp; t < a.nt; t += kWarps) {
        const float4 *hr = reinterpret_cast<const float4 *>(a.h + static_cast<size_t>(t) * a.n_embd);
        float ss = 0.0f;
        for (int i = lane; i < n4; i += 32) ss = dot4(hr[i], hr[i], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float scale = 1.0f / sqrtf(ss / static_cast<float>(a.n_embd) + a.eps);
        for (int i = lane; i < n4; i += 32) {
            const float4 v = hr[i];
            const float4 g = a.gain ? reinterpret_cast<const float4 *>(a.gain)[i] : make_float4(1.f, 1.f, 1.f, 1.f);
            const float4 y = make_float4(v.x * scale * g.x, v.y * scale * g.y, v.z * scale * g.z, v.w * scale * g.w);
            xs4[t * n4 + i] = y;
            if (blockIdx.x == 0) reinterpret_cast<float4 *>(a.xn + static_cast<size_t>(t) * a.n_embd)[i] = y;
        }
    }
    __syncthreads();

    const int nq = a.nh * a.hd, W = a.nk * a.hd_kv;
    const int pq = nq / 2, pk = W / 2, n_pairs = pq + 2 * pk;
    for (int task = blockIdx.x * kWarps + warp; task < n_pairs; task += gridDim.x * kWarps) {
        int kind, i = 0, j0, j1;  // kind: 0 q, 1 k, 2 v; i: rotating pair within its head
        if (task < pq) {
            kind = 0;
            const int half = a.hd >> 1, h = task / half;
            i = task % half;
            j0 = h * a.hd + (a.style == 0 ? i : 2 * i);
            j1 = h * a.hd + (a.style == 0 ? i + half : 2 * i + 1);
        } else if (task < pq + pk) {
            kind = 1;
            const int half = a.hd_kv >> 1, r = task - pq, h = r / half;
            i = r % half;
            j0 = nq + h * a.hd_kv + (a.style == 0 ? i : 2 * i);
            j1 = nq + h * a.hd_kv + (a.style == 0 ? i + half : 2 * i + 1);
        } else {
            kind = 2;
            j0 = nq + W + 2 * (task - pq - pk);
            j1 = j0 + 1;
        }
        const float4 *w0 = reinterpret_cast<const float4 *>(a.w + static_cast<size_t>(j0) * a.n_embd);
        const float4 *w1 = reinterpret_cast<const float4 *>(a.w + static_cast<size_t>(j1) * a.n_embd);
        float d0[kQkvMaxTok], d1[kQkvMaxTok];
#pragma unroll
        for (int t = 0; t < kQkvMaxTok; ++t) d0[t] = d1[t] = 0.0f;
        for (int c = lane; c < n4; c += 32) {
            const float4 x0 = ldg_stream(w0 + c), x1 = ldg_stream(w1 + c);
#pragma unroll
            for (int t = 0; t < kQkvMaxTok; ++t) {
                if (t < a.nt) {
                    const float4 xv = xs4[t * n4 + c];
                    d0[t] = dot4(x0, xv, d0[t]);
                    d1[t] = dot4(x1, xv, d1[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kQkvMaxTok; ++t) {
            if (t >= a.nt) break;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                d0[t] += __shfl_xor_sync(0xffffffffu, d0[t], o);
                d1[t] += __shfl_xor_sync(0xffffffffu, d1[t], o);
            }
        }
        if (lane != 0) continue;
        const float b0 = a.b ? a.b[j0] : 0.0f, b1 = a.b ? a.b[j1] : 0.0f;
#pragma unroll
        for (int t = 0; t < kQkvMaxTok; ++t) {
            if (t >= a.nt) break;
            float y0 = d0[t] + b0, y1 = d1[t] + b1;
            const int p = __ldg(a.pos + t);
            if (kind < 2) {
                if (p >= 0)
                    rot_pair(y0, y1, __fmul_rn(static_cast<float>(p), (kind == 0 ? tq : tk).f[i]));
                else if (task == 0)
                    flag_error(a.err, MINF_ERRBIT_ROPE_POS);  // left unrotated
            }
            if (kind == 0) {
                a.q[static_cast<size_t>(t) * nq + j0] = y0;
                a.q[static_cast<size_t>(t) * nq + j1] = y1;
                continue;
            }
            const int off = kind == 1 ? nq : nq + W;
            float *dst = kind == 1 ? a.k : a.v;
            dst[static_cast<size_t>(t) * W + (j0 - off)] = y0;
            dst[static_cast<size_t>(t) * W + (j1 - off)] = y1;
            if (p < 0 || p >= a.cap) {
                if (task == pq) flag_error(a.err, MINF_ERRBIT_STORE_POS);  // not stored
                continue;
            }
            float *reg = kind == 1 ? a.k_reg : a.v_reg;
            reg[static_cast<size_t>(p) * W + (j0 - off)] = y0;
            reg[static_cast<size_t>(p) * W + (j1 - off)] = y1;
        }
    }
}

}  // namespace

int launch_fused_qkv(const QkvArgs &a, float theta, float freq_scale, cudaStream_t s) {
    if (a.nt == 0) return MINF_OK;
    if (a.nt > kQkvMaxTok) return MINF_ERR_UNSUPPORTED;
    RopeTable tq, tk;
    rope_table(&tq, a.hd, theta, freq_scale);
    rope_table(&tk, a.hd_kv, theta, freq_scale);
    const size_t smem = static_cast<size_t>(a.nt) * a.n_embd * sizeof(float);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MINF_ERR_CUDA;
    static size_t attr_smem[64] = {};
    if (smem > 48 * 1024 && attr_smem[dev] < smem) {
        if (cudaFuncSetAttribute(fused_qkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return MINF_ERR_UNSUPPORTED;
        attr_smem[dev] = smem;
    }
    const int pairs = (a.nh * a.hd + 2 * a.nk * a.hd_kv) / 2;
    const int blocks = (pairs + kWarps - 1) / kWarps;
    fused_qkv_kernel<<<blocks, kWarps * 32, smem, s>>>(a, tq, tk);
    return cudaPeekAtLastError() == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

}  // namespace minf
