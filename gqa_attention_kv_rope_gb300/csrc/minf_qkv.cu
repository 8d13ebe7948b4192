// minf_qkv.cu -- the fused QKV decode op in one launch.
//
// "13 . The decode loop and graph reuse", §2.3: for a single token a GPU build merges the three
// projection matmuls, their three biases, the two RoPEs and the two KV stores into one op.  Here
// the launch also normalizes its input ("11 . Attention, vec ops, and the KV cache", §3.2.1):
//   xn = RMSNorm(h) * gain
//   y  = W xn + b          W: [n_out, n_embd] rows = nh*hd q outputs, nk*hd_kv k, nk*hd_kv v
//   q, k rotated at pos (§3.2.2); the rotated k and v stored at row pos of the regions (§3.2.3)
// for up to kQkvMaxTok tokens of one sequence.  A warp task is one rotating pair of outputs (or
// two consecutive v outputs) for every token; a CTA of 8 warps takes 8 tasks, and the grid
// covers every task in one wave (two CTAs an SM).  Each warp issues all of its two weight rows'
// 128-bit loads into registers at once, the CTA normalizes every token into shared memory
// meanwhile, and the warp then reduces its rows against all tokens, by butterfly, and its lane
// 0 adds the biases, rotates, writes the outputs and stores k and v.  The weights dominate the
// bytes, so the launch is bound by reading W once.  It is a programmatic dependent launch: the
// weight and bias reads go out before griddepcontrol.wait, so they overlap the end of the
// preceding kernel; everything else (h, gain, pos, all writes) comes after the wait.
#include <cmath>
#include <mutex>

#include "minf_common.cuh"
#include "minf_kernels.h"
#include "minf_sm103.cuh"

namespace minf {

namespace {

constexpr int kWarps = 8;
constexpr int kChunk = 8;                   // float4 of each weight row a lane holds in registers at once
constexpr size_t kQkvMaxSmem = 227 * 1024;  // dynamic shared memory a CTA may have

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

// One warp task: a rotating pair (j0, j1) of q or k outputs, or two consecutive v outputs.
struct Pair {
    int kind;  // 0 q, 1 k, 2 v
    int i;     // rotating pair within its head (q, k)
    int j0, j1;
};

__device__ __forceinline__ Pair pair_of(const QkvArgs &a, int task) {
    const int nq = a.nh * a.hd, W = a.nk * a.hd_kv, pq = nq / 2, pk = W / 2;
    Pair p;
    p.i = 0;
    if (task < pq + pk) {
        const bool is_q = task < pq;
        const int hd = is_q ? a.hd : a.hd_kv, half = hd >> 1, r = is_q ? task : task - pq, h = r / half;
        const int base = (is_q ? 0 : nq) + h * hd;
        p.kind = is_q ? 0 : 1;
        p.i = r % half;
        p.j0 = base + (a.style == 0 ? p.i : 2 * p.i);
        p.j1 = base + (a.style == 0 ? p.i + half : 2 * p.i + 1);
    } else {
        p.kind = 2;
        p.j0 = nq + W + 2 * (task - pq - pk);
        p.j1 = p.j0 + 1;
    }
    return p;
}

// The pair's two biases (weights too: read before the wait).
__device__ __forceinline__ float2 bias_of(const QkvArgs &a, const Pair &p) {
    return a.b ? make_float2(__ldg(a.b + p.j0), __ldg(a.b + p.j1)) : make_float2(0.0f, 0.0f);
}

// Issue the loads of columns [base, base + 32*kChunk) of the pair's two weight rows: all of them
// before any is used, so a warp has 2*kChunk 16-byte loads in flight.
__device__ __forceinline__ void load_chunk(const QkvArgs &a, const Pair &p, int base, int n4, int lane,
                                           float4 (&x0)[kChunk], float4 (&x1)[kChunk]) {
    const float4 *w0 = reinterpret_cast<const float4 *>(a.w + static_cast<size_t>(p.j0) * a.n_embd);
    const float4 *w1 = reinterpret_cast<const float4 *>(a.w + static_cast<size_t>(p.j1) * a.n_embd);
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
        const int c = base + u * 32 + lane;
        if (c < n4) {
            x0[u] = ldg_stream(w0 + c);
            x1[u] = ldg_stream(w1 + c);
        }
    }
}

// RMSNorm of every token by the whole CTA into xs4 [nt][n4] (block 0 also writes xn): thread i
// takes float4 columns i, i + 256, ..; the h and gain loads of all tokens go out together, then
// one reduction through shared memory gives each token its scale.  The positions are read into
// spos beside them.  Ends with __syncthreads.
template <int kT>
__device__ __forceinline__ void norm_tokens(const QkvArgs &a, float4 *xs4, float (&red)[kT][kWarps],
                                            int (&spos)[kT]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x < a.nt) spos[threadIdx.x] = __ldg(a.pos + threadIdx.x);  // beside the h loads
    const int n4 = a.n_embd >> 2;
    const float4 *g4 = reinterpret_cast<const float4 *>(a.gain);
    float ss[kT];
#pragma unroll
    for (int t = 0; t < kT; ++t) {
        ss[t] = 0.0f;
        if (t < a.nt) {
            const float4 *hr = reinterpret_cast<const float4 *>(a.h + static_cast<size_t>(t) * a.n_embd);
            for (int c = threadIdx.x; c < n4; c += kWarps * 32) ss[t] = dot4(hr[c], hr[c], ss[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < kT; ++t) {
        if (t >= a.nt) break;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], o);
        if (lane == 0) red[t][warp] = ss[t];
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < kT; ++t) {
        if (t >= a.nt) break;
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += red[t][w];
        const float scale = 1.0f / sqrtf(sum / static_cast<float>(a.n_embd) + a.eps);
        const float4 *hr = reinterpret_cast<const float4 *>(a.h + static_cast<size_t>(t) * a.n_embd);
        for (int c = threadIdx.x; c < n4; c += kWarps * 32) {
            const float4 v = hr[c];
            const float4 g = g4 ? g4[c] : make_float4(1.f, 1.f, 1.f, 1.f);
            const float4 y = make_float4(v.x * scale * g.x, v.y * scale * g.y, v.z * scale * g.z, v.w * scale * g.w);
            xs4[t * n4 + c] = y;
            if (blockIdx.x == 0) reinterpret_cast<float4 *>(a.xn + static_cast<size_t>(t) * a.n_embd)[c] = y;
        }
    }
    __syncthreads();
}

// Bias, RoPE and stores of one finished task (lane 0 of its warp).
template <int kT>
__device__ __forceinline__ void finish_task(const QkvArgs &a, const RopeTable &tq, const RopeTable &tk,
                                            const Pair &cur, int task, float b0, float b1, const int (&spos)[kT],
                                            const float (&d0)[kT], const float (&d1)[kT]) {
    const int nq = a.nh * a.hd, W = a.nk * a.hd_kv, pq = nq / 2;
    const int j0 = cur.j0, j1 = cur.j1;
#pragma unroll
    for (int t = 0; t < kT; ++t) {
        if (t >= a.nt) break;
        float y0 = d0[t] + b0, y1 = d1[t] + b1;
        const int p = spos[t];
        if (cur.kind < 2) {
            if (p >= 0)
                rot_pair(y0, y1, __fmul_rn(static_cast<float>(p), (cur.kind == 0 ? tq : tk).f[cur.i]));
            else if (task == 0)
                flag_error(a.err, MINF_ERRBIT_ROPE_POS);  // left unrotated
        }
        if (cur.kind == 0) {
            a.q[static_cast<size_t>(t) * nq + j0] = y0;
            a.q[static_cast<size_t>(t) * nq + j1] = y1;
            continue;
        }
        const int off = cur.kind == 1 ? nq : nq + W;
        float *dst = cur.kind == 1 ? a.k : a.v;
        dst[static_cast<size_t>(t) * W + (j0 - off)] = y0;
        dst[static_cast<size_t>(t) * W + (j1 - off)] = y1;
        if (p < 0 || p >= a.cap) {
            if (task == pq) flag_error(a.err, MINF_ERRBIT_STORE_POS);  // not stored
            continue;
        }
        float *reg = cur.kind == 1 ? a.k_reg : a.v_reg;
        reg[static_cast<size_t>(p) * W + (j0 - off)] = y0;
        reg[static_cast<size_t>(p) * W + (j1 - off)] = y1;
    }
}

// kT: the most tokens the instantiation takes (its accumulators live in registers).  Two CTAs
// fit an SM (<= 128 registers a thread): one of this launch and one of the next.
template <int kT>
__global__ void __launch_bounds__(kWarps * 32, 2) fused_qkv_kernel(QkvArgs a, const RopeTable tq, const RopeTable tk) {
    extern __shared__ float4 xs4[];  // [nt][n_embd / 4] normalized inputs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n4 = a.n_embd >> 2;
    const int nq = a.nh * a.hd, W = a.nk * a.hd_kv;
    const int pq = nq / 2, pk = W / 2, n_pairs = pq + 2 * pk;

    gdc_launch_dependents();
    // The first task's weights depend on nothing earlier on the stream: their loads go out
    // before the wait for the preceding kernel and before the norm.
    int task = blockIdx.x * kWarps + warp;
    Pair pr = pair_of(a, task < n_pairs ? task : 0);
    float4 x0[kChunk], x1[kChunk];
    float2 bias = make_float2(0.0f, 0.0f);
    if (task < n_pairs) {
        load_chunk(a, pr, 0, n4, lane, x0, x1);
        if (lane == 0) bias = bias_of(a, pr);
    }
    gdc_wait();

    __shared__ float red[kT][kWarps];
    __shared__ int spos[kT];
    norm_tokens<kT>(a, xs4, red, spos);

    while (task < n_pairs) {
        float d0[kT], d1[kT];
#pragma unroll
        for (int t = 0; t < kT; ++t) d0[t] = d1[t] = 0.0f;
        for (int base = 0; base < n4; base += 32 * kChunk) {
            if (base > 0) load_chunk(a, pr, base, n4, lane, x0, x1);
#pragma unroll
            for (int u = 0; u < kChunk; ++u) {
                const int c = base + u * 32 + lane;
                if (c >= n4) break;
#pragma unroll
                for (int t = 0; t < kT; ++t) {
                    if (t < a.nt) {
                        const float4 xv = xs4[t * n4 + c];
                        d0[t] = dot4(x0[u], xv, d0[t]);
                        d1[t] = dot4(x1[u], xv, d1[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kT; ++t) {
            if (t >= a.nt) break;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                d0[t] += __shfl_xor_sync(0xffffffffu, d0[t], o);
                d1[t] += __shfl_xor_sync(0xffffffffu, d1[t], o);
            }
        }
        const Pair cur = pr;
        const float2 cur_bias = bias;
        const int cur_task = task;
        task += gridDim.x * kWarps;
        if (task < n_pairs) {  // next task's loads go out before this one's epilogue
            pr = pair_of(a, task);
            load_chunk(a, pr, 0, n4, lane, x0, x1);
            if (lane == 0) bias = bias_of(a, pr);
        }
        if (lane == 0) finish_task<kT>(a, tq, tk, cur, cur_task, cur_bias.x, cur_bias.y, spos, d0, d1);
    }
}


}  // namespace

int launch_fused_qkv(const QkvArgs &a, float theta, float freq_scale, cudaStream_t s) {
    if (a.nt == 0) return MINF_OK;
    if (a.nt > kQkvMaxTok) return MINF_ERR_UNSUPPORTED;
    RopeTable tq, tk;
    rope_table(&tq, a.hd, theta, freq_scale);
    rope_table(&tk, a.hd_kv, theta, freq_scale);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MINF_ERR_CUDA;
    const int inst = a.nt == 1 ? 0 : a.nt <= 4 ? 1 : 2;
    void (*const kern)(QkvArgs, RopeTable, RopeTable) =
        inst == 0 ? fused_qkv_kernel<1> : inst == 1 ? fused_qkv_kernel<4> : fused_qkv_kernel<kQkvMaxTok>;
    const size_t smem = static_cast<size_t>(a.nt) * a.n_embd * sizeof(float);
    if (smem > kQkvMaxSmem) return MINF_ERR_UNSUPPORTED;  // the tokens' rows must fit shared memory
    // per device and instantiation, raised (never lowered) to the largest size a call has taken,
    // under a lock so that host threads with different token counts cannot undo one another
    static std::mutex attr_mu;
    static size_t attr_smem[64][3] = {};
    if (smem > 48 * 1024) {
        std::lock_guard<std::mutex> lock(attr_mu);
        if (attr_smem[dev][inst] < smem) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
                cudaSuccess)
                return MINF_ERR_UNSUPPORTED;
            attr_smem[dev][inst] = smem;
        }
    }
    const int pairs = (a.nh * a.hd + 2 * a.nk * a.hd_kv) / 2;
    const int blocks = (pairs + kWarps - 1) / kWarps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, tq, tk) == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

}  // namespace minf
