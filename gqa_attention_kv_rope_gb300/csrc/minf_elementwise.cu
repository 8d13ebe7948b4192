// minf_elementwise.cu -- RMSNorm, RoPE, the KV store, fused RoPE + KV store, SiLU*mul.
//
// These are memory-bound passes over short rows.  They use 128-bit loads where
// the row width allows and one thread per independent element (or per rotated
// pair), so every launch is a single coalesced sweep over its bytes.
#include <cuda_fp16.h>

#include <cmath>

#include "minf_common.cuh"
#include "minf_kernels.h"
#include "minf_prologue.cuh"
#include "minf_q8.cuh"

namespace minf {

void rope_table(RopeTable *t, int hd, float theta, float freq_scale) {
    // "11 . Attention, vec ops, and the KV cache", §2.3/§3.2.2: the angular speed of
    // subspace i is freq_scale / theta^(2i/hd); exact quotient in double, one rounding.
    const int half = hd / 2;
    for (int i = 0; i < kMaxHalf; ++i) {
        if (i < half) {
            double e = static_cast<double>(2 * i) / static_cast<double>(hd);
            t->f[i] = static_cast<float>(static_cast<double>(freq_scale) /
                                         std::pow(static_cast<double>(theta), e));
        } else {
            t->f[i] = 0.0f;
        }
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

// ----------------------------------------------------------------------------- RMSNorm
// "11 . Attention, vec ops, and the KV cache", §3.2.1: one warp per row (rms_norm_row).
template <bool kVec>
__global__ void __launch_bounds__(256) rms_norm_kernel(float *y, const float *x, const float *w,
                                                       int rows, int n, float eps) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= rows) return;
    rms_norm_row<kVec>(y, x, w, warp, n, eps);
}

// Rows of NV*128 values: a lane holds its NV float4s of the row in registers between the sum of
// squares and the scaling, so x is read once.  Same arithmetic in the same order as
// rms_norm_row (bit-identical results).
template <int NV>
__global__ void __launch_bounds__(256) rms_norm_reg_kernel(float *y, const float *x, const float *w, int rows,
                                                           float eps) {
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    constexpr int n = NV * 128;
    const float4 *x4 = reinterpret_cast<const float4 *>(x + static_cast<size_t>(row) * n);
    float4 v[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) v[k] = x4[lane + 32 * k];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        ss = fmaf(v[k].x, v[k].x, ss);
        ss = fmaf(v[k].y, v[k].y, ss);
        ss = fmaf(v[k].z, v[k].z, ss);
        ss = fmaf(v[k].w, v[k].w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float scale = 1.0f / sqrtf(ss / static_cast<float>(n) + eps);
    const float4 *w4 = reinterpret_cast<const float4 *>(w);
    float4 *y4 = reinterpret_cast<float4 *>(y + static_cast<size_t>(row) * n);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const float4 g = w ? w4[lane + 32 * k] : make_float4(1.f, 1.f, 1.f, 1.f);
        y4[lane + 32 * k] = make_float4(v[k].x * scale * g.x, v[k].y * scale * g.y, v[k].z * scale * g.z,
                                        v[k].w * scale * g.w);
    }
}

template <int NV>
void launch_rms_norm_reg(float *y, const float *x, const float *w, int rows, int n, float eps, int blocks,
                         cudaStream_t s) {
    if constexpr (NV > 1) {
        if (n != NV * 128) return launch_rms_norm_reg<NV - 1>(y, x, w, rows, n, eps, blocks, s);
    }
    rms_norm_reg_kernel<NV><<<blocks, 256, 0, s>>>(y, x, w, rows, eps);
}

int launch_rms_norm(float *y, const float *x, const float *w, int rows, int n, float eps,
                    cudaStream_t s) {
    if (rows == 0) return MINF_OK;
    const bool vec = (n % 4 == 0) && aligned16(x) && aligned16(y) && (!w || aligned16(w));
    const int threads = 256;
    const int blocks = (rows + 7) / 8;
    if (vec && n % 128 == 0 && n <= 16 * 128)
        launch_rms_norm_reg<16>(y, x, w, rows, n, eps, blocks, s);
    else if (vec)
        rms_norm_kernel<true><<<blocks, threads, 0, s>>>(y, x, w, rows, n, eps);
    else
        rms_norm_kernel<false><<<blocks, threads, 0, s>>>(y, x, w, rows, n, eps);
    return cudaPeekAtLastError() == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

// ----------------------------------------------------------------------------- RoPE
// (the rotation of a pair, rope_pair, is in minf_prologue.cuh)
// Rotates pair i of head row `row` (hd floats) in place; f: the angular speeds.
__device__ __forceinline__ void rope_row_pair(float *row, int i, int hd, int style, float p, const float *f) {
    const int half = hd >> 1;
    const int i0 = style == 0 ? i : 2 * i;
    const int i1 = style == 0 ? i + half : 2 * i + 1;
    float x0 = row[i0], x1 = row[i1];
    rope_pair(x0, x1, __fmul_rn(p, f[i]));
    row[i0] = x0;
    row[i1] = x1;
}

// The angular speeds, copied from the launch's table (kernel parameters, which lanes would read
// at different offsets one by one) into shared memory once per block.
__device__ __forceinline__ void table_to_smem(float *dst, const RopeTable &tab, int n) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = tab.f[i];
}

__global__ void __launch_bounds__(256) rope_kernel(float *x, const int32_t *pos, int nt, int nh,
                                                   int hd, int style, const RopeTable tab,
                                                   int32_t *err) {
    const int half = hd >> 1;
    __shared__ float sf[kMaxHalf];
    table_to_smem(sf, tab, half);
    __syncthreads();
    const long long total = static_cast<long long>(nt) * nh * half;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(idx % half);
        const long long th_idx = idx / half;  // t * nh + h
        const int t = static_cast<int>(th_idx / nh);
        const int p = __ldg(pos + t);
        if (p < 0) {
            if (i == 0 && th_idx % nh == 0) flag_error(err, MINF_ERRBIT_ROPE_POS);
            continue;
        }
        rope_row_pair(x + th_idx * hd, i, hd, style, static_cast<float>(p), sf);
    }
}

static int grid_for(long long work, int threads) {
    long long b = (work + threads - 1) / threads;
    const long long cap = static_cast<long long>(sm_count()) * 16;
    if (b > cap) b = cap;
    return static_cast<int>(b < 1 ? 1 : b);
}

int launch_rope(float *x, const int32_t *pos, int nt, int nh, int hd, float theta, float freq_scale,
                int style, int32_t *err, cudaStream_t s) {
    if (nt == 0) return MINF_OK;
    RopeTable tab;
    rope_table(&tab, hd, theta, freq_scale);
    const long long work = static_cast<long long>(nt) * nh * (hd / 2);
    rope_kernel<<<grid_for(work, 256), 256, 0, s>>>(x, pos, nt, nh, hd, style, tab, err);
    return cudaPeekAtLastError() == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

// ----------------------------------------------------------------------------- KV store
// "11 . Attention, vec ops, and the KV cache", §3.2.3: row pos[t] of each region gets the
// token's row, a plain copy; an out-of-range position is reported and never written.
template <typename T>
__global__ void __launch_bounds__(256) kv_append_kernel(T *k_reg, T *v_reg, int cap, int W,
                                                        const float *k_rows, const float *v_rows,
                                                        const int32_t *pos, int nt, int32_t *err) {
    const int w4 = W >> 2;
    const long long total = static_cast<long long>(nt) * w4;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(idx / w4);
        const int c = static_cast<int>(idx % w4);
        const int p = __ldg(pos + t);
        if (p < 0 || p >= cap) {
            if (c == 0) flag_error(err, MINF_ERRBIT_STORE_POS);
            continue;
        }
        const size_t src = static_cast<size_t>(t) * w4 + c;
        const size_t dst = static_cast<size_t>(p) * w4 + c;
        put4(k_reg, dst, reinterpret_cast<const float4 *>(k_rows)[src]);
        put4(v_reg, dst, reinterpret_cast<const float4 *>(v_rows)[src]);
    }
}

int launch_kv_append(void *k_reg, void *v_reg, int kv, int cap, int W, const float *k_rows,
                     const float *v_rows, const int32_t *pos, int nt, int32_t *err,
                     cudaStream_t s) {
    if (nt == 0) return MINF_OK;
    const long long work = static_cast<long long>(nt) * (W / 4);
    if (kv == kKvF16)
        kv_append_kernel<<<grid_for(work, 256), 256, 0, s>>>(static_cast<__half *>(k_reg), static_cast<__half *>(v_reg),
                                                              cap, W, k_rows, v_rows, pos, nt, err);
    else
        kv_append_kernel<<<grid_for(work, 256), 256, 0, s>>>(static_cast<float *>(k_reg), static_cast<float *>(v_reg),
                                                              cap, W, k_rows, v_rows, pos, nt, err);
    return cudaPeekAtLastError() == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

// Q8_0 store: eight consecutive threads quantize one 32-value block (four values each) and
// write its quants and scale.  Token t's row goes to row `row_of(t)` of the region (rb bytes a
// row), or nowhere when that is negative (the error bit was set there).
__device__ __forceinline__ void q8_store4(unsigned char *dst_row, int W, long long rb, int c, float4 x) {
    const unsigned mask = 0xffu << (threadIdx.x & 24u);  // this 8-thread group of the warp
    float d;
    const uint32_t q = quant4(x, mask, d);
    reinterpret_cast<uint32_t *>(dst_row)[c] = q;
    if ((c & 7) == 0) reinterpret_cast<__half *>(dst_row + W)[c >> 3] = __float2half_rn(d);
    if (c == 0)  // the row's zero padding after its scales
        for (long long b = W + W / 16; b < rb; b += 2) *reinterpret_cast<uint16_t *>(dst_row + b) = 0;
}

__global__ void __launch_bounds__(256) kv_append_q8_kernel(unsigned char *k_reg, unsigned char *v_reg, int cap, int W,
                                                           long long rb, const float *k_rows, const float *v_rows,
                                                           const int32_t *pos, int nt, const int64_t *row_off,
                                                           const int32_t *caps, const int32_t *table,
                                                           int max_blocks, int block_rows, int pool_blocks,
                                                           int32_t *err) {
    const int w4 = W >> 2;  // a multiple of 8: blocks never straddle thread groups
    const long long total = static_cast<long long>(nt) * w4;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(idx / w4);
        const int c = static_cast<int>(idx % w4);
        const int p = __ldg(pos + t);
        const int cap_t = table ? max_blocks * block_rows : (caps ? __ldg(caps + t) : cap);
        if (p < 0 || p >= cap_t) {
            if (c == 0) flag_error(err, MINF_ERRBIT_STORE_POS);
            continue;
        }
        long long row = (row_off ? __ldg(row_off + t) : 0) + p;
        if (table) {
            const int b = __ldg(table + static_cast<size_t>(t) * max_blocks + p / block_rows);
            if (b < 0 || b >= pool_blocks) {
                if (c == 0) flag_error(err, MINF_ERRBIT_BLOCK);
                continue;
            }
            row = static_cast<long long>(b) * block_rows + p % block_rows;
        }
        const size_t src = static_cast<size_t>(t) * w4 + c;
        q8_store4(k_reg + row * rb, W, rb, c, reinterpret_cast<const float4 *>(k_rows)[src]);
        q8_store4(v_reg + row * rb, W, rb, c, reinterpret_cast<const float4 *>(v_rows)[src]);
    }
}

int launch_kv_append_q8(void *k_reg, void *v_reg, int cap, int W, const float *k_rows, const float *v_rows,
                        const int32_t *pos, int nt, const int64_t *row_off, const int32_t *caps,
                        const int32_t *table, int max_blocks, int block_rows, int pool_blocks, int32_t *err,
                        cudaStream_t s) {
    if (nt == 0) return MINF_OK;
    const long long work = static_cast<long long>(nt) * (W / 4);
    kv_append_q8_kernel<<<grid_for(work, 256), 256, 0, s>>>(static_cast<unsigned char *>(k_reg),
                                                             static_cast<unsigned char *>(v_reg), cap, W, q8_row_bytes(W),
                                                             k_rows, v_rows, pos, nt, row_off, caps, table, max_blocks,
                                                             block_rows, pool_blocks, err);
    return cudaPeekAtLastError() == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

// One row per sequence through a block table ("IV.2: Zero-copy KV cache": the paged cache
// keeps a sequence as scattered fixed-size blocks).
template <typename T>
__global__ void __launch_bounds__(256) kv_append_paged_kernel(T *k_pool, T *v_pool, int pool_blocks, int block_rows,
                                                              int W, const int32_t *table, int max_blocks,
                                                              const float *k_rows, const float *v_rows,
                                                              const int32_t *pos, int n_seq, int32_t *err) {
    const int w4 = W >> 2;
    const long long total = static_cast<long long>(n_seq) * w4;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int s = static_cast<int>(idx / w4);
        const int c = static_cast<int>(idx % w4);
        const int p = __ldg(pos + s);
        if (p < 0 || p >= max_blocks * block_rows) {
            if (c == 0) flag_error(err, MINF_ERRBIT_STORE_POS);
            continue;
        }
        const int b = __ldg(table + static_cast<size_t>(s) * max_blocks + p / block_rows);
        if (b < 0 || b >= pool_blocks) {
            if (c == 0) flag_error(err, MINF_ERRBIT_BLOCK);
            continue;
        }
        const size_t dst = (static_cast<size_t>(b) * block_rows + p % block_rows) * w4 + c;
        const size_t src = static_cast<size_t>(s) * w4 + c;
        put4(k_pool, dst, reinterpret_cast<const float4 *>(k_rows)[src]);
        put4(v_pool, dst, reinterpret_cast<const float4 *>(v_rows)[src]);
    }
}

int launch_kv_append_paged(void *k_pool, void *v_pool, int kv, int pool_blocks, int block_rows, int W,
                           const int32_t *table, int max_blocks, const float *k_rows, const float *v_rows,
                           const int32_t *pos, int n_seq, int32_t *err, cudaStream_t s) {
    if (n_seq == 0) return MINF_OK;
    const long long work = static_cast<long long>(n_seq) * (W / 4);
    if (kv == kKvF16)
        kv_append_paged_kernel<<<grid_for(work, 256), 256, 0, s>>>(
            static_cast<__half *>(k_pool), static_cast<__half *>(v_pool), pool_blocks, block_rows, W, table,
            max_blocks, k_rows, v_rows, pos, n_seq, err);
    else
        kv_append_paged_kernel<<<grid_for(work, 256), 256, 0, s>>>(
            static_cast<float *>(k_pool), static_cast<float *>(v_pool), pool_blocks, block_rows, W, table,
            max_blocks, k_rows, v_rows, pos, n_seq, err);
    return cudaPeekAtLastError() == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

// ----------------------------------------------------------------------------- RoPE + store
// One sweep per token over three kinds of work item: a q pair, a k pair (rotated, written
// back in place and into the K region), and a float4 of v (copied into the V region).
// Batched callers give each token its own arena offset and capacity.  fq, fk: the angular
// speeds (in shared memory).  Item indices are 32-bit (the host keeps nt * items below 2^31).
template <typename T>
__device__ __forceinline__ void rope_kv_append_items(const RopeKvArgs &a, const float *fq, const float *fk,
                                                     int block, int blocks) {
    const int hq = a.hd >> 1, hk = a.hd_kv >> 1;
    const int nq = a.nh * hq, nkp = a.nk * hk, W = a.nk * a.hd_kv, nv = W >> 2;
    const int per_tok = nq + nkp + nv;
    const int total = a.nt * per_tok;
    for (int idx = block * blockDim.x + threadIdx.x; idx < total; idx += blocks * blockDim.x) {
        const int t = idx / per_tok;
        int r = idx - t * per_tok;
        const int p = __ldg(a.pos + t);
        const int cap_t = a.caps ? __ldg(a.caps + t) : a.cap;
        long long srow = (a.row_off ? __ldg(a.row_off + t) : 0) + p;  // the stored row
        const bool in_range = p >= 0 && p < cap_t;
        const bool storing = a.k_reg != nullptr;  // null: rotate only (another launch stores)
        bool store_ok = in_range && storing;
        if (a.table && in_range) {  // paged: the row's block, through the table
            const int b = __ldg(a.table + static_cast<size_t>(t) * a.max_blocks + p / a.block_rows);
            srow = static_cast<long long>(b) * a.block_rows + p % a.block_rows;
            store_ok = b >= 0 && b < a.pool_blocks;
        }
        if (r < nq) {  // q pair
            if (p < 0) {
                if (r == 0) flag_error(a.err, MINF_ERRBIT_ROPE_POS);
                continue;
            }
            const int h = r / hq, i = r - h * hq;
            rope_row_pair(a.q + (static_cast<size_t>(t) * a.nh + h) * a.hd, i, a.hd, a.style,
                          static_cast<float>(p), fq);
            continue;
        }
        r -= nq;
        if (r < nkp) {  // k pair: rotate, write back, store
            if (p < 0) continue;  // already flagged by the q branch
            const int h = r / hk, i = r - h * hk;
            float *row = a.k + (static_cast<size_t>(t) * a.nk + h) * a.hd_kv;
            const int i0 = a.style == 0 ? i : 2 * i;
            const int i1 = a.style == 0 ? i + hk : 2 * i + 1;
            float x0 = row[i0], x1 = row[i1];
            rope_pair(x0, x1, __fmul_rn(static_cast<float>(p), fk[i]));
            row[i0] = x0;
            row[i1] = x1;
            if (store_ok) {
                T *dst = static_cast<T *>(a.k_reg) + static_cast<size_t>(srow) * W + h * a.hd_kv;
                put1(dst, i0, x0);
                put1(dst, i1, x1);
            }
            continue;
        }
        r -= nkp;  // float4 of v
        if (!storing) continue;
        if (!store_ok) {
            if (r == 0) flag_error(a.err, in_range ? MINF_ERRBIT_BLOCK : MINF_ERRBIT_STORE_POS);
            continue;
        }
        const float4 v = reinterpret_cast<const float4 *>(a.v)[static_cast<size_t>(t) * nv + r];
        put4(static_cast<T *>(a.v_reg), static_cast<size_t>(srow) * nv + r, v);
    }
}

// Work items of a RoPE + store sweep over nt tokens.
inline long long rope_kv_items(const RopeKvArgs &a) {
    return (static_cast<long long>(a.nh) * (a.hd / 2) + a.nk * (a.hd_kv / 2) + a.nk * a.hd_kv / 4) * a.nt;
}

template <typename T>
__global__ void __launch_bounds__(256) rope_kv_append_kernel(RopeKvArgs a, const RopeTable tq,
                                                             const RopeTable tk) {
    __shared__ float fq[kMaxHalf], fk[kMaxHalf];
    table_to_smem(fq, tq, a.hd >> 1);
    table_to_smem(fk, tk, a.hd_kv >> 1);
    __syncthreads();
    rope_kv_append_items<T>(a, fq, fk, blockIdx.x, gridDim.x);
}

// The layer step's prologue in one launch: the first `norm_blocks` blocks compute the
// RMSNorm rows (one warp per row), the rest rotate q and k and store the rows.  It touches
// nothing the attention kernel after it reads before its own dependency wait, so it lets that
// launch start at once (programmatic dependent launch).  It is itself launched early: its
// blocks load the angular-speed tables, then wait for the preceding kernel before they read
// or write anything in memory (positions included).
template <typename T, bool kVec>
__global__ void __launch_bounds__(256) layer_prologue_kernel(RopeKvArgs a, const RopeTable tq, const RopeTable tk,
                                                             NormArgs nrm, int norm_blocks) {
    asm volatile("griddepcontrol.launch_dependents;");
    if (static_cast<int>(blockIdx.x) < norm_blocks) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
        if (warp < nrm.rows) rms_norm_row<kVec>(nrm.y, nrm.x, nrm.w, warp, nrm.n, nrm.eps);
        return;
    }
    __shared__ float fq[kMaxHalf], fk[kMaxHalf];  // norm blocks have returned: block-uniform
    table_to_smem(fq, tq, a.hd >> 1);
    table_to_smem(fk, tk, a.hd_kv >> 1);
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    rope_kv_append_items<T>(a, fq, fk, blockIdx.x - norm_blocks, gridDim.x - norm_blocks);
}

int launch_layer_prologue(const RopeKvArgs &a, float theta, float freq_scale, const NormArgs &nrm, cudaStream_t s) {
    if (a.nt == 0 && nrm.rows == 0) return MINF_OK;
    RopeTable tq, tk;
    rope_table(&tq, a.hd, theta, freq_scale);
    rope_table(&tk, a.hd_kv, theta, freq_scale);
    if (rope_kv_items(a) >= (1ll << 31)) return MINF_ERR_UNSUPPORTED;
    const int norm_blocks = (nrm.rows + 7) / 8;
    const int blocks = norm_blocks + grid_for(rope_kv_items(a), 256);
    const bool vec = (nrm.n % 4 == 0) && aligned16(nrm.x) && aligned16(nrm.y) && (!nrm.w || aligned16(nrm.w));
    // programmatic stream serialization: the blocks may be scheduled before the preceding kernel
    // completes; they wait for it (griddepcontrol.wait) before touching memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (a.kv == kKvF16)
        e = vec ? cudaLaunchKernelEx(&cfg, layer_prologue_kernel<__half, true>, a, tq, tk, nrm, norm_blocks)
                : cudaLaunchKernelEx(&cfg, layer_prologue_kernel<__half, false>, a, tq, tk, nrm, norm_blocks);
    else
        e = vec ? cudaLaunchKernelEx(&cfg, layer_prologue_kernel<float, true>, a, tq, tk, nrm, norm_blocks)
                : cudaLaunchKernelEx(&cfg, layer_prologue_kernel<float, false>, a, tq, tk, nrm, norm_blocks);
    return e == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

int launch_rope_kv_append(const RopeKvArgs &a, float theta, float freq_scale, cudaStream_t s) {
    if (a.nt == 0) return MINF_OK;
    RopeTable tq, tk;
    rope_table(&tq, a.hd, theta, freq_scale);
    rope_table(&tk, a.hd_kv, theta, freq_scale);
    if (rope_kv_items(a) >= (1ll << 31)) return MINF_ERR_UNSUPPORTED;
    const int blocks = grid_for(rope_kv_items(a), 256);
    if (a.kv == kKvF16)
        rope_kv_append_kernel<__half><<<blocks, 256, 0, s>>>(a, tq, tk);
    else
        rope_kv_append_kernel<float><<<blocks, 256, 0, s>>>(a, tq, tk);
    return cudaPeekAtLastError() == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

// ----------------------------------------------------------------------------- SiLU * up
// "11 . Attention, vec ops, and the KV cache", §3.2.5: silu(x) = x / (1 + e^-x).
__device__ __forceinline__ float silu_mul1(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__global__ void __launch_bounds__(256) silu_mul_vec_kernel(float4 *y, const float4 *g,
                                                           const float4 *u, long long n4) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float4 a = g[i], b = u[i];
        y[i] = make_float4(silu_mul1(a.x, b.x), silu_mul1(a.y, b.y), silu_mul1(a.z, b.z),
                           silu_mul1(a.w, b.w));
    }
}

__global__ void __launch_bounds__(256) silu_mul_kernel(float *y, const float *g, const float *u,
                                                       long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        y[i] = silu_mul1(g[i], u[i]);
}

int launch_silu_mul(float *y, const float *g, const float *u, long long n, cudaStream_t s) {
    if (n == 0) return MINF_OK;
    if (n % 4 == 0 && aligned16(y) && aligned16(g) && aligned16(u)) {
        const long long n4 = n / 4;
        const int blocks = grid_for(n4, 256);
        silu_mul_vec_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<float4 *>(y),
                                                   reinterpret_cast<const float4 *>(g),
                                                   reinterpret_cast<const float4 *>(u), n4);
    } else {
        silu_mul_kernel<<<grid_for(n, 256), 256, 0, s>>>(y, g, u, n);
    }
    return cudaPeekAtLastError() == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

}  // namespace minf
