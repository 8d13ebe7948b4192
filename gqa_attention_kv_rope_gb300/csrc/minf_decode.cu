// minf_decode.cu -- split-KV grouped-query decode attention with an online-softmax merge,
// and the fused single-launch decode layer step built on it.
//
// "11 . Attention, vec ops, and the KV cache", §3.2.4 defines the result (one query per
// sequence attends over rows [0, pos] of its kv head's cached K/V) and §2.5 names the GPU
// shape: split the KV axis across blocks, softmax online, then reduce the splits.
//
// Work decomposition.  A CTA owns (split, kv-head group, sequence): a contiguous run of
// cached rows of one kv head and GH of the g query heads that read it, so every K/V byte
// of the group is fetched from HBM once for all its query heads.  The split count S is
// fixed on the host from the sequence count and max_cap (never from pos) so that one
// launch fills the GPU in a single wave; each launch reads the window length from device
// memory and divides it into at most S equal runs.  The grid therefore never depends on
// pos, and a captured CUDA graph serves every position.
//
// Streaming.  Each of the 8 warps walks 8-row sub-tiles with 128-bit read-only loads that
// bypass L1 (each K/V byte is used once); 8 lanes share a K row for the dot products
// (three butterfly steps), and each lane owns a float4 of the output for the V pass.  A
// warp keeps its own running (max, sum, acc) in the log2 domain; the warps are folded in
// shared memory at the end.
//
// Merge.  A split writes its partial (m, l, acc) to the workspace; the last split of a
// (sequence, kv group) to arrive -- an atomic ticket, no spinning -- folds all partials:
// the (m, l) pairs are staged in shared memory, and the acc loads are spread over every
// thread of the CTA so they are in flight together.  It then resets the ticket.
//
// Fused layer step (kFused).  For one query token per sequence the same launch also does
// the rest of the layer's attention stage: every CTA rotates its q heads in registers
// (RoPE, the same rounding as the standalone kernel), the CTA whose run ends at row pos
// rotates k, writes the K/V row into the region and uses it from shared memory, one extra
// CTA per sequence computes the RMSNorm row, and the last CTA writes the rotated q and k
// back.  Launched with programmatic stream serialization, a layer's launch and its first
// K/V prefetches overlap the previous layer's tail; everything produced by the previous
// kernel is read only after griddepcontrol.wait.
#include <cmath>

#include "minf_common.cuh"
#include "minf_kernels.h"

namespace minf {

namespace {

constexpr int kNW = 8;                  // warps per CTA
constexpr int kThreads = kNW * 32;
constexpr int kSub = 8;                 // rows per warp sub-tile
constexpr int kResident = 152 * 2;      // GB300: 152 SMs x 2 resident 256-thread CTAs
constexpr int kMaxSplit = 64;           // partials per (sequence, kv group)
constexpr int kMaxRows = 512;           // longest run the host aims for (balance across sequences)
constexpr int kMinRows = 64;            // shortest run worth a CTA
constexpr int kPrefetchRows = 32;       // rows per CTA pulled into L2 before the dependency wait

struct WsLayout {
    size_t ml_off, acc_off, ticket_off, total;
};

int choose_splits(int n_seq, int pairs_per_seq, int max_cap) {
    const long long pairs = static_cast<long long>(n_seq) * pairs_per_seq;
    long long s_fill = (kResident + pairs - 1) / pairs;
    long long s_len = (static_cast<long long>(max_cap) + kMaxRows - 1) / kMaxRows;
    long long s_min = (static_cast<long long>(max_cap) + kMinRows - 1) / kMinRows;
    long long s = s_fill > s_len ? s_fill : s_len;
    if (s > s_min) s = s_min;
    if (s > kMaxSplit) s = kMaxSplit;
    if (s < 1) s = 1;
    return static_cast<int>(s);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

WsLayout ws_layout(int n_seq, int nh, int pairs_per_seq, int hd_kv, int splits) {
    WsLayout w;
    const size_t parts = static_cast<size_t>(n_seq) * nh * splits;
    w.ml_off = 0;
    w.acc_off = align256(parts * 2 * sizeof(float));
    w.ticket_off = w.acc_off + align256(parts * hd_kv * sizeof(float));
    w.total = w.ticket_off + align256(static_cast<size_t>(n_seq) * pairs_per_seq * sizeof(int));
    return w;
}

// Query heads of a group handled by one CTA: keep the q slice (GH*hd_kv/8 floats per
// lane) within 64 registers where the group allows it.
int heads_per_cta(int g, int hd_kv) {
    if (g * hd_kv / 8 <= 64) return g;
    if (g % 2 == 0 && (g / 2) * hd_kv / 8 <= 64) return g / 2;
    if (g % 4 == 0) return g / 4;
    return g;
}

struct KParams {
    float *out;
    const float *q, *k_reg, *v_reg;
    const int64_t *row_off;
    const int32_t *caps;
    const int32_t *pos;
    int cap, nh, nk, hd, n_split, groups;  // groups = g / GH
    float scale_log2;
    int32_t *err;
    float *ws_ml, *ws_acc;
    int *ws_ticket;
    // fused layer step only
    float *q_io, *k_io;       // rotated in place (q_io == q)
    const float *v_new;       // [n_seq, W]
    float *xn;                // [n_seq, n_embd]
    const float *h, *gain;
    float eps;
    int n_embd, style;
    RopeTable tab;            // angular speeds for hd (== hd_kv on the fused path)
};

__device__ __forceinline__ float4 f4scale(float4 v, float s) {
    return make_float4(v.x * s, v.y * s, v.z * s, v.w * s);
}

__device__ __forceinline__ void rope_rot(float &x0, float &x1, float sn, float cs) {
    const float a = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
    const float b = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs));
    x0 = a;
    x1 = b;
}

__device__ __forceinline__ float &f4at(float4 &v, int e) {
    return e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
}

// Rotates the KF4 float4s a lane holds (dims 4*sub + 32*i, i < KF4) of one head row of
// width HDKV, with sin/cos precomputed per pair.  Style 0 pairs (i, i + KF4/2) element by
// element; style 1 pairs (x, y) and (z, w) inside each float4.
template <int KF4>
__device__ __forceinline__ void rope_lane(float4 (&x)[KF4], const float (&sn)[2 * KF4],
                                          const float (&cs)[2 * KF4], int style) {
    if (style == 0) {
#pragma unroll
        for (int i = 0; i < KF4 / 2; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                rope_rot(f4at(x[i], e), f4at(x[i + KF4 / 2], e), sn[4 * i + e], cs[4 * i + e]);
    } else {
#pragma unroll
        for (int i = 0; i < KF4; ++i) {
            rope_rot(x[i].x, x[i].y, sn[2 * i], cs[2 * i]);
            rope_rot(x[i].z, x[i].w, sn[2 * i + 1], cs[2 * i + 1]);
        }
    }
}

template <int HDKV, int GH, bool kFused>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const KParams a) {
    constexpr int KF4 = HDKV / 32;    // float4 per lane per K row (8 lanes share a row)
    constexpr int VL = HDKV / 4;      // lanes per V row (a float4 each)
    constexpr int VRP = 32 / VL;      // V rows a warp covers per pass
    constexpr int VJ = kSub / VRP;    // passes per sub-tile
    __shared__ float sm_m[kNW][GH], sm_l[kNW][GH];
    __shared__ float4 sm_acc[kNW][GH][VL];
    __shared__ float sm_pm[GH][kMaxSplit], sm_pl[GH][kMaxSplit];
    __shared__ float sm_M[GH], sm_L[GH];
    __shared__ float4 sm_red[kThreads];
    __shared__ __align__(16) float sm_knew[HDKV], sm_vnew[HDKV];
    __shared__ int sm_last;

    const int s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = a.nk * HDKV;
    const int p = __ldg(a.pos + s);
    const int cap_s = a.caps ? __ldg(a.caps + s) : a.cap;
    const int L = p < 0 ? 0 : (p + 1 < cap_s ? p + 1 : cap_s);
    const long long base = a.row_off ? __ldg(a.row_off + s) : 0;

    if (kFused && blockIdx.x == a.n_split) {
        // The RMSNorm row of this sequence ("11 . Attention, vec ops, and the KV cache",
        // §3.2.1); h is produced upstream, so read it only after the dependency wait.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (blockIdx.y != 0 || warp != 0) return;
        const float *hr = a.h + static_cast<size_t>(s) * a.n_embd;
        float *yr = a.xn + static_cast<size_t>(s) * a.n_embd;
        const int n4 = a.n_embd >> 2;
        float ss = 0.0f;
        for (int i = lane; i < n4; i += 32) {
            const float4 v = reinterpret_cast<const float4 *>(hr)[i];
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float scale = 1.0f / sqrtf(ss / static_cast<float>(a.n_embd) + a.eps);
        for (int i = lane; i < n4; i += 32) {
            const float4 v = reinterpret_cast<const float4 *>(hr)[i];
            const float4 g = a.gain ? reinterpret_cast<const float4 *>(a.gain)[i]
                                    : make_float4(1.f, 1.f, 1.f, 1.f);
            reinterpret_cast<float4 *>(yr)[i] = make_float4(v.x * scale * g.x, v.y * scale * g.y,
                                                            v.z * scale * g.z, v.w * scale * g.w);
        }
        return;
    }

    const int split = blockIdx.x;
    const int hk = blockIdx.y / a.groups;
    const int h0 = hk * (a.nh / a.nk) + (blockIdx.y % a.groups) * GH;  // first query head
    if (split == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        int bits = 0;
        if (p < 0 || p >= cap_s) bits |= MINF_ERRBIT_ATTN_POS;
        if (kFused && (p < 0 || p >= cap_s)) bits |= MINF_ERRBIT_STORE_POS;
        if (kFused && p < 0) bits |= MINF_ERRBIT_ROPE_POS;
        if (bits) flag_error(a.err, bits);
    }
    float *out_s = a.out + (static_cast<size_t>(s) * a.nh + h0) * HDKV;
    if (L == 0) {  // empty window: defined as a zero output
        if (split == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int t = threadIdx.x; t < GH * HDKV; t += blockDim.x) out_s[t] = 0.0f;
        }
        return;
    }
    int T = (L + a.n_split - 1) / a.n_split;
    T = T < kMinRows ? kMinRows : ((T + kSub - 1) / kSub) * kSub;
    const int n_act = (L + T - 1) / T;
    if (split >= n_act) return;
    const int r_begin = split * T;
    const int r_end = r_begin + T < L ? r_begin + T : L;
    const float *Kb = a.k_reg + base * W + hk * HDKV;
    const float *Vb = a.v_reg + base * W + hk * HDKV;

    // Cached rows do not depend on the previous kernel: start pulling the first rows of
    // this run into L2 while that kernel drains.
    if (threadIdx.x < 2 * kPrefetchRows) {
        const int row = r_begin + (threadIdx.x >> 1);
        if (row < r_end) {
            const float *src = ((threadIdx.x & 1) ? Vb : Kb) + static_cast<size_t>(row) * W;
#pragma unroll
            for (int c = 0; c < HDKV * 4; c += 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(src) + c));
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    const int r4 = lane >> 3, sub = lane & 7;
    // this sequence's new row is in this run only on the fused path, when it was stored
    const bool own_new = kFused && p < cap_s && r_end == L;
    const int pnew = own_new ? p : -1;

    float4 qr[GH][KF4];
    float sn[2 * KF4], cs[2 * KF4];
    if (kFused) {
        // angles of the pairs this lane touches (the same for every head and for k)
        // style 0: element e of float4 i < KF4/2 is pair 4*sub + 32*i + e (its partner sits
        // in float4 i + KF4/2); style 1: float4 i holds pairs (4*sub + 32*i)/2 + {0, 1}
        const float pf = static_cast<float>(p);
        if (a.style == 0) {
#pragma unroll
            for (int i = 0; i < KF4 / 2; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    sincosf(__fmul_rn(pf, a.tab.f[4 * sub + 32 * i + e]), &sn[4 * i + e], &cs[4 * i + e]);
        } else {
#pragma unroll
            for (int i = 0; i < KF4; ++i)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    sincosf(__fmul_rn(pf, a.tab.f[(4 * sub + 32 * i) / 2 + e]), &sn[2 * i + e],
                            &cs[2 * i + e]);
        }
    }
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
        const float4 *qh =
            reinterpret_cast<const float4 *>(a.q + (static_cast<size_t>(s) * a.nh + h0 + hh) * a.hd);
#pragma unroll
        for (int i = 0; i < KF4; ++i) qr[hh][i] = qh[sub + 8 * i];
        if (kFused) rope_lane<KF4>(qr[hh], sn, cs, a.style);
    }
    if (own_new && warp == 0 && r4 == 0) {
        // rotate this kv head's k and stage the new K/V row (8 lanes x KF4 float4)
        float4 kx[KF4];
        const float4 *kh =
            reinterpret_cast<const float4 *>(a.k_io + (static_cast<size_t>(s) * a.nk + hk) * HDKV);
        const float4 *vh = reinterpret_cast<const float4 *>(a.v_new + static_cast<size_t>(s) * W + hk * HDKV);
#pragma unroll
        for (int i = 0; i < KF4; ++i) kx[i] = kh[sub + 8 * i];
        rope_lane<KF4>(kx, sn, cs, a.style);
        float4 *kdst = reinterpret_cast<float4 *>(const_cast<float *>(Kb) + static_cast<size_t>(p) * W);
        float4 *vdst = reinterpret_cast<float4 *>(const_cast<float *>(Vb) + static_cast<size_t>(p) * W);
#pragma unroll
        for (int i = 0; i < KF4; ++i) {
            const float4 vx = vh[sub + 8 * i];
            reinterpret_cast<float4 *>(sm_knew)[sub + 8 * i] = kx[i];
            reinterpret_cast<float4 *>(sm_vnew)[sub + 8 * i] = vx;
            kdst[sub + 8 * i] = kx[i];
            vdst[sub + 8 * i] = vx;
        }
    }
    if (kFused) __syncthreads();
    const float sl = a.scale_log2;
    float m[GH], l[GH];
    float4 acc[GH];
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.0f;
        acc[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int vrow = lane / VL, vcol = lane % VL;

    for (int r0 = r_begin + warp * kSub; r0 < r_end; r0 += kNW * kSub) {
        float4 kv[2][KF4];
        float4 vv[VJ];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int row = r0 + 4 * it + r4;
#pragma unroll
            for (int i = 0; i < KF4; ++i) {
                if (row >= r_end)
                    kv[it][i] = make_float4(0.f, 0.f, 0.f, 0.f);
                else if (kFused && row == pnew)
                    kv[it][i] = reinterpret_cast<const float4 *>(sm_knew)[sub + 8 * i];
                else
                    kv[it][i] = ldg_stream(reinterpret_cast<const float4 *>(Kb + static_cast<size_t>(row) * W) +
                                           sub + 8 * i);
            }
        }
#pragma unroll
        for (int j = 0; j < VJ; ++j) {
            const int row = r0 + vrow + VRP * j;
            if (row >= r_end)
                vv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            else if (kFused && row == pnew)
                vv[j] = reinterpret_cast<const float4 *>(sm_vnew)[vcol];
            else
                vv[j] = ldg_stream(reinterpret_cast<const float4 *>(Vb + static_cast<size_t>(row) * W) + vcol);
        }
        float pr[2][GH];
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) {
            float sc[2];
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                float d = 0.0f;
#pragma unroll
                for (int i = 0; i < KF4; ++i) {
                    d = fmaf(qr[hh][i].x, kv[it][i].x, d);
                    d = fmaf(qr[hh][i].y, kv[it][i].y, d);
                    d = fmaf(qr[hh][i].z, kv[it][i].z, d);
                    d = fmaf(qr[hh][i].w, kv[it][i].w, d);
                }
                d += __shfl_xor_sync(0xffffffffu, d, 1);
                d += __shfl_xor_sync(0xffffffffu, d, 2);
                d += __shfl_xor_sync(0xffffffffu, d, 4);
                sc[it] = (r0 + 4 * it + r4) < r_end ? d * sl : -INFINITY;
            }
            float mx = fmaxf(sc[0], sc[1]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m[hh], mx);
            const float corr = ex2_approx(m[hh] - m_new);
            pr[0][hh] = ex2_approx(sc[0] - m_new);
            pr[1][hh] = ex2_approx(sc[1] - m_new);
            float ps = pr[0][hh] + pr[1][hh];
            ps += __shfl_xor_sync(0xffffffffu, ps, 8);
            ps += __shfl_xor_sync(0xffffffffu, ps, 16);
            l[hh] = fmaf(l[hh], corr, ps);
            acc[hh] = f4scale(acc[hh], corr);
            m[hh] = m_new;
        }
#pragma unroll
        for (int j = 0; j < VJ; ++j) {
            const int rl = vrow + VRP * j;  // row within the sub-tile, 0..7
            const int it = (VRP * j) / 4;   // the same for every lane of the pass
            const int src = (rl & 3) * 8;
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) {
                const float w = __shfl_sync(0xffffffffu, it ? pr[1][hh] : pr[0][hh], src);
                acc[hh].x = fmaf(w, vv[j].x, acc[hh].x);
                acc[hh].y = fmaf(w, vv[j].y, acc[hh].y);
                acc[hh].z = fmaf(w, vv[j].z, acc[hh].z);
                acc[hh].w = fmaf(w, vv[j].w, acc[hh].w);
            }
        }
    }
    // Fold the VRP row phases of the warp (they share m), then the warps.
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
#pragma unroll
        for (int o = VL; o < 32; o <<= 1) {
            acc[hh].x += __shfl_xor_sync(0xffffffffu, acc[hh].x, o);
            acc[hh].y += __shfl_xor_sync(0xffffffffu, acc[hh].y, o);
            acc[hh].z += __shfl_xor_sync(0xffffffffu, acc[hh].z, o);
            acc[hh].w += __shfl_xor_sync(0xffffffffu, acc[hh].w, o);
        }
        if (lane < VL) sm_acc[warp][hh][lane] = acc[hh];
        if (lane == 0) {
            sm_m[warp][hh] = m[hh];
            sm_l[warp][hh] = l[hh];
        }
    }
    __syncthreads();

    const size_t part0 = (static_cast<size_t>(s) * a.nh + h0) * a.n_split;  // head h0, split 0
    for (int t = threadIdx.x; t < GH * VL; t += blockDim.x) {
        const int hh = t / VL, c = t % VL;
        float M = sm_m[0][hh];
#pragma unroll
        for (int w = 1; w < kNW; ++w) M = fmaxf(M, sm_m[w][hh]);
        float Ls = 0.0f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
            const float f = ex2_approx(sm_m[w][hh] - M);  // empty warps: m = -inf -> 0
            Ls = fmaf(sm_l[w][hh], f, Ls);
            const float4 x = sm_acc[w][hh][c];
            A.x = fmaf(x.x, f, A.x);
            A.y = fmaf(x.y, f, A.y);
            A.z = fmaf(x.z, f, A.z);
            A.w = fmaf(x.w, f, A.w);
        }
        if (n_act == 1) {
            const float inv = 1.0f / Ls;
            reinterpret_cast<float4 *>(out_s + hh * HDKV)[c] = f4scale(A, inv);
        } else {
            const size_t part = part0 + static_cast<size_t>(hh) * a.n_split + split;
            if (c == 0) {
                a.ws_ml[2 * part] = M;
                a.ws_ml[2 * part + 1] = Ls;
            }
            reinterpret_cast<float4 *>(a.ws_acc + part * HDKV)[c] = A;
        }
    }

    bool last = true;
    int *ticket = a.ws_ticket + static_cast<size_t>(s) * a.nk * a.groups + blockIdx.y;
    if (n_act > 1) {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) sm_last = (atomicAdd(ticket, 1) == n_act - 1);
        __syncthreads();
        last = sm_last;
    }
    if (!last) return;

    if (kFused) {
        // every other run of this group has finished reading q and k: write them back rotated
        if (lane < 8) {
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) {
                if (hh % kNW != warp) continue;
                float4 *qh = reinterpret_cast<float4 *>(a.q_io + (static_cast<size_t>(s) * a.nh + h0 + hh) * a.hd);
#pragma unroll
                for (int i = 0; i < KF4; ++i) qh[lane + 8 * i] = qr[hh][i];
            }
        }
        // k is rotated in place even when its row could not be stored (pos >= cap); the
        // owner of the new row already holds it rotated, any other CTA rotates it again
        // with the same angles and rounding
        if (warp == kNW - 1 && r4 == 0) {
            float4 kx[KF4];
            float4 *kh = reinterpret_cast<float4 *>(a.k_io + (static_cast<size_t>(s) * a.nk + hk) * HDKV);
            if (own_new) {
#pragma unroll
                for (int i = 0; i < KF4; ++i) kx[i] = reinterpret_cast<const float4 *>(sm_knew)[sub + 8 * i];
            } else {
#pragma unroll
                for (int i = 0; i < KF4; ++i) kx[i] = kh[sub + 8 * i];
                rope_lane<KF4>(kx, sn, cs, a.style);
            }
#pragma unroll
            for (int i = 0; i < KF4; ++i) kh[sub + 8 * i] = kx[i];
        }
    }
    if (n_act == 1) return;

    __threadfence();
    // stage the partials' (m, l) and fold them per head
    for (int t = threadIdx.x; t < GH * n_act; t += blockDim.x) {
        const int hh = t / n_act, j = t % n_act;
        const size_t part = part0 + static_cast<size_t>(hh) * a.n_split + j;
        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.ws_ml) + part);
        sm_pm[hh][j] = ml.x;
        sm_pl[hh][j] = ml.y;
    }
    __syncthreads();
    for (int hh = warp; hh < GH; hh += kNW) {
        float M = -INFINITY;
        for (int j = lane; j < n_act; j += 32) M = fmaxf(M, sm_pm[hh][j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float Ls = 0.0f;
        for (int j = lane; j < n_act; j += 32) {
            const float f = ex2_approx(sm_pm[hh][j] - M);
            sm_pm[hh][j] = f;  // becomes the partial's weight
            Ls = fmaf(sm_pl[hh][j], f, Ls);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
        if (lane == 0) {
            sm_M[hh] = M;
            sm_L[hh] = Ls;
        }
    }
    __syncthreads();
    // weighted sum of the acc partials: (head, column) pairs x a slice of the splits each
    constexpr int kPairs = GH * VL;
    constexpr int kWays = kThreads / kPairs > 0 ? kThreads / kPairs : 1;
    for (int t = threadIdx.x; t < kPairs * kWays; t += blockDim.x) {
        const int pair = t % kPairs, way = t / kPairs;
        const int hh = pair / VL, c = pair % VL;
        const size_t ph = part0 + static_cast<size_t>(hh) * a.n_split;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int j = way; j < n_act; j += kWays) {
            const float f = sm_pm[hh][j];
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(a.ws_acc + (ph + j) * HDKV) + c);
            A.x = fmaf(x.x, f, A.x);
            A.y = fmaf(x.y, f, A.y);
            A.z = fmaf(x.z, f, A.z);
            A.w = fmaf(x.w, f, A.w);
        }
        sm_red[way * kPairs + pair] = A;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < kPairs; t += blockDim.x) {
        const int hh = t / VL, c = t % VL;
        float4 A = sm_red[t];
        for (int w = 1; w < kWays; ++w) {
            const float4 x = sm_red[w * kPairs + t];
            A.x += x.x;
            A.y += x.y;
            A.z += x.z;
            A.w += x.w;
        }
        reinterpret_cast<float4 *>(out_s + hh * HDKV)[c] = f4scale(A, 1.0f / sm_L[hh]);
    }
    if (threadIdx.x == 0) *ticket = 0;  // ready for the next call or graph replay
}

template <int HDKV, int GH, bool kFused>
cudaError_t launch_t(const KParams &k, dim3 grid, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_kernel<HDKV, GH, kFused>, k);
}

template <int HDKV, bool kFused>
cudaError_t dispatch_gh(int gh, const KParams &k, dim3 grid, cudaStream_t s, bool pdl) {
    switch (gh) {
        case 1: return launch_t<HDKV, 1, kFused>(k, grid, s, pdl);
        case 2: return launch_t<HDKV, 2, kFused>(k, grid, s, pdl);
        case 3: return launch_t<HDKV, 3, kFused>(k, grid, s, pdl);
        case 4: return launch_t<HDKV, 4, kFused>(k, grid, s, pdl);
        case 5: return launch_t<HDKV, 5, kFused>(k, grid, s, pdl);
        case 6: return launch_t<HDKV, 6, kFused>(k, grid, s, pdl);
        case 7: return launch_t<HDKV, 7, kFused>(k, grid, s, pdl);
        case 8: return launch_t<HDKV, 8, kFused>(k, grid, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

struct Plan {
    int gh, groups, S;
    WsLayout w;
};

Plan plan_for(int n_seq, int nh, int nk, int hd_kv, int max_cap) {
    Plan p;
    const int g = nh / nk;
    p.gh = heads_per_cta(g, hd_kv);
    p.groups = g / p.gh;
    p.S = choose_splits(n_seq, nk * p.groups, max_cap);
    p.w = ws_layout(n_seq, nh, nk * p.groups, hd_kv, p.S);
    return p;
}

int fill(KParams &k, const DecodeArgs &d, const Plan &pl) {
    if (!d.ws || d.ws_bytes < pl.w.total || !aligned16(d.ws)) return MINF_ERR_WORKSPACE;
    char *ws = static_cast<char *>(d.ws);
    k.out = d.out;
    k.q = d.q;
    k.k_reg = d.k_reg;
    k.v_reg = d.v_reg;
    k.row_off = d.row_off;
    k.caps = d.caps;
    k.pos = d.pos;
    k.cap = d.cap;
    k.nh = d.nh;
    k.nk = d.nk;
    k.hd = d.hd;
    k.n_split = pl.S;
    k.groups = pl.groups;
    k.scale_log2 = d.scale * kLog2e;
    k.err = d.err;
    k.ws_ml = reinterpret_cast<float *>(ws + pl.w.ml_off);
    k.ws_acc = reinterpret_cast<float *>(ws + pl.w.acc_off);
    k.ws_ticket = reinterpret_cast<int *>(ws + pl.w.ticket_off);
    k.q_io = nullptr;
    k.k_io = nullptr;
    k.v_new = nullptr;
    k.xn = nullptr;
    k.h = nullptr;
    k.gain = nullptr;
    k.eps = 0.0f;
    k.n_embd = 0;
    k.style = 0;
    return MINF_OK;
}

}  // namespace

bool decode_supported(int nh, int nk, int hd, int hd_kv) {
    if (hd_kv != 64 && hd_kv != 128) return false;
    if (hd % 4 != 0 || hd > 256) return false;
    const int g = nh / nk;
    return g >= 1 && g <= 8;
}

bool fused_step_supported(int nh, int nk, int hd, int hd_kv, int n_embd) {
    if (!decode_supported(nh, nk, hd, hd_kv) || hd != hd_kv || n_embd % 4 != 0) return false;
    const int g = nh / nk;
    return heads_per_cta(g, hd_kv) == g;  // one CTA per kv head owns its k row and q heads
}

size_t decode_workspace_bytes(int n_seq, int nh, int nk, int hd_kv, int max_cap) {
    if (n_seq <= 0 || nh <= 0 || nk <= 0 || hd_kv <= 0 || max_cap <= 0 || nh % nk) return 0;
    return plan_for(n_seq, nh, nk, hd_kv, max_cap).w.total;
}

int launch_decode(const DecodeArgs &d, cudaStream_t s) {
    if (d.n_seq == 0) return MINF_OK;
    if (d.n_seq > 65535) return MINF_ERR_UNSUPPORTED;
    const Plan pl = plan_for(d.n_seq, d.nh, d.nk, d.hd_kv, d.cap);
    KParams k;
    int st = fill(k, d, pl);
    if (st != MINF_OK) return st;
    const dim3 grid(pl.S, d.nk * pl.groups, d.n_seq);
    cudaError_t e = d.hd_kv == 64 ? dispatch_gh<64, false>(pl.gh, k, grid, s, false)
                                  : dispatch_gh<128, false>(pl.gh, k, grid, s, false);
    if (e == cudaErrorInvalidValue) return MINF_ERR_UNSUPPORTED;
    return e == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

int launch_decode_step(const DecodeArgs &d, const DecodeStepExtra &x, cudaStream_t s) {
    if (d.n_seq == 0) return MINF_OK;
    if (d.n_seq > 65535) return MINF_ERR_UNSUPPORTED;
    const Plan pl = plan_for(d.n_seq, d.nh, d.nk, d.hd_kv, d.cap);
    KParams k;
    int st = fill(k, d, pl);
    if (st != MINF_OK) return st;
    k.q_io = const_cast<float *>(d.q);
    k.k_io = x.k;
    k.v_new = x.v;
    k.xn = x.xn;
    k.h = x.h;
    k.gain = x.gain;
    k.eps = x.eps;
    k.n_embd = x.n_embd;
    k.style = x.style;
    rope_table(&k.tab, d.hd_kv, x.theta, x.freq_scale);
    const dim3 grid(pl.S + 1, d.nk * pl.groups, d.n_seq);  // + the RMSNorm CTA per sequence
    cudaError_t e = d.hd_kv == 64 ? dispatch_gh<64, true>(pl.gh, k, grid, s, x.pdl)
                                  : dispatch_gh<128, true>(pl.gh, k, grid, s, x.pdl);
    if (e == cudaErrorInvalidValue) return MINF_ERR_UNSUPPORTED;
    return e == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

}  // namespace minf
