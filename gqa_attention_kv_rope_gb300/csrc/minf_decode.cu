// minf_decode.cu -- split-KV grouped-query decode attention with an online-softmax merge.
//
// "11 . Attention, vec ops, and the KV cache", §3.2.4 defines the result (one query per
// sequence attends over rows [0, pos] of its kv head's cached K/V) and §2.5 names the GPU
// shape: split the KV axis across blocks, softmax online, then reduce the splits.
//
// Work decomposition.  A CTA owns (split, kv-head group, sequence): a contiguous run of
// cached rows of one kv head and GH of the g query heads that read it, so every K/V byte
// of the group is fetched from HBM once for all its query heads.  The split count S is
// fixed on the host from max_cap (never from pos), so one launch shape serves every
// position and the call can be captured in a CUDA graph; each replay reads the window
// length from device memory and divides it into at most S runs.
//
// Inside a CTA each of the 4 warps streams 8-row sub-tiles with 128-bit read-only loads
// (L1 no-allocate: each byte is used once), keeps its own running (max, sum, acc) in the
// log2 domain, and the warps are folded at the end.  A split writes its partial
// (m, l, acc) to the workspace; the last split of a (sequence, kv head) to arrive -- an
// atomic ticket, no spinning -- folds all partials into the output and resets the ticket.
#include <cmath>

#include "minf_common.cuh"
#include "minf_kernels.h"

namespace minf {

namespace {

constexpr int kWarps = 4;
constexpr int kSub = 8;                 // rows per warp sub-tile
constexpr int kMinRows = kWarps * kSub; // a split covers a multiple of 32 rows
constexpr int kFillCtas = 152 * 8;      // GB300: 152 SMs x 8 resident 128-thread CTAs
constexpr int kRowsPerSplit = 256;      // longest split the host aims for

struct WsLayout {
    size_t ml_off, acc_off, ticket_off, total;
};

int choose_splits(int n_seq, int nk_groups, int max_cap) {
    const long long pairs = static_cast<long long>(n_seq) * nk_groups;
    long long s_fill = (kFillCtas + pairs - 1) / pairs;
    long long s_len = (static_cast<long long>(max_cap) + kRowsPerSplit - 1) / kRowsPerSplit;
    long long s_max = (static_cast<long long>(max_cap) + kMinRows - 1) / kMinRows;
    long long s = s_fill > s_len ? s_fill : s_len;
    if (s > s_max) s = s_max;
    if (s < 1) s = 1;
    if (s > 65535) s = 65535;
    return static_cast<int>(s);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

WsLayout ws_layout(int n_seq, int nh, int nk, int hd_kv, int splits) {
    WsLayout w;
    const size_t parts = static_cast<size_t>(n_seq) * nh * splits;
    w.ml_off = 0;
    w.acc_off = align256(parts * 2 * sizeof(float));
    w.ticket_off = w.acc_off + align256(parts * hd_kv * sizeof(float));
    w.total = w.ticket_off + align256(static_cast<size_t>(n_seq) * nk * sizeof(int));
    return w;
}

// Heads of a group handled by one CTA: keep the pre-scaled q slice (GH*hd_kv/8 floats
// per lane) within 64 registers where the group allows it.
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
};

template <int HDKV, int GH>
__global__ void __launch_bounds__(kWarps * 32) decode_split_kernel(const KParams a) {
    constexpr int KF4 = HDKV / 32;    // float4 per lane per K row (8 lanes share a row)
    constexpr int VL = HDKV / 4;      // lanes per V row (a float4 each)
    constexpr int VRP = 32 / VL;      // V rows a warp covers per pass
    constexpr int VJ = kSub / VRP;    // passes per sub-tile
    __shared__ float sm_m[kWarps][GH], sm_l[kWarps][GH];
    __shared__ float4 sm_acc[kWarps][GH][VL];
    __shared__ int sm_last;

    const int split = blockIdx.x;
    const int hk = blockIdx.y / a.groups;
    const int h0 = hk * (a.nh / a.nk) + (blockIdx.y % a.groups) * GH;  // first query head
    const int s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = a.nk * HDKV;

    const int p = __ldg(a.pos + s);
    const int cap_s = a.caps ? __ldg(a.caps + s) : a.cap;
    const int L = p < 0 ? 0 : (p + 1 < cap_s ? p + 1 : cap_s);
    if ((p < 0 || p >= cap_s) && split == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        flag_error(a.err, MINF_ERRBIT_ATTN_POS);
    float *out_s = a.out + (static_cast<size_t>(s) * a.nh + h0) * HDKV;
    if (L == 0) {  // empty window: defined as a zero output
        if (split == 0)
            for (int t = threadIdx.x; t < GH * HDKV; t += blockDim.x) out_s[t] = 0.0f;
        return;
    }
    int T = (L + a.n_split - 1) / a.n_split;
    T = ((T + kMinRows - 1) / kMinRows) * kMinRows;
    const int n_act = (L + T - 1) / T;
    if (split >= n_act) return;
    const int r_begin = split * T;
    const int r_end = r_begin + T < L ? r_begin + T : L;

    const long long base = a.row_off ? __ldg(a.row_off + s) : 0;
    const float *Kb = a.k_reg + base * W + hk * HDKV;
    const float *Vb = a.v_reg + base * W + hk * HDKV;

    const int r4 = lane >> 3, sub = lane & 7;
    float4 qr[GH][KF4];
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
        const float4 *qh =
            reinterpret_cast<const float4 *>(a.q + (static_cast<size_t>(s) * a.nh + h0 + hh) * a.hd);
#pragma unroll
        for (int i = 0; i < KF4; ++i) {
            float4 v = __ldg(qh + sub + 8 * i);
            qr[hh][i] = make_float4(v.x * a.scale_log2, v.y * a.scale_log2, v.z * a.scale_log2,
                                    v.w * a.scale_log2);
        }
    }
    float m[GH], l[GH];
    float4 acc[GH];
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.0f;
        acc[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int vrow = lane / VL, vcol = lane % VL;

    for (int r0 = r_begin + warp * kSub; r0 < r_end; r0 += kWarps * kSub) {
        float4 kv[2][KF4];
        float4 vv[VJ];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int row = r0 + 4 * it + r4;
#pragma unroll
            for (int i = 0; i < KF4; ++i)
                kv[it][i] = row < r_end ? ldg_stream(reinterpret_cast<const float4 *>(
                                              Kb + static_cast<size_t>(row) * W) + sub + 8 * i)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < VJ; ++j) {
            const int row = r0 + vrow + VRP * j;
            vv[j] = row < r_end ? ldg_stream(reinterpret_cast<const float4 *>(
                                      Vb + static_cast<size_t>(row) * W) + vcol)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
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
                sc[it] = (r0 + 4 * it + r4) < r_end ? d : -INFINITY;
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
            acc[hh].x *= corr;
            acc[hh].y *= corr;
            acc[hh].z *= corr;
            acc[hh].w *= corr;
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
        for (int w = 1; w < kWarps; ++w) M = fmaxf(M, sm_m[w][hh]);
        float Ls = 0.0f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
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
            reinterpret_cast<float4 *>(out_s + hh * HDKV)[c] =
                make_float4(A.x * inv, A.y * inv, A.z * inv, A.w * inv);
        } else {
            const size_t part = part0 + static_cast<size_t>(hh) * a.n_split + split;
            if (c == 0) {
                a.ws_ml[2 * part] = M;
                a.ws_ml[2 * part + 1] = Ls;
            }
            reinterpret_cast<float4 *>(a.ws_acc + part * HDKV)[c] = A;
        }
    }
    if (n_act == 1) return;

    __threadfence();
    __syncthreads();
    int *ticket = a.ws_ticket + static_cast<size_t>(s) * a.nk * a.groups + blockIdx.y;
    if (threadIdx.x == 0) sm_last = (atomicAdd(ticket, 1) == n_act - 1);
    __syncthreads();
    if (!sm_last) return;
    __threadfence();
    for (int t = threadIdx.x; t < GH * VL; t += blockDim.x) {
        const int hh = t / VL, c = t % VL;
        const size_t ph = part0 + static_cast<size_t>(hh) * a.n_split;
        float M = -INFINITY;
        for (int j = 0; j < n_act; ++j) M = fmaxf(M, __ldcg(a.ws_ml + 2 * (ph + j)));
        float Ls = 0.0f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < n_act; ++j) {
            const float f = ex2_approx(__ldcg(a.ws_ml + 2 * (ph + j)) - M);
            Ls = fmaf(__ldcg(a.ws_ml + 2 * (ph + j) + 1), f, Ls);
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(a.ws_acc + (ph + j) * HDKV) + c);
            A.x = fmaf(x.x, f, A.x);
            A.y = fmaf(x.y, f, A.y);
            A.z = fmaf(x.z, f, A.z);
            A.w = fmaf(x.w, f, A.w);
        }
        const float inv = 1.0f / Ls;
        reinterpret_cast<float4 *>(out_s + hh * HDKV)[c] =
            make_float4(A.x * inv, A.y * inv, A.z * inv, A.w * inv);
    }
    if (threadIdx.x == 0) *ticket = 0;  // ready for the next call or graph replay
}

template <int HDKV, int GH>
void launch_t(const KParams &k, dim3 grid, cudaStream_t s) {
    decode_split_kernel<HDKV, GH><<<grid, kWarps * 32, 0, s>>>(k);
}

template <int HDKV>
bool dispatch_gh(int gh, const KParams &k, dim3 grid, cudaStream_t s) {
    switch (gh) {
        case 1: launch_t<HDKV, 1>(k, grid, s); return true;
        case 2: launch_t<HDKV, 2>(k, grid, s); return true;
        case 3: launch_t<HDKV, 3>(k, grid, s); return true;
        case 4: launch_t<HDKV, 4>(k, grid, s); return true;
        case 5: launch_t<HDKV, 5>(k, grid, s); return true;
        case 6: launch_t<HDKV, 6>(k, grid, s); return true;
        case 7: launch_t<HDKV, 7>(k, grid, s); return true;
        case 8: launch_t<HDKV, 8>(k, grid, s); return true;
        default: return false;
    }
}

}  // namespace

bool decode_supported(int nh, int nk, int hd, int hd_kv) {
    if (hd_kv != 64 && hd_kv != 128) return false;
    if (hd % 4 != 0 || hd > 256) return false;
    const int g = nh / nk;
    return g >= 1 && g <= 8;
}

size_t decode_workspace_bytes(int n_seq, int nh, int nk, int hd_kv, int max_cap) {
    if (n_seq <= 0 || nh <= 0 || nk <= 0 || hd_kv <= 0 || max_cap <= 0 || nh % nk) return 0;
    const int groups = (nh / nk) / heads_per_cta(nh / nk, hd_kv);
    const int S = choose_splits(n_seq, nk * groups, max_cap);
    return ws_layout(n_seq, nh, nk * groups, hd_kv, S).total;
}

int launch_decode(const DecodeArgs &d, cudaStream_t s) {
    if (d.n_seq == 0) return MINF_OK;
    const int g = d.nh / d.nk;
    const int gh = heads_per_cta(g, d.hd_kv);
    const int groups = g / gh;
    const int S = choose_splits(d.n_seq, d.nk * groups, d.cap);
    const WsLayout w = ws_layout(d.n_seq, d.nh, d.nk * groups, d.hd_kv, S);
    if (!d.ws || d.ws_bytes < w.total || !aligned16(d.ws)) return MINF_ERR_WORKSPACE;
    char *ws = static_cast<char *>(d.ws);
    KParams k;
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
    k.n_split = S;
    k.groups = groups;
    k.scale_log2 = d.scale * kLog2e;
    k.err = d.err;
    k.ws_ml = reinterpret_cast<float *>(ws + w.ml_off);
    k.ws_acc = reinterpret_cast<float *>(ws + w.acc_off);
    k.ws_ticket = reinterpret_cast<int *>(ws + w.ticket_off);
    const dim3 grid(S, d.nk * groups, d.n_seq);
    if (d.n_seq > 65535) return MINF_ERR_UNSUPPORTED;
    bool ok = d.hd_kv == 64 ? dispatch_gh<64>(gh, k, grid, s) : dispatch_gh<128>(gh, k, grid, s);
    if (!ok) return MINF_ERR_UNSUPPORTED;
    return cudaPeekAtLastError() == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

}  // namespace minf
