// minf_decode.cuh -- split-KV grouped-query decode attention with an online-softmax merge,
// and the fused single-launch decode layer step built on it (the kernel, for fp32 and binary16
// regions; minf_decode.cu plans and launches it, minf_decode_f16.cu instantiates binary16).
//
// "11 . Attention, vec ops, and the KV cache", §3.2.4 defines the result (one query per
// sequence attends over rows [0, pos] of its kv head's cached K/V) and §2.5 names the GPU
// shape: split the KV axis across blocks, softmax online, then reduce the splits.
//
// Work.  A unit is (sequence, kv-head group, split): a contiguous run of cached rows of one
// kv head and the GH query heads of the group that read it, so every K/V byte is fetched
// from HBM once for all those heads.  The split count S is fixed on the host from the
// sequence count and max_cap (never from pos); each launch reads the window length from
// device memory and cuts it into at most S runs of whole pipeline stages.  The grid is
// persistent -- one CTA per SM takes unit blockIdx.x, then further units from a counter in
// the workspace (a batch is ordered longest sequence first) -- so the shape never depends on
// pos and a captured CUDA graph serves every position.
//
// Streaming.  Warp 8 is the producer: one lane issues TMA tensor copies of K and V tiles
// (R rows x hd_kv, 64 KB per stage) into a 3-stage ring of shared memory, running ahead
// across units, gated by per-stage full/empty mbarriers; with each slot it publishes the
// slot's (unit, stage), so the consumers follow the units it drew.  Warps 0-7 consume: each
// takes an 8-row sub-tile of the stage; 8 lanes share a K row for the dot products (three
// butterfly steps) and each lane owns a float4 of the output for the V pass; each warp keeps
// its own running (max, sum, acc) in the log2 domain, folded in shared memory at the end of
// a unit.  The consumer warps synchronise on an mbarrier rather than a named barrier, so
// that, like every other wait here, the wait is bounded.  Warp 9 (the utility warp) zeroes
// the outputs of empty windows and flags out-of-range positions.
//
// Merge.  The run that ends the window (a group's last split, the shortest) is the merger.
// Every other unit stores its partial (m, l, acc) in the workspace, each word encoded so that
// zero means "not yet written", and is done -- no atomic, no wait.  The merger polls those words
// (every consumer thread its share of the splits, all of a chunk's loads in flight together)
// until each is written, folds them in split order, adds its own partial, writes the output and
// zeroes the words it read for the next call.
//
// Fused layer step (kFused).  For one query token per sequence the same launch also does
// the rest of the layer's attention stage: each unit rotates its q heads in registers
// (RoPE, the same rounding as the standalone kernel), the unit whose run ends at row pos
// rotates k, writes it back, appends the K/V row to the region and uses it from shared
// memory, the utility warp computes the RMSNorm rows, and the last unit of a group writes
// the rotated q back.  The loads of q, k and v are issued before anything that waits on the
// position, so a unit's prologue costs one memory round trip.  With programmatic stream
// serialization the producer starts streaming cached rows (which no preceding kernel
// writes) before griddepcontrol.wait; everything the preceding kernel may produce -- q, k,
// v, h, the workspace and its counters, the outputs -- is touched only after it.
#pragma once

#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>

#include "minf_common.cuh"
#include "minf_kernels.h"
#include "minf_q8.cuh"
#include "minf_sm103.cuh"

namespace minf {
namespace dec {

// Consumer warps: 16 (4-row sub-tiles) when a unit's q heads are few enough for their registers,
// else 8 (8-row sub-tiles); either way a 64-row slice of a stage is one sub-tile per warp.  Then
// a producer warp and a utility warp.
template <int NW>
struct Warps {
    static constexpr int kNW = NW;               // consumer warps
    static constexpr int kCons = NW * 32;        // consumer threads
    static constexpr int kProducer = NW;         // TMA producer warp
    static constexpr int kUtility = NW + 1;      // RMSNorm rows, the appended row, empty windows, flags
    static constexpr int kThreads = kCons + 64;  // + producer + utility
    static constexpr int kSub = 64 / NW;         // rows per warp sub-tile
};
// The consumer warp count for a unit of GH q heads of width HDKV.
constexpr int consumer_warps(int gh, int hd_kv) { return (void)gh, (void)hd_kv, 8; }
constexpr int kNST = 3;                 // pipeline stages
constexpr int kPreWait = 2;             // stages a producer issues before the dependency wait
constexpr unsigned kPreWaitGapNs = 500; // between two of them: the previous launch merges meanwhile
constexpr int kStageBytes = 64 * 1024;  // K + V tile of one stage
constexpr int kGridTarget = 152;        // GB300: one persistent CTA per SM
constexpr int kMaxSplit = 64;           // partials per (sequence, kv group)
constexpr int kMaxRows = 4096;          // longest unit when pairs outnumber the SMs
constexpr int kBatchMinRows = 1024;     // shortest unit worth a split when pairs outnumber the SMs
constexpr int kMaxSort = 256;           // batches up to this many sequences are visited longest first

// Rows of the region are stored as fp32 or binary16; the kernel reads and writes them four
// elements at a time and computes in fp32 (the conversion to binary16 rounds to nearest
// even, the conversion back is exact).
__device__ __forceinline__ float4 ld4(const float *p, int i4) { return reinterpret_cast<const float4 *>(p)[i4]; }
__device__ __forceinline__ float4 ld4(const __half *p, int i4) {
    const uint2 u = reinterpret_cast<const uint2 *>(p)[i4];
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st4(float *p, int i4, float4 v) { reinterpret_cast<float4 *>(p)[i4] = v; }
__device__ __forceinline__ void st4(__half *p, int i4, float4 v) {
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&a);
    u.y = *reinterpret_cast<const uint32_t *>(&b);
    reinterpret_cast<uint2 *>(p)[i4] = u;
}

// Q8 (minf_q8.cuh) tags Q8_0 rows: the row's int8 quants, then one binary16 scale per 32
// values, padded to 16 bytes; a value reads back as scale * quant.

template <typename T>
struct Elem {
    static constexpr int bytes = sizeof(T);
    static constexpr bool q8 = false;
};
template <>
struct Elem<Q8> {
    static constexpr int bytes = 1;
    static constexpr bool q8 = true;
};

// A stage holds R rows of K and of V.  For Q8_0 each row also brings a 16-byte slice of its
// scales (those of the 256/HDKV kv heads sharing that slice), and stages are smaller.
template <int HDKV, typename T>
struct Cfg {
    static constexpr bool Q = Elem<T>::q8;
    static constexpr int R = Q ? (HDKV == 64 ? 256 : 128) : kStageBytes / (2 * HDKV * Elem<T>::bytes);
    static constexpr int SPW = R / 64;                            // sub-tiles per warp per stage
    static constexpr int kQBytes = R * HDKV * Elem<T>::bytes;     // values (or quants) of one tensor
    static constexpr int kSBytes = Q ? R * 16 : 0;                // scale slices of one tensor
    static constexpr int kTensorBytes = kQBytes + kSBytes;
    static constexpr int kSlotBytes = 2 * kTensorBytes;          // one ring slot: K then V
};

// Elements 4*i4 .. 4*i4+3 of a tile row: qrow is the row's values (or quants), srow its scale
// slice, sc the index of this kv head's first scale in the slice.
template <int HDKV, typename T>
__device__ __forceinline__ float4 ld_row4(const unsigned char *qrow, const unsigned char *srow, int sc, int i4) {
    if constexpr (Elem<T>::q8) {
        const uint32_t q = reinterpret_cast<const uint32_t *>(qrow)[i4];
        const float scale = __half2float(reinterpret_cast<const __half *>(srow)[sc + (i4 >> 3)]);
        return deq4(q, scale);
    } else {
        return ld4(reinterpret_cast<const T *>(qrow), i4);
    }
}

// The same four elements without the Q8_0 scale (exact integers as floats; the values
// themselves for fp32 and binary16): the kernel applies a block's scale once to a partial sum.
template <int HDKV, typename T>
__device__ __forceinline__ float4 ld_row4_raw(const unsigned char *qrow, int i4) {
    if constexpr (Elem<T>::q8) {
        return int8x4_to_float4(reinterpret_cast<const uint32_t *>(qrow)[i4]);
    } else {
        return ld4(reinterpret_cast<const T *>(qrow), i4);
    }
}

// Q8_0: the scales of this kv head's HDKV/32 blocks in a row's scale slice (srow), as floats,
// in the lane's rotated block order: s[i] is block (i + rot) mod HDKV/32.
template <int HDKV>
__device__ __forceinline__ void ld_scales(const unsigned char *srow, int sc, int rot, float (&s)[HDKV / 32]) {
    if constexpr (HDKV == 128) {
        const uint2 u = *reinterpret_cast<const uint2 *>(srow + 2 * sc);
        // rotate the four halves right by rot places (a 64-bit rotation by 16 * rot bits)
        const uint32_t x = (rot & 2) ? u.y : u.x, y = (rot & 2) ? u.x : u.y;
        const int sh = (rot & 1) * 16;
        const uint32_t lo = __funnelshift_r(x, y, sh), hi = __funnelshift_r(y, x, sh);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
        s[0] = a.x;
        s[1] = a.y;
        s[2] = b.x;
        s[3] = b.y;
    } else {
        uint32_t u = *reinterpret_cast<const uint32_t *>(srow + 2 * sc);
        u = __funnelshift_r(u, u, (rot & 1) * 16);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u));
        s[0] = a.x;
        s[1] = a.y;
    }
}

struct KParams {
    float *out;
    const float *q;
    const int64_t *row_off;
    const int32_t *caps;
    const int32_t *pos;
    int cap, n_seq, nh, nk, hd, n_split, groups;  // groups = g / GH
    int min_rows;          // shortest unit (rows)
    // paged regions (table non-null): logical row j of sequence s is pool row
    // table[s*max_blocks + j/block_rows]*block_rows + j%block_rows; the pool has pool_rows rows;
    // each stage is copied in pieces of box_rows rows (one block, or one stage if blocks are larger)
    const int32_t *table;
    int max_blocks, block_rows, box_rows;
    long long pool_rows;
    long long row_bytes;   // Q8_0: bytes of a region row (quants, scales, padding)
    int sorted;            // visit sequences longest first
    float scale_log2;
    int32_t *err;
    float *ws_ml, *ws_acc;
    int *ws_ticket;        // units of many heads: one merge ticket per (sequence, first q head)
    int *ws_ctr, *ws_done;  // dynamic unit counter and the count of finished producers
    int *ws_tag;           // the workspace's layout tag (its control block)
    int ws_key;            // this call's layout: the tags it accepts are 0 and this one
    int early;             // positions and cached rows are read before the dependency wait
    // fused layer step only
    float *q_io, *k_io;    // rotated in place (q_io == q)
    void *k_reg, *v_reg;   // the new row is written here (the region's storage type)
    const float *v_new;    // [n_seq, W]
    float *xn;             // [n_seq, n_embd]
    const float *h, *gain;
    float eps;
    int n_embd, style;
    RopeTable tab;         // angular speeds for hd (== hd_kv on the fused path)
};

// Requests the 128-byte lines [p, p + bytes) into L2, one line per lane (a hint: the load that
// follows may come after a dependency wait, when the data is current in L2 either way).
__device__ __forceinline__ void prefetch_l2(const void *p, int bytes, int lane) {
    for (int off = lane * 128; off < bytes; off += 32 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char *>(p) + off));
}

// Split partials in the workspace are stored encoded so that an all-zero word means "not yet
// written": the bits of the value, complemented (the one pattern that would encode to zero, a
// NaN with every bit set, is stored as the canonical NaN instead).
__device__ __forceinline__ uint32_t part_enc(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b == 0xFFFFFFFFu ? 0x7FFFFFFFu : b) ^ 0xFFFFFFFFu;
}
__device__ __forceinline__ float part_dec(uint32_t e) { return __uint_as_float(e ^ 0xFFFFFFFFu); }
// Loads that see other CTAs' stores each time they run (no L1, never merged across a poll loop).
__device__ __forceinline__ uint2 ld_relaxed_v2(const uint2 *p) {
    uint2 v;
    asm volatile("ld.relaxed.gpu.global.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint4 ld_relaxed_v4(const uint4 *p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ float4 f4scale(float4 v, float s) {
    const float2 ss = make_float2(s, s);
    return cat2(mul2(lo2(v), ss), mul2(hi2(v), ss));
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
// width HDKV with precomputed sin/cos.  Style 0 pairs float4 i with i + KF4/2 element by
// element (dims d and d + HDKV/2); style 1 pairs (x, y) and (z, w) inside each float4.
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

// Sin and cos of the pair angles a lane needs for rope_lane.  The 4 lanes of a warp with the
// same `sub` (one per r4) need the same 2*KF4 angles, so each computes a quarter of them and
// they are exchanged by shuffles.  Style 0: angle k is pair 4*sub + 32*(k/4) + k%4; style 1:
// pair (4*sub + 32*(k/2))/2 + k%2 (matching rope_lane's indexing).
template <int KF4>
__device__ __forceinline__ void rope_angles(float (&sn)[2 * KF4], float (&cs)[2 * KF4], float pf,
                                            const float *tab, int style, int sub, int r4) {
    constexpr int NA = 2 * KF4;
    constexpr int NQ = NA / 4;
    float ms[NQ], mc[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        const int k = 4 * q + r4;
        const int j = style == 0 ? 4 * sub + 32 * (k >> 2) + (k & 3) : (4 * sub + 32 * (k >> 1)) / 2 + (k & 1);
        sincosf(__fmul_rn(pf, tab[j]), &ms[q], &mc[q]);
    }
#pragma unroll
    for (int k = 0; k < NA; ++k) {
        const int src = (k & 3) * 8 + sub;
        sn[k] = __shfl_sync(0xffffffffu, ms[k >> 2], src);
        cs[k] = __shfl_sync(0xffffffffu, mc[k >> 2], src);
    }
}

// The same angles from shared tables of the sines and cosines of every pair (tsn[i], tcs[i]
// for pair i), indexed as rope_angles indexes its angles.
template <int KF4>
__device__ __forceinline__ void rope_angles_tab(float (&sn)[2 * KF4], float (&cs)[2 * KF4], const float *tsn,
                                                const float *tcs, int style, int sub) {
#pragma unroll
    for (int k = 0; k < 2 * KF4; ++k) {
        const int j = style == 0 ? 4 * sub + 32 * (k >> 2) + (k & 3) : (4 * sub + 32 * (k >> 1)) / 2 + (k & 1);
        sn[k] = tsn[j];
        cs[k] = tcs[j];
    }
}

struct Unit {
    int s, y, j, p, cap_s, L, n_act, r_begin, r_end;
    long long base;
};

// Window of sequence s: rows [0, L) with L = min(pos + 1, cap); empty for a negative position.
__device__ __forceinline__ int window_of(const KParams &a, int s) {
    const int p = __ldg(a.pos + s);
    const int cap_s = a.caps ? __ldg(a.caps + s) : a.cap;
    return p < 0 ? 0 : (p + 1 < cap_s ? p + 1 : cap_s);
}

// The unit u decodes to (sequence, pair, split) and, from the sequence's position, to the
// run of rows it owns.  Units [0, grid) are the CTAs' first units; in a batch, where the units
// outnumber the CTAs, the rest are drawn from the counter, sequences longest first (`order`).
// Within a sequence the pair varies fastest and the split slowest, so the highest CTA indices
// hold the last splits of every pair: the shortest run (the window's ragged end) and the
// splits a short window leaves empty.  The block scheduler places CTAs in index order as SMs
// free up, so those light units land on the SMs that the previous launch left last -- the ones
// whose CTA merged a group -- and a late start there does not delay this launch's merges.
// Split j of a window of L rows covers rows [j*T, (j+1)*T) with T the smallest multiple of the
// stage height (and at least min_rows) that cuts L into at most n_split runs; the n_act
// active splits fill partial slots [0, n_act).  Producer and consumers derive the unit
// identically.
template <int R>
__device__ __forceinline__ Unit unit_of(const KParams &a, int u, const int *order) {
    Unit t;
    const int P = a.nk * a.groups;
    const int w = u % (a.n_split * P);
    t.y = w % P;
    t.j = w / P;
    const int rank = u / (a.n_split * P);
    t.s = order ? order[rank] : rank;
    t.p = __ldg(a.pos + t.s);
    t.cap_s = a.caps ? __ldg(a.caps + t.s) : a.cap;
    t.L = t.p < 0 ? 0 : (t.p + 1 < t.cap_s ? t.p + 1 : t.cap_s);
    int T = (t.L + a.n_split - 1) / a.n_split;
    T = ((T + R - 1) / R) * R;
    if (T < a.min_rows) T = a.min_rows;
    t.n_act = t.L > 0 ? (t.L + T - 1) / T : 0;
    t.r_begin = t.j * T;
    t.r_end = t.j < t.n_act ? (t.r_begin + T < t.L ? t.r_begin + T : t.L) : t.r_begin;
    t.base = a.row_off ? __ldg(a.row_off + t.s) : 0;
    return t;
}

__device__ __forceinline__ bool unit_active(const Unit &t) { return t.r_end > t.r_begin; }

// Barrier of the consumer warps, on an mbarrier so that its wait is bounded like every other
// wait in the kernel (one elected arrival per warp; release/acquire order the shared memory).
__device__ __forceinline__ void cons_sync(unsigned long long *bar, uint32_t &phase, volatile int *abort_flag,
                                          int32_t *err) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    mbar_wait(bar, phase, abort_flag, err);
    phase ^= 1u;
    __syncwarp();
}

// The fused step's new row, by the lanes of one warp with r4 == 0 (sub = lane): rotates k
// (sin/cos from rope_angles) and writes it back, stores the K/V row at pos -- through the
// block table when paged, a missing block flagged -- and stages it in shared memory for the
// tile patch.  pnew < 0: the row is past the region (rotated and written back only).
template <int HDKV, typename T>
__device__ __forceinline__ void append_new_row(const KParams &a, const Unit &t, int hk, int pnew,
                                               const float (&sn)[HDKV / 16], const float (&cs)[HDKV / 16],
                                               int sub, float *sm_knew, float *sm_vnew) {
    constexpr int KF4 = HDKV / 32;
    constexpr bool Q = Elem<T>::q8;
    const int W = a.nk * HDKV;
    float4 *kh = reinterpret_cast<float4 *>(a.k_io + (static_cast<size_t>(t.s) * a.nk + hk) * HDKV);
    const float4 *vh = reinterpret_cast<const float4 *>(a.v_new + static_cast<size_t>(t.s) * W + hk * HDKV);
    float4 kx[KF4], vx[KF4];
#pragma unroll
    for (int i = 0; i < KF4; ++i) {
        kx[i] = kh[sub + 8 * i];
        vx[i] = vh[sub + 8 * i];
    }
    rope_lane<KF4>(kx, sn, cs, a.style);
#pragma unroll
    for (int i = 0; i < KF4; ++i) kh[sub + 8 * i] = kx[i];
    if (pnew >= 0) {
        long long prow = t.base + t.p;
        if (a.table) {  // the row's block, through the table
            const int b = __ldg(a.table + static_cast<size_t>(t.s) * a.max_blocks + t.p / a.block_rows);
            prow = static_cast<long long>(b) * a.block_rows + t.p % a.block_rows;
            if (b < 0 || prow >= a.pool_rows) {
                prow = -1;
                if (sub == 0) flag_error(a.err, MINF_ERRBIT_BLOCK);
            }
        }
        if constexpr (Q) {
            // quantize the row's blocks (block i is element group i of lanes 0-7);
            // staged as bytes (quants, then scales) for the same lanes' patch
            unsigned char *Kg = static_cast<unsigned char *>(a.k_reg) + prow * a.row_bytes;
            unsigned char *Vg = static_cast<unsigned char *>(a.v_reg) + prow * a.row_bytes;
#pragma unroll
            for (int i = 0; i < KF4; ++i) {
                float dk, dv;
                const uint32_t qk = quant4(kx[i], 0xffu, dk), qv = quant4(vx[i], 0xffu, dv);
                reinterpret_cast<uint32_t *>(sm_knew)[sub + 8 * i] = qk;
                reinterpret_cast<uint32_t *>(sm_vnew)[sub + 8 * i] = qv;
                const __half hk16 = __float2half_rn(dk), hv16 = __float2half_rn(dv);
                if (sub == 0) {
                    reinterpret_cast<__half *>(reinterpret_cast<unsigned char *>(sm_knew) + HDKV)[i] = hk16;
                    reinterpret_cast<__half *>(reinterpret_cast<unsigned char *>(sm_vnew) + HDKV)[i] = hv16;
                }
                if (prow >= 0) {
                    reinterpret_cast<uint32_t *>(Kg + hk * HDKV)[sub + 8 * i] = qk;
                    reinterpret_cast<uint32_t *>(Vg + hk * HDKV)[sub + 8 * i] = qv;
                    if (sub == 0) {
                        reinterpret_cast<__half *>(Kg + W)[hk * (HDKV / 32) + i] = hk16;
                        reinterpret_cast<__half *>(Vg + W)[hk * (HDKV / 32) + i] = hv16;
                    }
                }
            }
            if (prow >= 0 && hk == 0 && sub == 0)  // the row's zero padding after its scales
                for (long long b = W + W / 16; b < a.row_bytes; b += 2) {
                    *reinterpret_cast<uint16_t *>(Kg + b) = 0;
                    *reinterpret_cast<uint16_t *>(Vg + b) = 0;
                }
        } else {
#pragma unroll
            for (int i = 0; i < KF4; ++i) {
                // staged for the same lanes, which patch the row's stage when it arrives
                reinterpret_cast<float4 *>(sm_knew)[sub + 8 * i] = kx[i];
                reinterpret_cast<float4 *>(sm_vnew)[sub + 8 * i] = vx[i];
            }
            if (prow >= 0) {
                T *Kg = static_cast<T *>(a.k_reg) + prow * W + hk * HDKV;
                T *Vg = static_cast<T *>(a.v_reg) + prow * W + hk * HDKV;
#pragma unroll
                for (int i = 0; i < KF4; ++i) {
                    st4(Kg, sub + 8 * i, kx[i]);
                    st4(Vg, sub + 8 * i, vx[i]);
                }
            }
        }
    }
}

template <int HDKV, int GH, bool kFused, typename T, int NW = consumer_warps(GH, HDKV)>
__global__ void __launch_bounds__(Warps<NW>::kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmKs, const __grid_constant__ CUtensorMap tmVs,
                  const KParams a) {
    using C = Cfg<HDKV, T>;
    constexpr int kNW = Warps<NW>::kNW, kCons = Warps<NW>::kCons, kSub = Warps<NW>::kSub;
    constexpr int kProducer = Warps<NW>::kProducer, kUtility = Warps<NW>::kUtility;
    constexpr int KP = kSub / 4;  // K passes of four rows per sub-tile
    constexpr bool Q = C::Q;
    constexpr int R = C::R, SPW = C::SPW;
    constexpr int EB = Elem<T>::bytes;
    constexpr int kScaleHeads = 256 / HDKV;  // Q8_0: kv heads whose scales share a 16-byte slice
    constexpr int KF4 = HDKV / 32;  // float4 per lane per K row (8 lanes share a row)
    constexpr int VL = HDKV / 4;    // lanes per V row (a float4 each)
    constexpr int VRP = 32 / VL;    // V rows a warp covers per pass
    constexpr int VJ = kSub / VRP;  // passes per sub-tile
    constexpr int NACC = GH <= 2 ? 2 : 1;  // V accumulator sets a lane keeps per head
    // sub-tiles whose rows share one online-softmax update (their scores are held at once)
    constexpr int GRP = GH <= 2 ? SPW : (GH <= 4 ? (SPW < 2 ? SPW : 2) : 1);
    static_assert(SPW % GRP == 0, "sub-tile groups");

    extern __shared__ unsigned char smem_raw[];
    // 1024-aligned ring, derived from the shared array itself so loads stay in the shared space
    unsigned char *ring = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
    __shared__ unsigned long long full[kNST], empty[kNST], meta_full[kNST], cons_bar, knew_bar;
    __shared__ int2 sm_meta[kNST];  // (unit, stage) of each ring slot; unit < 0 ends the stream
    __shared__ int sm_order[kMaxSort];
    __shared__ float sm_m[kNW][GH], sm_l[kNW][GH];
    __shared__ float4 sm_acc[kNW][GH][VL];
    __shared__ float4 sm_red[kCons];
    __shared__ float sm_redM[kCons], sm_redL[kCons];
    __shared__ __align__(16) float sm_knew[HDKV], sm_vnew[HDKV];
    __shared__ int sm_abort, sm_wsbad, sm_last;
    __shared__ float sm_tab[kFused ? HDKV / 2 : 1];  // angular speeds, read by lane-varying index
    __shared__ float sm_sn[kFused ? HDKV / 2 : 1], sm_cs[kFused ? HDKV / 2 : 1];  // first unit's sin, cos

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int W = a.nk * HDKV;
    const int P = a.nk * a.groups;
    const int n_units = a.n_seq * P * a.n_split;
    volatile int *abort_flag = &sm_abort;

    // The producer lane issues ring stage p_it next; the first p_st0 stages of its first unit go
    // out before the CTA's first barrier (the stage copies need nothing the other threads set up).
    uint32_t p_it = 0;
    int p_st0 = 0;
    unsigned long long t_first = 0;  // when the producer issued its first stage before the barrier
    // Copies one stage (st) of unit t (number u) into the next ring slot.
    auto issue_stage = [&](const Unit &t, int u, int st, uint32_t it_) {
        const int slot = it_ % kNST;
        const int hk = t.y / a.groups;
        sm_meta[slot] = make_int2(u, st);
        mbar_arrive(&meta_full[slot]);  // publishes the slot's unit to the consumers
        unsigned char *sb = ring + static_cast<size_t>(slot) * C::kSlotBytes;
        mbar_expect_tx(&full[slot], C::kSlotBytes);
        // x of the tile copies: in elements of the map (bytes for Q8_0, whose scale slice of this
        // kv head starts xs bytes into the row)
        const int xs = a.row_bytes ? static_cast<int>(W + (hk / kScaleHeads) * 16) : 0;
        if (!a.table) {
            const int row = static_cast<int>(t.base) + t.r_begin + st * R;
            tma_load_2d_stream(sb, &tmK, hk * HDKV, row, &full[slot]);
            tma_load_2d_stream(sb + C::kTensorBytes, &tmV, hk * HDKV, row, &full[slot]);
            if (Q) {
                tma_load_2d(sb + C::kQBytes, &tmKs, xs, row, &full[slot]);
                tma_load_2d(sb + C::kTensorBytes + C::kQBytes, &tmVs, xs, row, &full[slot]);
            }
        } else {
            // one copy per block piece; a block the table does not hold reads as zeros (its rows
            // start past the pool) and is reported
            for (int c = 0; c < R / a.box_rows; ++c) {
                const int lrow = t.r_begin + st * R + c * a.box_rows;
                const int blk = lrow / a.block_rows;
                const int b = blk < a.max_blocks ? __ldg(a.table + static_cast<size_t>(t.s) * a.max_blocks + blk) : -1;
                const long long prow = static_cast<long long>(b) * a.block_rows + lrow % a.block_rows;
                const bool ok = b >= 0 && prow < a.pool_rows;
                if (!ok && lrow < t.L) flag_error(a.err, MINF_ERRBIT_BLOCK);
                const int row = ok ? static_cast<int>(prow) : static_cast<int>(a.pool_rows);
                const int qo = c * a.box_rows * HDKV * EB;
                tma_load_2d(sb + qo, &tmK, hk * HDKV, row, &full[slot]);
                tma_load_2d(sb + C::kTensorBytes + qo, &tmV, hk * HDKV, row, &full[slot]);
                if (Q) {
                    const int so = C::kQBytes + c * a.box_rows * 16;
                    tma_load_2d(sb + so, &tmKs, xs, row, &full[slot]);
                    tma_load_2d(sb + C::kTensorBytes + so, &tmVs, xs, row, &full[slot]);
                }
            }
        }
    };
    if (tid == kProducer * 32) {
        // the tensor maps and every barrier of the CTA, by the lane that issues the copies
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        if (Q) {
            prefetch_tensormap(&tmKs);
            prefetch_tensormap(&tmVs);
        }
        for (int i = 0; i < kNST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kNW);
            mbar_init(&meta_full[i], 1);
        }
        mbar_init(&cons_bar, kNW);
        mbar_init(&knew_bar, 1);
        sm_abort = 0;
        mbar_init_fence();
        // With early start and no ordering of a batch to wait for, the first unit's first stage
        // goes out now: before the angular speeds are staged and the CTA's barrier, a few
        // microseconds earlier than the rest of the CTA gets going.
        if (a.early && !a.sorted) {
            const Unit t = unit_of<R>(a, blockIdx.x, nullptr);
            if (unit_active(t)) {
                issue_stage(t, static_cast<int>(blockIdx.x), 0, 0);
                p_st0 = 1;
                p_it = 1;
                t_first = gtimer();
            }
        }
    }
    if (kFused)
        for (int i = tid; i < HDKV / 2; i += blockDim.x) sm_tab[i] = a.tab.f[i];
    // Without early start nothing is read before the launch ahead of this one has finished:
    // the positions and the cached rows may be its outputs.
    if (!a.early) gdc_wait();
    // A batch is visited longest sequence first (with early start the positions are not written
    // by a preceding kernel, so this runs before the dependency wait): rank = number of longer
    // windows.
    const int *order = nullptr;
    if (a.sorted) {
        for (int s = tid; s < a.n_seq; s += blockDim.x) {
            const int Ls = window_of(a, s);
            int rank = 0;
            for (int o = 0; o < a.n_seq; ++o) {
                const int Lo = window_of(a, o);
                rank += (Lo > Ls) || (Lo == Ls && o < s);
            }
            sm_order[rank] = s;
        }
        order = sm_order;
    }
    __syncthreads();
    // When every unit is a first unit (one per CTA), the CTA whose unit ends at the window's
    // last row has its utility warp append the new row, beside the consumers' start; the
    // consumers patch it into its tile from shared memory once knew_bar says it is staged.
    const bool early = n_units <= static_cast<int>(gridDim.x);
    const Unit t0 = unit_of<R>(a, blockIdx.x, order);  // positions: not written by a preceding kernel
    const bool util_append = kFused && early && unit_active(t0) && t0.r_end == t0.L;

    if (warp == kUtility) {
        // ---------------------------------------------------------------- utility warp
        if (kFused && util_append) {  // the rows it will read after the wait, into L2 now
            const int hk = t0.y / a.groups;
            prefetch_l2(a.k_io + (static_cast<size_t>(t0.s) * a.nk + hk) * HDKV, HDKV * 4, lane);
            prefetch_l2(a.v_new + static_cast<size_t>(t0.s) * W + hk * HDKV, HDKV * 4, lane);
        }
        if (kFused && static_cast<int>(blockIdx.x) < a.n_seq)
            prefetch_l2(a.h + static_cast<size_t>(blockIdx.x) * a.n_embd, a.n_embd * 4, lane);
        // the appended row's angles: its position is not written by a preceding kernel
        float sn[2 * KF4], cs[2 * KF4];
        if (util_append) rope_angles<KF4>(sn, cs, static_cast<float>(t0.p), sm_tab, a.style, lane & 7, lane >> 3);
        gdc_wait();
        if (util_append) {
            // the rotated k written back, the K/V row stored and staged, then -- the row in
            // memory -- the dependent launch released for this CTA
            const int hk = t0.y / a.groups;
            const int pnew = t0.p < t0.cap_s ? t0.p : -1;
            if (lane < 8) append_new_row<HDKV, T>(a, t0, hk, pnew, sn, cs, lane, sm_knew, sm_vnew);
            __syncwarp();
            if (lane == 0) mbar_arrive(&knew_bar);
            if (pnew >= 0) __threadfence();
            __syncwarp();
            if (lane == 0) gdc_launch_dependents();
        }
        // RMSNorm rows ("11 . Attention, vec ops, and the KV cache", §3.2.1), spread over the
        // CTAs; h is produced upstream, so it is read only after the dependency wait.
        for (int s = blockIdx.x; kFused && s < a.n_seq; s += gridDim.x) {
            const float *hr = a.h + static_cast<size_t>(s) * a.n_embd;
            float *yr = a.xn + static_cast<size_t>(s) * a.n_embd;
            const int n4 = a.n_embd >> 2;
            float ss = 0.0f;
#pragma unroll 8
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
#pragma unroll 8
            for (int i = lane; i < n4; i += 32) {
                const float4 v = reinterpret_cast<const float4 *>(hr)[i];
                const float4 g = a.gain ? reinterpret_cast<const float4 *>(a.gain)[i]
                                        : make_float4(1.f, 1.f, 1.f, 1.f);
                reinterpret_cast<float4 *>(yr)[i] = make_float4(v.x * scale * g.x, v.y * scale * g.y,
                                                                v.z * scale * g.z, v.w * scale * g.w);
            }
        }
        // Outputs and error bits that belong to whole sequences: a sequence with an empty
        // window has no unit, and its output is defined as zero.
        for (int s = blockIdx.x; s < a.n_seq; s += gridDim.x) {
            const int p = __ldg(a.pos + s);
            const int cap_s = a.caps ? __ldg(a.caps + s) : a.cap;
            if (lane == 0 && (p < 0 || p >= cap_s)) {
                int bits = MINF_ERRBIT_ATTN_POS;
                if (kFused) bits |= MINF_ERRBIT_STORE_POS | (p < 0 ? MINF_ERRBIT_ROPE_POS : 0);
                flag_error(a.err, bits);
            }
            if (p < 0)
                for (int i = lane; i < a.nh * HDKV; i += 32) a.out[static_cast<size_t>(s) * a.nh * HDKV + i] = 0.0f;
        }
        return;  // writes only this kernel's own outputs: nothing a dependent launch may prefetch
    }
    if (warp == kProducer) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t it = p_it;
            bool waited = false;
            int ptag = 0;  // the workspace's tag, read once the launch before this one has finished
            auto wait_dep = [&]() {
                gdc_wait();
                waited = true;
                ptag = ld_relaxed(a.ws_tag);
            };
            int u = blockIdx.x;  // the first unit is this CTA's own; the rest come from a counter
            while (u < n_units && !*abort_flag) {
                const Unit t = unit_of<R>(a, u, order);
                if (unit_active(t)) {
                    const int n_st = (t.r_end - t.r_begin + R - 1) / R;
                    // the first unit's first p_st0 stages went out before the CTA's barrier
                    for (int st = u == static_cast<int>(blockIdx.x) ? p_st0 : 0; st < n_st && !*abort_flag;
                         ++st, ++it) {
                        const int slot = it % kNST;
                        // Cached rows need no wait, but only kPreWait stages go out before it, and
                        // kPreWaitGapNs apart: this launch's CTAs start as the previous launch's
                        // leave, while its merging splits poll their partials in L2, and a deeper
                        // or denser burst slows those round trips more than it saves here.
                        if (!waited && it > 0 && it < kPreWait && t_first)
                            while (gtimer() - t_first < kPreWaitGapNs) {
                            }
                        if (!waited && it >= kPreWait) wait_dep();
                        if (it >= kNST) {
                            if (!mbar_wait(&empty[slot], ((it / kNST) & 1) ^ 1, abort_flag, a.err)) break;
                        }
                        issue_stage(t, u, st, it);
                    }
                }
                if (early) break;  // every unit is a first unit: nothing to draw
                if (!waited) wait_dep();  // the unit counter lives in the workspace a preceding launch may use
                // a workspace of another layout: no further units (the consumers flag it)
                u = (ptag == 0 || ptag == a.ws_key) ? static_cast<int>(gridDim.x) + atomicAdd(a.ws_ctr, 1) : n_units;
            }
            // With one unit a CTA the producer touches nothing a preceding launch may write: the end
            // of the stream goes out without waiting, and the counters stay unused.
            if (!waited && !early) wait_dep();
            // end of the stream for this CTA's consumers
            const int slot = it % kNST;
            if (it < kNST || mbar_wait(&empty[slot], ((it / kNST) & 1) ^ 1, abort_flag, a.err)) {
                sm_meta[slot] = make_int2(-1, 0);
                mbar_arrive(&meta_full[slot]);
            }
            // the last producer to finish resets the counters for the next call or graph replay
            // (the fences order every producer's draws before its count, and the reset after)
            if (!early) __threadfence();
            if (!early && atomicAdd(a.ws_done, 1) == static_cast<int>(gridDim.x) - 1) {
                __threadfence();
                *a.ws_ctr = 0;
                *a.ws_done = 0;
                // a fresh workspace takes this call's layout (never over a poisoned tag)
                if (ptag == 0) atomicCAS(a.ws_tag, 0, a.ws_key);
            }
            if (*abort_flag) {
                // let copies already issued land before the CTA's shared memory goes away
                for (uint32_t k = it > kNST ? it - kNST : 0; k < it; ++k)
                    if (!mbar_try(&full[k % kNST], (k / kNST) & 1)) {
                        const unsigned long long t0 = gtimer();
                        while (!mbar_try(&full[k % kNST], (k / kNST) & 1) && gtimer() - t0 < kWaitBudgetNs) {
                        }
                    }
                if (!waited) gdc_wait();  // (the workspace may still be the preceding launch's)
                *a.ws_tag = kWsPoison;  // its counters may be left non-zero: refused until zero-filled
            }
        }
        return;  // the producer never releases dependents: only consumers know the rows are written
    }

    // -------------------------------------------------------------------- consumers
    // A dependent launch may start streaming cached rows before its own wait, so release it only
    // once every row this CTA appends is in memory.  The run that ends at the window's last row
    // appends; when every unit is a first unit, a CTA releases at once, or -- when it appends --
    // its utility warp does right after the append; otherwise a CTA releases when it is done.
    bool released = false;
    const int r4 = lane >> 3, sub = lane & 7;
    // The four rows of a K pass (r4) take their 16-byte blocks in rotated order, block
    // (i + rot) mod KF4 at step i, so narrow rows (binary16, Q8_0) land in different banks.
    const int rot = r4 & (KF4 - 1);
    const int vrow = lane / VL, vcol = lane % VL;
    const float sl = a.scale_log2;
    uint32_t cphase = 0;
    uint32_t it = 0;  // ring stage counter, in step with the producer's
    // The first unit is this CTA's own and needs no word from the producer.
    Unit t = t0;
    bool have = unit_active(t);
    bool first_unit = true;
    bool scratch_used = false;  // a previous unit of this CTA has read sm_acc, sm_m, sm_l, sm_red
    if (have && warp < GH) {  // this unit's q rows, into L2 before the wait
        const int h0 = (t.y / a.groups) * (a.nh / a.nk) + (t.y % a.groups) * GH;
        prefetch_l2(a.q + (static_cast<size_t>(t.s) * a.nh + h0 + warp) * a.hd, HDKV * 4, lane);
    }
    // The first unit's RoPE sines and cosines, one pair a thread, before the wait (the position
    // is not written by a preceding kernel): after it, rotating q costs only table reads.
    const bool pre_ang = kFused && have;
    if (kFused) {
        if (pre_ang)
            for (int i = tid; i < HDKV / 2; i += kCons)
                sincosf(__fmul_rn(static_cast<float>(t.p), sm_tab[i]), &sm_sn[i], &sm_cs[i]);
        cons_sync(&cons_bar, cphase, abort_flag, a.err);
    }
    gdc_wait();
    if (early) {
        if (!util_append) gdc_launch_dependents();  // this CTA appends no row
        released = true;
    }
    // The workspace's tag, checked before the first partial is written (the load is in flight
    // meanwhile): a workspace another layout left may hold non-zero words where this call's
    // partials are, which would read as written.
    const int ctag = tid == 0 ? ld_relaxed(a.ws_tag) : 0;
    bool ws_checked = false;
    while (true) {
        if (!have) {
            // the producer publishes the unit it drew with the unit's first stage
            const int slot = it % kNST;
            if (!mbar_wait(&meta_full[slot], (it / kNST) & 1, abort_flag, a.err)) break;
            const int u = sm_meta[slot].x;
            if (u < 0) break;
            t = unit_of<R>(a, u, order);
        }
        have = false;
        // -------------------------------------------------------------- start of a unit
        const int hk = t.y / a.groups;
        const int h0 = hk * (a.nh / a.nk) + (t.y % a.groups) * GH;  // first query head
        const int n_st = (t.r_end - t.r_begin + R - 1) / R;
        float4 qr[GH][KF4];
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) {
            const float4 *qh =
                reinterpret_cast<const float4 *>(a.q + (static_cast<size_t>(t.s) * a.nh + h0 + hh) * a.hd);
#pragma unroll
            for (int i = 0; i < KF4; ++i) qr[hh][i] = qh[sub + 8 * i];
        }
        // The unit whose run ends at the window's last row owns k: it rotates it, writes it back
        // and, when the row fits the region, appends the new K/V row and puts it, from shared
        // memory, in place of what its tile copy read (no other unit reads k).
        const bool k_writer = kFused && t.r_end == t.L;
        const int pnew = k_writer && t.p < t.cap_s ? t.p : -1;
        const bool util_unit = util_append && first_unit;  // appended by the utility warp
        const bool tab_unit = pre_ang && first_unit;        // angles already in shared memory
        first_unit = false;
        if (kFused) {
            float sn[2 * KF4], cs[2 * KF4];
            if (tab_unit)
                rope_angles_tab<KF4>(sn, cs, sm_sn, sm_cs, a.style, sub);
            else
                rope_angles<KF4>(sn, cs, static_cast<float>(t.p), sm_tab, a.style, sub, r4);
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) rope_lane<KF4>(qr[hh], sn, cs, a.style);
            if (k_writer && !util_unit && warp == 0 && r4 == 0)
                append_new_row<HDKV, T>(a, t, hk, pnew, sn, cs, sub, sm_knew, sm_vnew);
        }
        // q's blocks in the lane's rotated order (the lanes that write q back have rot = 0)
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) {
            float4 t0[KF4];
#pragma unroll
            for (int i = 0; i < KF4; ++i) t0[i] = qr[hh][i];
#pragma unroll
            for (int i = 0; i < KF4; ++i) {
                float4 v = t0[i];
#pragma unroll
                for (int r = 1; r < KF4; ++r)
                    if (rot == r) v = t0[(i + r) & (KF4 - 1)];
                qr[hh][i] = v;
            }
        }
        float m[GH], l[GH];
        float4 accs[NACC][GH];  // V rows alternate between NACC accumulators (shorter FMA chains)
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) {
            m[hh] = -INFINITY;
            l[hh] = 0.0f;
#pragma unroll
            for (int c = 0; c < NACC; ++c) accs[c][hh] = make_float4(0.f, 0.f, 0.f, 0.f);
        }

        // -------------------------------------------------------------- the unit's stages
        for (int st = 0; st < n_st; ++st, ++it) {
            const int slot = it % kNST;
            mbar_wait(&full[slot], (it / kNST) & 1, abort_flag, a.err);
            unsigned char *Kq = ring + static_cast<size_t>(slot) * C::kSlotBytes;  // K values / quants
            unsigned char *Ksc = Kq + C::kQBytes;                                 // K scale slices
            unsigned char *Vq = Kq + C::kTensorBytes;
            unsigned char *Vsc = Vq + C::kQBytes;
            const int sc0 = (hk % kScaleHeads) * (HDKV / 32);  // this head's first scale in a slice
            const int row0 = t.r_begin + st * R;
            if (kFused && pnew >= row0 && pnew < row0 + R) {
                // the tile may hold the row as it was before this launch appended it: the lanes
                // that staged the new row put it in its place (and hand the slot back to the
                // async proxy in order)
                if (util_unit && warp == 0) mbar_wait(&knew_bar, 0, abort_flag, a.err);
                if (warp == 0 && r4 == 0) {
                    const int rn = pnew - row0;
                    if constexpr (Q) {
#pragma unroll
                        for (int i = 0; i < KF4; ++i) {
                            reinterpret_cast<uint32_t *>(Kq + rn * HDKV)[sub + 8 * i] =
                                reinterpret_cast<const uint32_t *>(sm_knew)[sub + 8 * i];
                            reinterpret_cast<uint32_t *>(Vq + rn * HDKV)[sub + 8 * i] =
                                reinterpret_cast<const uint32_t *>(sm_vnew)[sub + 8 * i];
                            if (sub == 0) {
                                reinterpret_cast<__half *>(Ksc + rn * 16)[sc0 + i] =
                                    reinterpret_cast<const __half *>(reinterpret_cast<const unsigned char *>(sm_knew) + HDKV)[i];
                                reinterpret_cast<__half *>(Vsc + rn * 16)[sc0 + i] =
                                    reinterpret_cast<const __half *>(reinterpret_cast<const unsigned char *>(sm_vnew) + HDKV)[i];
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < KF4; ++i) {
                            st4(reinterpret_cast<T *>(Kq) + rn * HDKV, sub + 8 * i,
                                reinterpret_cast<const float4 *>(sm_knew)[sub + 8 * i]);
                            st4(reinterpret_cast<T *>(Vq) + rn * HDKV, sub + 8 * i,
                                reinterpret_cast<const float4 *>(sm_vnew)[sub + 8 * i]);
                        }
                    }
                    fence_async_smem();
                }
                cons_sync(&cons_bar, cphase, abort_flag, a.err);
            }
            // The warp's SPW sub-tiles of kSub rows, GRP at a time: the scores of all their rows
            // first (a K row is spread over 8 lanes, four rows per pass), then one online-softmax
            // update for them, then their V rows (one per pass of VL lanes).  Q8_0 blocks apply
            // their scale once: to a block's partial dot product (K), and to the weight (V).
#pragma unroll 1
            for (int g0 = 0; g0 < SPW; g0 += GRP) {  // one pass when the heads are few
            float sc[GRP][KP][GH];
#pragma unroll
            for (int sp = 0; sp < GRP; ++sp) {
                const int rr0 = (warp * SPW + g0 + sp) * kSub;  // sub-tile's first row within the stage
#pragma unroll
                for (int it2 = 0; it2 < KP; ++it2) {
                    const int rr = rr0 + 4 * it2 + r4;
                    float4 kv[KF4];
#pragma unroll
                    for (int i = 0; i < KF4; ++i)
                        kv[i] = ld_row4_raw<HDKV, T>(Kq + rr * HDKV * EB, sub + 8 * ((i + rot) & (KF4 - 1)));
                    float ks[Q ? KF4 : 1];
                    if constexpr (Q) ld_scales<HDKV>(Ksc + rr * 16, sc0, rot, ks);
#pragma unroll
                    for (int hh = 0; hh < GH; ++hh) {
                        // packed pairs: even and odd elements summed apart, added at the end
                        float2 d2 = make_float2(0.0f, 0.0f);
#pragma unroll
                        for (int i = 0; i < KF4; ++i) {
                            if constexpr (Q) {
                                float2 b2 = mul2(lo2(qr[hh][i]), lo2(kv[i]));
                                b2 = fma2(hi2(qr[hh][i]), hi2(kv[i]), b2);
                                d2 = fma2(make_float2(ks[i], ks[i]), b2, d2);
                            } else {
                                d2 = fma2(lo2(qr[hh][i]), lo2(kv[i]), d2);
                                d2 = fma2(hi2(qr[hh][i]), hi2(kv[i]), d2);
                            }
                        }
                        float d = d2.x + d2.y;
                        d += __shfl_xor_sync(0xffffffffu, d, 1);
                        d += __shfl_xor_sync(0xffffffffu, d, 2);
                        d += __shfl_xor_sync(0xffffffffu, d, 4);
                        sc[sp][it2][hh] = (row0 + rr) < t.r_end ? d * sl : -INFINITY;
                    }
                }
            }
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) {
                float mx = sc[0][0][hh];
#pragma unroll
                for (int sp = 0; sp < GRP; ++sp)
#pragma unroll
                    for (int it2 = 0; it2 < KP; ++it2) mx = fmaxf(mx, sc[sp][it2][hh]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m[hh], mx);
                // rows wholly past the run leave the state untouched
                const bool none = (m_new == -INFINITY);
                const float corr = none ? 1.0f : ex2_approx(m[hh] - m_new);
                float ps = 0.0f;
#pragma unroll
                for (int sp = 0; sp < GRP; ++sp)
#pragma unroll
                    for (int it2 = 0; it2 < KP; ++it2) {
                        const float pv = none ? 0.0f : ex2_approx(sc[sp][it2][hh] - m_new);
                        sc[sp][it2][hh] = pv;  // from here on: the row's weight
                        ps += pv;
                    }
                ps += __shfl_xor_sync(0xffffffffu, ps, 8);
                ps += __shfl_xor_sync(0xffffffffu, ps, 16);
                l[hh] = fmaf(l[hh], corr, ps);
#pragma unroll
                for (int c = 0; c < NACC; ++c) accs[c][hh] = f4scale(accs[c][hh], corr);
                m[hh] = m_new;
            }
#pragma unroll
            for (int sp = 0; sp < GRP; ++sp) {
                const int rr0 = (warp * SPW + g0 + sp) * kSub;
#pragma unroll
                for (int jv = 0; jv < VJ; ++jv) {
                    const int rl = vrow + VRP * jv;  // row within the sub-tile, 0..kSub-1
                    const int rr = rr0 + rl;
                    const bool in_run = row0 + rr < t.r_end;
                    // past the run: anything finite (its weight is 0)
                    const float4 v = in_run ? ld_row4_raw<HDKV, T>(Vq + rr * HDKV * EB, vcol)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                    float vs = 1.0f;
                    if constexpr (Q)
                        vs = __half2float(reinterpret_cast<const __half *>(Vsc + rr * 16)[sc0 + (vcol >> 3)]);
                    const int it2 = (VRP * jv) / 4;  // the same for every lane of the pass
                    const int src = (rl & 3) * 8;
#pragma unroll
                    for (int hh = 0; hh < GH; ++hh) {
                        float w = __shfl_sync(0xffffffffu, sc[sp][it2][hh], src);
                        if constexpr (Q) w *= vs;
                        float4 &ac = accs[((g0 + sp) * VJ + jv) % NACC][hh];
                        const float2 w2 = make_float2(w, w);
                        ac = cat2(fma2(w2, lo2(v), lo2(ac)), fma2(w2, hi2(v), hi2(ac)));
                    }
                }
            }
            }  // sub-tile group
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // ------------------------------------------------------------ end of the unit
        if (scratch_used)  // the previous unit's readers of the shared scratch are done
            cons_sync(&cons_bar, cphase, abort_flag, a.err);
        scratch_used = true;
        float4 acc[GH];
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) {
            acc[hh] = accs[0][hh];
#pragma unroll
            for (int c = 1; c < NACC; ++c)
                acc[hh] = make_float4(acc[hh].x + accs[c][hh].x, acc[hh].y + accs[c][hh].y,
                                      acc[hh].z + accs[c][hh].z, acc[hh].w + accs[c][hh].w);
        }
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
        if (tid == 0 && !ws_checked) {
            sm_wsbad = !(ctag == 0 || ctag == a.ws_key);
            if (sm_wsbad) flag_error(a.err, MINF_ERRBIT_WORKSPACE);
            // a fresh workspace takes this call's layout (when units are drawn, the last producer
            // does it; here no producer counts its finish)
            if (early && ctag == 0) atomicCAS(a.ws_tag, 0, a.ws_key);
        }
        ws_checked = true;
        cons_sync(&cons_bar, cphase, abort_flag, a.err);
        if (sm_wsbad) continue;  // nothing that depends on the workspace: no partial, merge or output
        // The run that ends the window (the group's last split, the shortest) merges: every other
        // split stores its partial (m, l, acc) encoded so that zero reads as "not yet written" and
        // leaves at once -- no atomic, no wait -- and the merger polls the partial words themselves
        // until all are written, folds them in a fixed order and zeroes them for the next call.
        float *out_s = a.out + (static_cast<size_t>(t.s) * a.nh + h0) * HDKV;
        const size_t part0 = (static_cast<size_t>(t.s) * a.nh + h0) * a.n_split;  // head h0, split 0
        constexpr int kPairs = GH * VL;  // (head, float4 column) pairs of the unit's output
        static_assert(kPairs <= kCons, "one pair per consumer thread");
        const bool multi = t.n_act > 1;
        // Units of many heads (GH >= 5) merge by ticket instead: every split stores its partial
        // and the last to arrive folds them all.  The polling merge's registers weighed on their
        // stage loop (the 7-head decode step: 12.8 against 10.8 us without it).
        constexpr bool kTicket = GH >= 5;
        const bool merger = !kTicket && t.j == t.n_act - 1;
        float own_M = -INFINITY, own_L = 0.0f;  // this unit's partial, for thread tid's pair
        float4 own_A = make_float4(0.f, 0.f, 0.f, 0.f);
        if (tid < kPairs) {
            const int hh = tid / VL, c = tid % VL;
            float M = sm_m[0][hh];
#pragma unroll
            for (int w = 1; w < kNW; ++w) M = fmaxf(M, sm_m[w][hh]);
            float Ls = 0.0f;
            float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kNW; ++w) {
                const float f = sm_m[w][hh] == -INFINITY ? 0.0f : ex2_approx(sm_m[w][hh] - M);
                Ls = fmaf(sm_l[w][hh], f, Ls);
                const float4 x = sm_acc[w][hh][c];
                A.x = fmaf(x.x, f, A.x);
                A.y = fmaf(x.y, f, A.y);
                A.z = fmaf(x.z, f, A.z);
                A.w = fmaf(x.w, f, A.w);
            }
            if (!multi) {
                reinterpret_cast<float4 *>(out_s + hh * HDKV)[c] = f4scale(A, 1.0f / Ls);
            } else if (!merger) {
                const size_t part = part0 + static_cast<size_t>(hh) * a.n_split + t.j;
                if (c == 0)
                    reinterpret_cast<uint2 *>(a.ws_ml)[part] = make_uint2(part_enc(M), part_enc(Ls));
                reinterpret_cast<uint4 *>(a.ws_acc + part * HDKV)[c] =
                    make_uint4(part_enc(A.x), part_enc(A.y), part_enc(A.z), part_enc(A.w));
            } else {
                own_M = M;
                own_L = Ls;
                own_A = A;
            }
        }
        if constexpr (kTicket) {
            if (multi) {
                int *ticket = a.ws_ticket + static_cast<size_t>(t.s) * a.nh + h0;
                cons_sync(&cons_bar, cphase, abort_flag, a.err);  // every partial store of the CTA first
                if (tid == 0) {
                    // acq_rel: publishes this CTA's partials and, for the last arrival, makes every
                    // other split's visible to the loads below
                    int old;
                    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(ticket) : "memory");
                    sm_last = old == t.n_act - 1;
                }
                cons_sync(&cons_bar, cphase, abort_flag, a.err);
                if (!sm_last) continue;
                // one round trip: each thread folds its share of the splits, then the shares
                constexpr int kWays = kCons / kPairs;
                for (int i = tid; i < kPairs * kWays; i += kCons) {
                    const int pair = i % kPairs, way = i / kPairs;
                    const int hh = pair / VL, c = pair % VL;
                    const size_t ph2 = part0 + static_cast<size_t>(hh) * a.n_split;
                    float M = -INFINITY, Ls = 0.0f;
                    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                    for (int j = way; j < t.n_act; j += kWays) {
                        const uint2 mlv = __ldcg(reinterpret_cast<const uint2 *>(a.ws_ml) + (ph2 + j));
                        const uint4 xv = __ldcg(reinterpret_cast<const uint4 *>(a.ws_acc + (ph2 + j) * HDKV) + c);
                        const float mj = part_dec(mlv.x), lj = part_dec(mlv.y);
                        const float Mn = fmaxf(M, mj);
                        const float fo = M == -INFINITY ? 0.0f : ex2_approx(M - Mn);
                        const float fn = mj == -INFINITY ? 0.0f : ex2_approx(mj - Mn);
                        A = make_float4(fmaf(part_dec(xv.x), fn, A.x * fo), fmaf(part_dec(xv.y), fn, A.y * fo),
                                        fmaf(part_dec(xv.z), fn, A.z * fo), fmaf(part_dec(xv.w), fn, A.w * fo));
                        Ls = fmaf(lj, fn, Ls * fo);
                        M = Mn;
                    }
                    sm_red[way * kPairs + pair] = A;
                    sm_redM[way * kPairs + pair] = M;
                    sm_redL[way * kPairs + pair] = Ls;
                }
                cons_sync(&cons_bar, cphase, abort_flag, a.err);
                // the partials read go back to zero for the next call, and the ticket
                for (int i = tid; i < kPairs * kWays; i += kCons) {
                    const int pair = i % kPairs, way = i / kPairs;
                    const int hh = pair / VL, c = pair % VL;
                    const size_t ph2 = part0 + static_cast<size_t>(hh) * a.n_split;
                    for (int j = way; j < t.n_act; j += kWays) {
                        reinterpret_cast<uint4 *>(a.ws_acc + (ph2 + j) * HDKV)[c] = make_uint4(0u, 0u, 0u, 0u);
                        if (c == 0) reinterpret_cast<uint2 *>(a.ws_ml)[ph2 + j] = make_uint2(0u, 0u);
                    }
                }
                if (tid == 0) *ticket = 0;
                if (tid < kPairs) {
                    const int hh = tid / VL, c = tid % VL;
                    float M = sm_redM[tid];
                    for (int w = 1; w < kWays; ++w) M = fmaxf(M, sm_redM[w * kPairs + tid]);
                    float Ls = 0.0f;
                    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int w = 0; w < kWays; ++w) {
                        const float mw = sm_redM[w * kPairs + tid];
                        const float f = mw == -INFINITY ? 0.0f : ex2_approx(mw - M);
                        const float4 x = sm_red[w * kPairs + tid];
                        A = make_float4(fmaf(x.x, f, A.x), fmaf(x.y, f, A.y), fmaf(x.z, f, A.z), fmaf(x.w, f, A.w));
                        Ls = fmaf(sm_redL[w * kPairs + tid], f, Ls);
                    }
                    reinterpret_cast<float4 *>(out_s + hh * HDKV)[c] = f4scale(A, 1.0f / Ls);
                }
            }
        } else {
        if (multi && !merger) continue;  // the partial is stored: this unit is done

        if (multi) {  // (polling merge)
            // Each thread polls and folds its share of the other splits (those of index
            // way mod kWays, kChunk of them with their loads in flight together), in split order;
            // then the shares are folded in shared memory, and this unit's own partial last.
            constexpr int kWays = kCons / kPairs;
            constexpr int kChunk = GH <= 2 ? 8 : (GH <= 4 ? 4 : 2);
            const int n_oth = t.n_act - 1;  // the other splits: 0 .. n_act - 2
            for (int i = tid; i < kPairs * kWays; i += kCons) {
                const int pair = i % kPairs, way = i / kPairs;
                const int hh = pair / VL, c = pair % VL;
                const size_t ph2 = part0 + static_cast<size_t>(hh) * a.n_split;
                float M = -INFINITY, Ls = 0.0f;
                float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int j0 = way; j0 < n_oth; j0 += kWays * kChunk) {
                    uint2 mlv[kChunk];
                    uint4 xv[kChunk];
                    uint32_t pend = 0;
#pragma unroll
                    for (int k = 0; k < kChunk; ++k)
                        if (j0 + k * kWays < n_oth) pend |= 1u << k;
                    const unsigned long long tb = gtimer();
                    while (pend && !*abort_flag) {
#pragma unroll
                        for (int k = 0; k < kChunk; ++k)
                            if (pend >> k & 1u) {
                                const size_t part = ph2 + j0 + k * kWays;
                                mlv[k] = ld_relaxed_v2(reinterpret_cast<const uint2 *>(a.ws_ml) + part);
                                xv[k] = ld_relaxed_v4(reinterpret_cast<const uint4 *>(a.ws_acc + part * HDKV) + c);
                            }
#pragma unroll
                        for (int k = 0; k < kChunk; ++k)
                            if ((pend >> k & 1u) && mlv[k].x && mlv[k].y && xv[k].x && xv[k].y && xv[k].z && xv[k].w)
                                pend &= ~(1u << k);
                        if (pend && gtimer() - tb > kWaitBudgetNs) {
                            *abort_flag = 1;
                            flag_error(a.err, MINF_ERRBIT_TIMEOUT);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < kChunk; ++k) {
                        if (j0 + k * kWays >= n_oth) break;
                        const float mj = part_dec(mlv[k].x), lj = part_dec(mlv[k].y);
                        const float4 x = make_float4(part_dec(xv[k].x), part_dec(xv[k].y), part_dec(xv[k].z),
                                                     part_dec(xv[k].w));
                        const float Mn = fmaxf(M, mj);
                        const float fo = M == -INFINITY ? 0.0f : ex2_approx(M - Mn);
                        const float fn = mj == -INFINITY ? 0.0f : ex2_approx(mj - Mn);
                        A = make_float4(fmaf(x.x, fn, A.x * fo), fmaf(x.y, fn, A.y * fo), fmaf(x.z, fn, A.z * fo),
                                        fmaf(x.w, fn, A.w * fo));
                        Ls = fmaf(lj, fn, Ls * fo);
                        M = Mn;
                    }
                }
                sm_red[way * kPairs + pair] = A;
                sm_redM[way * kPairs + pair] = M;
                sm_redL[way * kPairs + pair] = Ls;
            }
            cons_sync(&cons_bar, cphase, abort_flag, a.err);
            // every poll is done: the partials read go back to zero for the next call
            for (int i = tid; i < kPairs * kWays; i += kCons) {
                const int pair = i % kPairs, way = i / kPairs;
                const int hh = pair / VL, c = pair % VL;
                const size_t ph2 = part0 + static_cast<size_t>(hh) * a.n_split;
                for (int j = way; j < n_oth; j += kWays) {
                    reinterpret_cast<uint4 *>(a.ws_acc + (ph2 + j) * HDKV)[c] = make_uint4(0u, 0u, 0u, 0u);
                    if (c == 0) reinterpret_cast<uint2 *>(a.ws_ml)[ph2 + j] = make_uint2(0u, 0u);
                }
            }
            if (tid < kPairs) {
                const int hh = tid / VL, c = tid % VL;
                float M = own_M;
                for (int w = 0; w < kWays; ++w) M = fmaxf(M, sm_redM[w * kPairs + tid]);
                const float fo = own_M == -INFINITY ? 0.0f : ex2_approx(own_M - M);
                float Ls = 0.0f;
                float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int w = 0; w < kWays; ++w) {
                    const float mw = sm_redM[w * kPairs + tid];
                    const float f = mw == -INFINITY ? 0.0f : ex2_approx(mw - M);
                    const float4 x = sm_red[w * kPairs + tid];
                    A = make_float4(fmaf(x.x, f, A.x), fmaf(x.y, f, A.y), fmaf(x.z, f, A.z), fmaf(x.w, f, A.w));
                    Ls = fmaf(sm_redL[w * kPairs + tid], f, Ls);
                }
                A = make_float4(fmaf(own_A.x, fo, A.x), fmaf(own_A.y, fo, A.y), fmaf(own_A.z, fo, A.z),
                                fmaf(own_A.w, fo, A.w));
                Ls = fmaf(own_L, fo, Ls);
                reinterpret_cast<float4 *>(out_s + hh * HDKV)[c] = f4scale(A, 1.0f / Ls);
            }
        }
        }  // (polling merge)
        if (kFused && lane < 8) {
            // every other unit of this group has finished reading q: write it back rotated
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) {
                if (hh % kNW != warp) continue;
                float4 *qh = reinterpret_cast<float4 *>(a.q_io + (static_cast<size_t>(t.s) * a.nh + h0 + hh) * a.hd);
#pragma unroll
                for (int i = 0; i < KF4; ++i) qh[lane + 8 * i] = qr[hh][i];
            }
        }
    }
    if (*abort_flag && tid == 0) *a.ws_tag = kWsPoison;  // a wait expired: refused until zero-filled
    if (!released) gdc_launch_dependents();
}

template <int HDKV, int GH, bool kFused, typename T>
cudaError_t launch_t(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tks,
                     const CUtensorMap &tvs, const KParams &k, int grid, cudaStream_t s,
                     bool pdl) {
    const size_t smem = static_cast<size_t>(kNST) * Cfg<HDKV, T>::kSlotBytes + 1024;
    constexpr int kThreads = Warps<consumer_warps(GH, HDKV)>::kThreads;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static std::atomic<bool> attr_set[64];  // per device, shared by host threads
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<HDKV, GH, kFused, T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_kernel<HDKV, GH, kFused, T>, tk, tv, tks, tvs, k);
}

template <int HDKV, bool kFused, typename T>
cudaError_t dispatch_gh(int gh, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tks,
                     const CUtensorMap &tvs, const KParams &k, int grid,
                        cudaStream_t s, bool pdl) {
    switch (gh) {
        case 1: return launch_t<HDKV, 1, kFused, T>(tk, tv, tks, tvs, k, grid, s, pdl);
        case 2: return launch_t<HDKV, 2, kFused, T>(tk, tv, tks, tvs, k, grid, s, pdl);
        case 3: return launch_t<HDKV, 3, kFused, T>(tk, tv, tks, tvs, k, grid, s, pdl);
        case 4: return launch_t<HDKV, 4, kFused, T>(tk, tv, tks, tvs, k, grid, s, pdl);
        case 5: return launch_t<HDKV, 5, kFused, T>(tk, tv, tks, tvs, k, grid, s, pdl);
        case 6: return launch_t<HDKV, 6, kFused, T>(tk, tv, tks, tvs, k, grid, s, pdl);
        case 7: return launch_t<HDKV, 7, kFused, T>(tk, tv, tks, tvs, k, grid, s, pdl);
        case 8: return launch_t<HDKV, 8, kFused, T>(tk, tv, tks, tvs, k, grid, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}


// Launch for a storage type: the geometry's head dimension, fused or not, heads per unit.
template <typename T>
cudaError_t dispatch(int hd_kv, bool fused, int gh, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tks,
                     const CUtensorMap &tvs, const KParams &k,
                     int grid, cudaStream_t s, bool pdl) {
    if (fused)
        return hd_kv == 64 ? dispatch_gh<64, true, T>(gh, tk, tv, tks, tvs, k, grid, s, pdl)
                           : dispatch_gh<128, true, T>(gh, tk, tv, tks, tvs, k, grid, s, pdl);
    return hd_kv == 64 ? dispatch_gh<64, false, T>(gh, tk, tv, tks, tvs, k, grid, s, pdl)
                       : dispatch_gh<128, false, T>(gh, tk, tv, tks, tvs, k, grid, s, pdl);
}

}  // namespace dec

// The binary16 and Q8_0 instantiations live in their own translation units
// (minf_decode_f16.cu, minf_decode_q8.cu).
cudaError_t dispatch_decode_f16(int hd_kv, bool fused, int gh, const CUtensorMap &tk, const CUtensorMap &tv,
                                const CUtensorMap &tks, const CUtensorMap &tvs, const dec::KParams &k, int grid,
                                cudaStream_t s, bool pdl);
cudaError_t dispatch_decode_q8(int hd_kv, bool fused, int gh, const CUtensorMap &tk, const CUtensorMap &tv,
                               const CUtensorMap &tks, const CUtensorMap &tvs, const dec::KParams &k, int grid,
                               cudaStream_t s, bool pdl);

}  // namespace minf
