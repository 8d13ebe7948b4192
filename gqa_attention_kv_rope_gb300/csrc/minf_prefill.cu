// minf_prefill.cu -- causal prefill attention on the 5th-generation tensor cores.
//
// "11 . Attention, vec ops, and the KV cache", §3.2.4 defines the result: token t attends
// over rows [0, min(pos[t] + 1, cap)) of its kv head's K/V regions (causal by length, no
// mask matrix), with softmax(scale * q . k) weights on V.  §2.5 names the GPU shape: tile
// the (query, key) matrix and apply the softmax online, block by block.
//
// Tiling.  A CTA owns one query head, 128 consecutive query tokens (the M = 128 rows of the
// tensor-core tiles) and one chunk of the keys of that head's kv head, which it walks in tiles
// of 32 up to the largest window among its tokens.  The chunks of a query tile run in separate
// CTAs; each writes its rows' (max, sum, output) partials and the last chunk to arrive (an
// atomic ticket) folds them, so a long causal window is spread over many SMs.  Per key tile:
//   S  = Q K^T        tcgen05.mma kind::f16, M=128 N=32 K=hd_kv, fp32 accumulator in TMEM
//   softmax            CUDA cores: one thread per query row reads its S row from TMEM,
//                      masks keys beyond its window, updates its running max and sum, and
//                      writes P = 2^(s*scale*log2e - m) into shared memory
//   O_t = P V          tcgen05.mma kind::tf32, M=128 N=hd_kv K=32, into a second TMEM range
//   O  = O*corr + O_t  in registers
// Precision: every operand is split into two halves, x = hi + lo, and each product is the sum
// of three MMAs hi*hi + hi*lo + lo*hi, which brings the tensor-core result to fp32 accuracy.
// For S the halves are binary16: each Q row and each K row is first scaled by a power of two
// that puts its largest magnitude in [2^14, 2^15), so that both halves stay normal, and the
// scales are undone exactly on S (K = 16 per instruction: half the instructions of TF32).  P
// and V^T use TF32 halves (hi = x rounded to TF32, lo = the remainder rounded to TF32: the
// split-precision "3xTF32" scheme).  Q and K tiles arrive by TMA (cp.async.bulk.tensor,
// 128-byte swizzle); Q is converted by the softmax threads, K by two staging warps, which also
// transpose and split V into the K-major layout the MMA takes.  These are generic-proxy writes,
// fenced to the async proxy before the MMA that reads them is released.  Warp 4 is the
// producer: one elected thread issues the TMA copies and the S products; warp 7's first thread
// issues the P*V products (each thread commits its own).
//
// Pipelining.  S has two TMEM buffers and the producer issues S(i+1) as soon as key tile i+1
// is converted (and P(i-1) has been published, so S(i-1)'s buffer is free), without waiting for
// P(i)V(i), which the other thread issues: the tensor cores form the next scores while the
// softmax warps work on the current ones, and neither product waits behind the other's issue
// (a thread issues a tensor-core instruction only every ~35-50 ns).  O_t has two TMEM buffers as well: the softmax warps publish
// P(i) first and fold O_t(i-1) into their registers after it, while the tensor cores form
// O_t(i) (with hd_kv 64 P also has two buffers in shared memory; with hd_kv 128, where shared
// memory holds one, P(i) waits until O_t(i-1) has read P(i-1)).
//
// Two kernels run these items.  prefill_kernel is one CTA per item (the attention alone, after
// a separate RoPE + store launch).  prefill_step_kernel is a whole prefill layer step in one
// cooperative launch of at most one CTA an SM: the step's row work (RMSNorm, RoPE on q and k,
// the K/V store) over the whole grid, a grid barrier, then the items that have keys in turn.
//
// Every mbarrier wait and the grid barrier are bounded by a 200 ms global-timer budget; a wait
// that expires sets MINF_ERRBIT_TIMEOUT, makes every role leave its loop, and the CTA still
// frees its TMEM.
#include <cuda.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cmath>
#include <cstddef>
#include <type_traits>

#include "minf_common.cuh"
#include "minf_kernels.h"
#include "minf_prologue.cuh"
#include "minf_q8.cuh"
#include "minf_sm103.cuh"

namespace minf {

namespace {

constexpr int BM = 128;              // query rows per CTA
constexpr int BN = 32;               // keys per tile
constexpr int kSoftThreads = 128;    // warps 0-3: TMEM lanes 0..127, one query row each
constexpr int kProducerWarp = 4;
constexpr int kStageWarp0 = 5;       // warps 5-6: K split, V^T staging
constexpr int kStageThreads = 64;
constexpr int kPvWarp = 7;           // issues the P*V products
constexpr int kThreadsP = kSoftThreads + 32 + kStageThreads + 32;
// TMEM: S(i) at column (i % 2) * BN, O_t(i) at column 128 + (i % 2) * HDKV
template <int HDKV>
constexpr uint32_t tmem_cols() { return 128 + 2 * HDKV <= 256 ? 256 : 512; }
template <int HDKV>
__device__ __forceinline__ uint32_t o_col(int i) { return 128u + static_cast<uint32_t>(i & 1) * HDKV; }
__device__ __forceinline__ uint32_t s_col(int i) { return static_cast<uint32_t>(i & 1) * BN; }

// Operands are held as hi + lo pairs (x = hi + lo to about 2^-22 relative; binary16 halves of
// scaled rows for Q and K, TF32 halves for P and V^T): each product is formed from three
// tensor-core MMAs, hi*hi + hi*lo + lo*hi, so the narrow inputs of the tensor core cost no
// accuracy beyond fp32 accumulation.
// K and V^T tiles are double-buffered where shared memory allows (hd_kv 64): key tile j lives
// in buffer j % NB.
template <int HDKV>
struct Smem {
    static constexpr int NB = HDKV == 64 ? 2 : 1;   // K and V^T tile buffers
    static constexpr int NP = HDKV == 64 ? 2 : 1;   // P buffers
    // Q and K arrive by TMA as fp32 in qh and kh (32-column SW128 slabs); their binary16
    // hi + lo halves (64-column SW128 slabs, hi then lo) are written into ql and kl
    float qh[HDKV / 32][BM * 32], ql[HDKV / 32][BM * 32];
    float kh[NB][HDKV / 32][BN * 32], kl[NB][HDKV / 32][BN * 32];
    float ph[NP][BN / 32][BM * 32], pl[NP][BN / 32][BM * 32];        // P: keys along K
    float vh[NB][BN / 32][HDKV * 32], vl[NB][BN / 32][HDKV * 32];    // V^T: keys along K
    unsigned long long bar_q, bar_k[NB], bar_qs, bar_kk[NB], bar_vv[NB], bar_s[2], bar_p[2], bar_o[2];
    unsigned long long bar_ks[4];  // slot j % 4 of ks written (key tile j)
    unsigned long long bar_m;      // merge: other chunks' partial outputs copied in
    alignas(16) float ks[4][BN];  // per key of tile j (slot j % 4): the factor undoing its row's scale
    uint32_t tmem_base;
    int abort_flag;
    int lmax;
};

// After the last product of a CTA its shared memory is free.  The output rows are staged from
// the start of qh (kStg bytes, padded rows); the merge of key chunks copies other chunks'
// partial outputs (kPart bytes each) into the kN slots that follow, up to the end of vl.
template <int HDKV>
struct MergeSlots {
    static constexpr int kRS = HDKV + 4;  // staged row stride in floats (no bank conflicts)
    static constexpr size_t kStg = (static_cast<size_t>(BM) * kRS * 4 + 127) & ~static_cast<size_t>(127);
    static constexpr size_t kPart = static_cast<size_t>(HDKV) * BM * 4;
    static constexpr size_t kEnd = offsetof(Smem<HDKV>, vl) + sizeof(Smem<HDKV>::vl) - offsetof(Smem<HDKV>, qh);
    static constexpr int kN = static_cast<int>((kEnd - kStg) / kPart);
    static_assert(kEnd == sizeof(Smem<HDKV>::qh) + sizeof(Smem<HDKV>::ql) + sizeof(Smem<HDKV>::kh) +
                              sizeof(Smem<HDKV>::kl) + sizeof(Smem<HDKV>::ph) + sizeof(Smem<HDKV>::pl) +
                              sizeof(Smem<HDKV>::vh) + sizeof(Smem<HDKV>::vl),
                  "qh .. vl are contiguous");
    static_assert(kN >= 1, "one chunk's partials fit");
};

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle layout
// (8-row x 128-byte atoms, atoms 1024 bytes apart along M/N).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset: next 8 rows
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::tf32, fp32 accumulate, A and B tf32, both K-major.
__host__ __device__ constexpr uint32_t tf32_idesc(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// One split-precision product step: D (+)= Ah*Bh + Ah*Bl + Al*Bh, three MMAs issued together
// (the first accumulates into D only when `accumulate` is non-zero).
// kind::f16 with binary16 A and B, fp32 accumulate, both K-major.
__host__ __device__ constexpr uint32_t f16_idesc(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// One split-precision product step on binary16 halves (K = 16): D (+)= Ah*Bh + Ah*Bl + Al*Bh.
__device__ __forceinline__ void mma3_f16(uint32_t d_tmem, uint64_t ah, uint64_t al, uint64_t bh, uint64_t bl,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p, t;\n setp.ne.b32 p, %5, 0;\n setp.ne.b32 t, %7, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %3, %6, p;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %4, %6, t;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %3, %6, t;\n}" ::"r"(d_tmem),
        "l"(ah), "l"(al), "l"(bh), "l"(bl), "r"(accumulate), "r"(idesc), "r"(1u)
        : "memory");
}

// The scores' operands as binary16 halves.  A row (a query row of Q, a key row of K) is scaled
// by a power of two that puts its largest magnitude in [2^14, 2^15); then hi = fp16(x*s) and
// lo = fp16(x*s - hi) are both normal binary16 values for every element within 2^28 of that
// largest one, and hi + lo carries x*s to about 2^-22 relative -- the accuracy of the TF32
// split, at twice the K of a TF32 instruction.  The scale is exact and undone in fp32 on S.
// Returns the factor 1/s (1 for a zero row).
__device__ __forceinline__ float f16_row_scale(float amax, float &s) {
    const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xff) - 127;  // floor(log2(amax))
    int sh = amax > 0.0f ? 14 - ex : 0;
    sh = sh > 126 ? 126 : (sh < -126 ? -126 : sh);
    s = __uint_as_float(static_cast<uint32_t>(sh + 127) << 23);
    return __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
}

// Eight scaled values -> eight hi and eight lo binary16 values (16 bytes each).
__device__ __forceinline__ void f16_split8(const float (&x)[8], float s, uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = x[2 * i] * s, b = x[2 * i + 1] * s;
        const __half ah = __float2half_rn(a), bh = __float2half_rn(b);
        const __half al = __float2half_rn(a - __half2float(ah)), bl = __float2half_rn(b - __half2float(bh));
        const __half2 hh = __halves2half2(ah, bh), ll = __halves2half2(al, bl);
        h[i] = *reinterpret_cast<const uint32_t *>(&hh);
        l[i] = *reinterpret_cast<const uint32_t *>(&ll);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Byte offset of the 16-byte chunk holding binary16 elements 8c..8c+7 of `row` in a 64-column
// SW128 slab (128-byte rows).
__device__ __forceinline__ uint32_t sw128_off16(int row, int c) {
    return static_cast<uint32_t>(row) * 128u + ((static_cast<uint32_t>(c) ^ static_cast<uint32_t>(row & 7)) << 4);
}

__device__ __forceinline__ void mma3_tf32(uint32_t d_tmem, uint64_t ah, uint64_t al, uint64_t bh, uint64_t bl,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p, t;\n setp.ne.b32 p, %5, 0;\n setp.ne.b32 t, %7, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %3, %6, p;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %4, %6, t;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %2, %3, %6, t;\n}" ::"r"(d_tmem),
        "l"(ah), "l"(al), "l"(bh), "l"(bl), "r"(accumulate), "r"(idesc), "r"(1u)
        : "memory");
}

__device__ __forceinline__ void mma_commit(unsigned long long *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32]) {
    uint32_t u[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]),
          "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]),
          "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]),
          "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __uint_as_float(u[i]);
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Byte offset of element (row, col) of a K-major SW128 slab (col < 32 fp32).
__device__ __forceinline__ uint32_t sw128_off(int row, int col) {
    return static_cast<uint32_t>(row) * 128u +
           ((static_cast<uint32_t>(col >> 2) ^ static_cast<uint32_t>(row & 7)) << 4) +
           static_cast<uint32_t>(col & 3) * 4u;
}

struct PParams {
    float *out;
    const void *k_reg, *v_reg;  // fp32, binary16 or Q8_0 rows (only fp32 K is read by TMA)
    long long row_bytes;        // Q8_0: bytes of a region row
    const int32_t *pos;
    int32_t *err;
    int nt, nh, nk, hd, cap, W;
    int n_qt, n_kc, kc_tiles;  // query tiles, key chunks per query tile, key tiles per chunk
    float scale_log2;
    float *ws_o, *ws_ml;       // chunk partials: o as [.., d/4][row] of float4, (m, l) as [.., 2][row]
    int *ws_ticket;            // one per (query tile, head)
    int *ws_tag;               // the workspace's layout tag (its control block), null without one
    int ws_key;                // this call's layout
};

// Round to the nearest TF32 value (10 explicit mantissa bits), ties away from zero: half a TF32
// unit (bit 12) is added to the magnitude's bit pattern and the 13 low bits are cleared; a
// carry moves into the exponent as it should.  The same result as cvt.rna.tf32.f32 for every
// finite input, on the integer pipe instead of the conversion unit.
__device__ __forceinline__ float tf32_rna(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo) {
    hi = tf32_rna(x);
    lo = tf32_rna(x - hi);
}

// Four consecutive region elements as fp32 (binary16 converts exactly).
__device__ __forceinline__ float4 ld4(const float *p, int i4) { return reinterpret_cast<const float4 *>(p)[i4]; }
__device__ __forceinline__ float4 ld4(const __half *p, int i4) {
    const uint2 u = reinterpret_cast<const uint2 *>(p)[i4];
    const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 y = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(x.x, x.y, y.x, y.y);
}

// The (query tile, key chunk) pair of pair index idx.  Pairs with kc <= qt come first (chunk
// slowest), then the others: in a causal prefill from position 0 with chunks as long as query
// tiles, the first set is exactly the pairs with keys, so every CTA with work is in the first
// wave and no CTA with work waits behind ones that leave at once.  (Any order is correct; this
// one only decides which CTAs start first.)
__device__ __forceinline__ void pair_of(int idx, int n_qt, int n_kc, int &qt, int &kc) {
    int base = 0;
    for (int c = 0; c < n_kc && c < n_qt; ++c) {  // kc <= qt: qt = c .. n_qt-1
        const int cnt = n_qt - c;
        if (idx < base + cnt) {
            kc = c;
            qt = c + (idx - base);
            return;
        }
        base += cnt;
    }
    for (int c = 1; c < n_kc; ++c) {  // kc > qt: qt = 0 .. min(c, n_qt)-1
        const int cnt = c < n_qt ? c : n_qt;
        if (idx < base + cnt) {
            kc = c;
            qt = idx - base;
            return;
        }
        base += cnt;
    }
    kc = n_kc;  // idx past the last pair: no work
    qt = 0;
}

constexpr int kStepMaxQt = 64;  // query tiles (nt <= 8192) the items are enumerated over

struct StepParams {
    float *q, *k;           // [nt, nh, hd], [nt, nk, hd_kv]: rotated in place
    const float *v;         // [nt, W]
    void *k_st, *v_st;      // the regions (written at pos; the items read them as a.k_reg, a.v_reg)
    int style;              // 0: pairs (i, i + hd/2); 1: pairs (2i, 2i + 1)
    float *xn;              // [nt, n_embd] RMSNorm output
    const float *hx, *gain; // [nt, n_embd], [n_embd] (gain nullable)
    int n_embd, norm_vec;   // norm_vec: float4 rows (n_embd % 4 == 0, 16-byte aligned rows and gain)
    float eps;
    int *bar;               // grid barrier: arrivals, departures (zero between launches), then
                            // the workspace's control block (its layout tag at bar[kWsTag])
};


// A CTA of the fused step counts its departure from the grid barrier once it has left the
// wait; the last to depart zeroes both counts for the next launch.
__device__ __forceinline__ void step_depart(const StepParams &x, int key) {
    const int old = atomicAdd(x.bar + kWsBarDepart, 1);
    if (old == static_cast<int>(gridDim.x) - 1) {
        x.bar[kWsBarArrive] = 0;
        x.bar[kWsBarDepart] = 0;
        // the workspace now holds this layout (a tag a timed-out item has poisoned stays so)
        const int tag = ld_relaxed(x.bar + kWsTag);
        if (tag != kWsPoison) atomicCAS(x.bar + kWsTag, tag, key);
    }
}

// One work item: query tile qt of head h against key chunk kc (tiles tile0 .. tile0 + n_tiles - 1
// of the keys), by every role of the CTA; its TMEM and mbarriers are ready (barriers in their
// first phase).  lmax: the widest window among the tile's tokens; L_t: this thread's row window
// (-1: the softmax threads read their positions themselves, while the Q tile is copied).
struct Item {
    int h, hk, qt, kc, t0, L_t, lmax, n_act, tile0, n_tiles;
    uint32_t tmem;
    const StepParams *dep;  // fused step: this CTA departs the grid barrier during this item
    int ws_tag;             // thread 0: the workspace's tag as the call found it (checked before
                            // a ticket is taken; the fused step checked it before its barrier)
};

// fp32 regions: K tiles arrive by TMA into kh and the staging warps convert them into kl.
// binary16 and Q8_0 regions: the staging warps read the K tile themselves, converting.
template <int HDKV, typename T>
__device__ __forceinline__ void attend(Smem<HDKV> &sm, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                       const PParams &a, const Item &it) {
    constexpr bool kTmaK = std::is_same<T, float>::value;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = it.h, hk = it.hk, qt = it.qt, kc = it.kc, t0 = it.t0, lmax = it.lmax;
    int L_t = it.L_t;
    const int n_act = it.n_act, tile0 = it.tile0, n_tiles = it.n_tiles;
    const uint32_t tmem = it.tmem;
    volatile int *abort_flag = &sm.abort_flag;
    constexpr uint32_t kQBytes = BM * HDKV * 4, kKBytes = BN * HDKV * 4;

    constexpr int NB = Smem<HDKV>::NB;
    constexpr int NP = Smem<HDKV>::NP;
    if (warp == kProducerWarp) {
        if (lane == 0 && n_tiles > 0) {
            mbar_expect_tx(&sm.bar_q, kQBytes);
#pragma unroll
            for (int c = 0; c < HDKV / 32; ++c) tma_load_2d(sm.qh[c], &tm_q, h * a.hd + 32 * c, t0, &sm.bar_q);
            auto load_k = [&](int j) {  // key tile j -> buffer j % NB
                const int b = j % NB;
                mbar_expect_tx(&sm.bar_k[b], kKBytes);
#pragma unroll
                for (int c = 0; c < HDKV / 32; ++c)
                    tma_load_2d(sm.kh[b][c], &tm_k, hk * HDKV + 32 * c, (tile0 + j) * BN, &sm.bar_k[b]);
            };
            if (kTmaK)
                for (int j = 0; j < NB && j < n_tiles; ++j) load_k(j);
            // Descriptors of the binary16 slabs of Q and of every K buffer (64 columns, 128-byte
            // rows; hi slabs then lo slabs), built once: a K step of 16 (32 bytes) moves the
            // start-address field (address / 16) by 2 within a 1024-aligned slab
            uint64_t dq[2][HDKV / 64], dk[NB][2][HDKV / 64];
#pragma unroll
            for (int c = 0; c < HDKV / 64; ++c) {
                const uint32_t qb = su32(&sm.ql[0][0]);
                dq[0][c] = sw128_desc(qb + c * (BM * 128));
                dq[1][c] = sw128_desc(qb + (HDKV / 64 + c) * (BM * 128));
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const uint32_t kb = su32(&sm.kl[b][0][0]);
                    dk[b][0][c] = sw128_desc(kb + c * (BN * 128));
                    dk[b][1][c] = sw128_desc(kb + (HDKV / 64 + c) * (BN * 128));
                }
            }
            constexpr uint32_t kIdS = f16_idesc(BM, BN);
            // S(j) = Q K(j)^T into S buffer j % 2 (Q and K tile j converted by then)
            auto issue_s = [&](int j) {
                const int b = j % NB;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < HDKV / 16; ++kk) {
                    const uint64_t o = 2 * (kk & 3);
                    const int c = kk >> 2;
                    // (buffer chosen by selects: a run-time index would move the array to local memory)
                    const uint64_t kh = (NB == 2 && b) ? dk[NB - 1][0][c] : dk[0][0][c];
                    const uint64_t kl = (NB == 2 && b) ? dk[NB - 1][1][c] : dk[0][1][c];
                    mma3_f16(tmem + s_col(j), dq[0][c] + o, dq[1][c] + o, kh + o, kl + o, kIdS, kk > 0);
                }
                mma_commit(&sm.bar_s[j & 1]);
            };
            bool ok = mbar_wait(&sm.bar_qs, 0, abort_flag, a.err) && mbar_wait(&sm.bar_kk[0], 0, abort_flag, a.err);
            if (ok) issue_s(0);
            for (int i = 0; ok && i < n_tiles; ++i) {
                // K buffer i % NB is free once S(i) is complete: the copy of key tile i + NB
                if (kTmaK && i + NB < n_tiles) {
                    if (!mbar_wait(&sm.bar_s[i & 1], (i >> 1) & 1, abort_flag, a.err)) break;
                    load_k(i + NB);
                }
                // S(i+1) ahead of O_t(i): its S buffer last held S(i-1), read before P(i-1) was
                // published
                if (i + 1 < n_tiles) {
                    const int j = i + 1;
                    if (j >= 2 && !mbar_wait(&sm.bar_p[j & 1], ((j - 2) >> 1) & 1, abort_flag, a.err)) break;
                    if (!mbar_wait(&sm.bar_kk[j % NB], (j / NB) & 1, abort_flag, a.err)) break;
                    issue_s(j);
                }
            }
        }
    } else if (warp == kPvWarp) {
        // O_t(i) = P(i) V(i) into O buffer i % 2 once P(i) is published and V^T(i) staged, from
        // a second thread: one thread issues a tensor-core instruction only every ~35-50 ns, and
        // S(i+1) and O_t(i) need not wait behind each other's issue
        if (lane == 0 && it.dep) step_depart(*it.dep, a.ws_key);  // (P(0) is microseconds away)
        if (lane == 0 && n_tiles > 0) {
            uint64_t dp[NP][2][BN / 32], dv[NB][2][BN / 32];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
#pragma unroll
                for (int b = 0; b < NP; ++b) {
                    dp[b][0][c] = sw128_desc(su32(sm.ph[b][c]));
                    dp[b][1][c] = sw128_desc(su32(sm.pl[b][c]));
                }
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    dv[b][0][c] = sw128_desc(su32(sm.vh[b][c]));
                    dv[b][1][c] = sw128_desc(su32(sm.vl[b][c]));
                }
            }
            constexpr uint32_t kIdO = tf32_idesc(BM, HDKV);
            for (int i = 0; i < n_tiles; ++i) {
                if (!mbar_wait(&sm.bar_p[i & 1], (i >> 1) & 1, abort_flag, a.err)) break;
                if (!mbar_wait(&sm.bar_vv[i % NB], (i / NB) & 1, abort_flag, a.err)) break;
                tc_fence_after();
                const int b = i % NB, pb = i % NP;
#pragma unroll
                for (int kk = 0; kk < BN / 8; ++kk) {
                    const uint64_t o = 2 * (kk & 3);
                    const int c = kk >> 2;
                    const uint64_t ph = (NP == 2 && pb) ? dp[NP - 1][0][c] : dp[0][0][c];
                    const uint64_t pl = (NP == 2 && pb) ? dp[NP - 1][1][c] : dp[0][1][c];
                    const uint64_t vh = (NB == 2 && b) ? dv[NB - 1][0][c] : dv[0][0][c];
                    const uint64_t vl = (NB == 2 && b) ? dv[NB - 1][1][c] : dv[0][1][c];
                    mma3_tf32(tmem + o_col<HDKV>(i), ph + o, pl + o, vh + o, vl + o, kIdO, kk > 0);
                }
                mma_commit(&sm.bar_o[i & 1]);
            }
        }
    } else if (warp >= kStageWarp0) {
        // staging: K tiles into scaled binary16 halves, V tiles transposed and split into TF32 (K-major)
        const int st = tid - (kSoftThreads + 32);  // 0 .. kStageThreads-1
        const int vk = st & (BN - 1), vq = st / BN;  // key of the tile, half of the dims
        constexpr int kV4 = HDKV / 8;                // float4 of a V row per thread
        // This thread's slice of the next V tile is loaded one tile ahead, so its latency
        // overlaps the current tile's work.
        float4 vnext[kV4];
        // element group d4 (4 values) of this kv head in region row `key` (dequantized for Q8_0)
        auto kv4 = [&](const void *reg, int key, int d4) -> float4 {
            if constexpr (std::is_same<T, Q8>::value) {
                const unsigned char *row = static_cast<const unsigned char *>(reg) + static_cast<size_t>(key) * a.row_bytes;
                return ld4_q8(row, a.W, hk * (HDKV / 4) + d4);
            } else {
                return ld4(static_cast<const T *>(reg) + static_cast<size_t>(key) * a.W + hk * HDKV, d4);
            }
        };
        auto load_v = [&](int tile) {
            const int key = tile * BN + vk;
#pragma unroll
            for (int c = 0; c < kV4; ++c)
                vnext[c] = key < lmax ? kv4(a.v_reg, key, vq * kV4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        };
        // K tile j -> buffer j % NB as scaled binary16 hi + lo halves, a key row per pair of
        // adjacent lanes (each half the row; the row's largest magnitude by one shuffle), and
        // the key's unscale factor into slot j % 4 (fp32 K: read from its TMA copy; binary16 and
        // Q8_0: read and converted here; keys past the widest window are zero)
        auto stage_k = [&](int j) -> bool {
            const int b = j % NB;
            const int key = st >> 1, h2 = st & 1;  // key of the tile, half of the row
            constexpr int kH4 = HDKV / 8;          // float4 of half a row
            float4 kv[kH4];
            // (the pair exchange below is a warp shuffle: the warp leaves together or not at all)
            if (kTmaK) {
                if (!__all_sync(0xffffffffu, mbar_wait(&sm.bar_k[b], (j / NB) & 1, abort_flag, a.err))) return false;
#pragma unroll
                for (int c = 0; c < kH4; ++c) {
                    const int d4 = h2 * kH4 + c;
                    kv[c] = *reinterpret_cast<const float4 *>(
                        reinterpret_cast<const unsigned char *>(sm.kh[b][d4 >> 3]) + sw128_off(key, 4 * (d4 & 7)));
                }
            } else {
                // the buffer last held key tile j - NB: S(j - NB) must have read it
                if (j >= NB) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&sm.bar_s[(j - NB) & 1], ((j - NB) >> 1) & 1, abort_flag, a.err)))
                        return false;
                    tc_fence_after();
                }
                const int gkey = (tile0 + j) * BN + key;
#pragma unroll
                for (int c = 0; c < kH4; ++c)
                    kv[c] = gkey < lmax ? kv4(a.k_reg, gkey, h2 * kH4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float amax = 0.0f;
#pragma unroll
            for (int c = 0; c < kH4; ++c)
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(kv[c].x), fabsf(kv[c].y)), fmaxf(fabsf(kv[c].z), fabsf(kv[c].w))));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            float ksc;
            const float kinv = f16_row_scale(amax, ksc);
            unsigned char *k16 = reinterpret_cast<unsigned char *>(&sm.kl[b][0][0]);
#pragma unroll
            for (int c = 0; c < kH4 / 2; ++c) {
                const float x[8] = {kv[2 * c].x, kv[2 * c].y, kv[2 * c].z, kv[2 * c].w,
                                    kv[2 * c + 1].x, kv[2 * c + 1].y, kv[2 * c + 1].z, kv[2 * c + 1].w};
                uint4 hi, lo;
                f16_split8(x, ksc, hi, lo);
                const int g = h2 * (kH4 / 2) + c;  // group of 8 binary16 elements in the row
                const uint32_t off = static_cast<uint32_t>(g >> 3) * (BN * 128) + sw128_off16(key, g & 7);
                *reinterpret_cast<uint4 *>(k16 + off) = hi;
                *reinterpret_cast<uint4 *>(k16 + (HDKV / 64) * (BN * 128) + off) = lo;
            }
            if (h2 == 0) sm.ks[j & 3][key] = kinv * a.scale_log2;  // exact: kinv is a power of two
            mbar_arrive(&sm.bar_ks[j & 3]);  // the factors, to the softmax threads (tile j + 4 needs P(j) first)
            fence_async_smem();  // split K -> visible to the tensor cores
            tc_fence_before();
            mbar_arrive(&sm.bar_kk[b]);
            return true;
        };
        // V tile j (held in vnext) -> V^T hi/lo in buffer j % NB, once O_t(j - NB) has read it
        auto stage_v = [&](int j) -> bool {
            const int b = j % NB;
            if (j >= NB) {
                if (!mbar_wait(&sm.bar_o[(j - NB) & 1], ((j - NB) >> 1) & 1, abort_flag, a.err)) return false;
                tc_fence_after();
            }
            unsigned char *vth = reinterpret_cast<unsigned char *>(sm.vh[b][vk >> 5]);
            unsigned char *vtl = reinterpret_cast<unsigned char *>(sm.vl[b][vk >> 5]);
#pragma unroll
            for (int c = 0; c < kV4; ++c) {
                const int d4 = vq * kV4 + c;
                const float vv[4] = {vnext[c].x, vnext[c].y, vnext[c].z, vnext[c].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float hi, lo;
                    split_tf32(vv[e], hi, lo);
                    const uint32_t off = sw128_off(4 * d4 + e, vk & 31);
                    *reinterpret_cast<float *>(vth + off) = hi;
                    *reinterpret_cast<float *>(vtl + off) = lo;
                }
            }
            fence_async_smem();  // V^T -> visible to the tensor cores
            tc_fence_before();
            mbar_arrive(&sm.bar_vv[b]);
            if (j + 1 < n_tiles) load_v(tile0 + j + 1);
            return true;
        };
        // K runs a tile ahead of V where there are two buffers (S(i+1) is issued before O_t(i));
        // with one buffer, K(i+1) can only land once S(i) is complete, so V(i) goes first.
        bool ok = n_tiles > 0;
        if (ok) {
            load_v(tile0);
            ok = stage_k(0);
        }
        for (int i = 0; ok && i < n_tiles; ++i) {
            if (NB == 2 && i + 1 < n_tiles && !stage_k(i + 1)) break;
            if (!stage_v(i)) break;
            if (NB == 1 && i + 1 < n_tiles && !stage_k(i + 1)) break;
        }
    } else {
        // softmax and epilogue: thread tid owns query row tid (TMEM lane tid)
        if (L_t < 0) {  // ("11 . Attention...", §3.2.4: vl = min(pos[t] + 1, nkv))
            const int p = t0 + tid < a.nt ? __ldg(a.pos + t0 + tid) : -1;
            L_t = p < 0 ? 0 : (p + 1 < a.cap ? p + 1 : a.cap);
        }
        const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float qinv = 1.0f;  // the factor undoing this query row's binary16 scale (a power of two)
        float o[HDKV];
#pragma unroll
        for (int d = 0; d < HDKV; ++d) o[d] = 0.0f;
        float m = -INFINITY, l = 0.0f;
        float corr_prev = 1.0f;  // the correction that goes with O_t(i-1)
        // o = o * c + O_t(j), from O buffer j % 2
        auto fold_o = [&](int j, float c) {
#pragma unroll
            for (int cc = 0; cc < HDKV / 32; ++cc) {
                float r[32];
                tmem_ld32(trow + o_col<HDKV>(j) + 32 * cc, r);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[32 * cc + e] = fmaf(o[32 * cc + e], c, r[e]);
            }
        };
        bool ok = n_tiles > 0;
        if (ok) ok = mbar_wait(&sm.bar_q, 0, abort_flag, a.err);
        if (ok) {
            // this thread's query row (row tid) into binary16 hi and lo halves, scaled
            auto q4 = [&](int d4) {  // fp32 elements 4*d4.. of the row, from the TMA slabs
                return *reinterpret_cast<const float4 *>(reinterpret_cast<const unsigned char *>(sm.qh[d4 >> 3]) +
                                                        sw128_off(tid, 4 * (d4 & 7)));
            };
            float amax = 0.0f;
#pragma unroll 8
            for (int d4 = 0; d4 < HDKV / 4; ++d4) {
                const float4 v = q4(d4);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
            float qs;
            qinv = f16_row_scale(amax, qs);
            unsigned char *q16 = reinterpret_cast<unsigned char *>(&sm.ql[0][0]);
#pragma unroll 4
            for (int g = 0; g < HDKV / 8; ++g) {
                const float4 u = q4(2 * g), w = q4(2 * g + 1);
                const float x[8] = {u.x, u.y, u.z, u.w, w.x, w.y, w.z, w.w};
                uint4 hi, lo;
                f16_split8(x, qs, hi, lo);
                const uint32_t off = static_cast<uint32_t>(g >> 3) * (BM * 128) + sw128_off16(tid, g & 7);
                *reinterpret_cast<uint4 *>(q16 + off) = hi;
                *reinterpret_cast<uint4 *>(q16 + (HDKV / 64) * (BM * 128) + off) = lo;
            }
            fence_async_smem();  // split Q -> visible to the tensor cores
            tc_fence_before();
            mbar_arrive(&sm.bar_qs);
        }
        // Per tile i: P(i) from S(i), published; then O_t(i-1) folded in while the tensor
        // cores form O_t(i) and S(i+1).
        for (int i = 0; ok && i < n_tiles; ++i) {
            const int j0 = (tile0 + i) * BN;
            if (!mbar_wait(&sm.bar_s[i & 1], (i >> 1) & 1, abort_flag, a.err) ||
                !mbar_wait(&sm.bar_ks[i & 3], (i >> 2) & 1, abort_flag, a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float r[32];
            tmem_ld32(trow + s_col(i), r);
            // r * ks: the key's binary16 scale undone and scale * log2(e) applied (one rounding);
            // the query row's scale, a power of two, is undone exactly on the max and inside the
            // exponent's fused multiply-add
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
                const float4 f = reinterpret_cast<const float4 *>(sm.ks[i & 3])[e4];
                r[4 * e4] *= f.x;
                r[4 * e4 + 1] *= f.y;
                r[4 * e4 + 2] *= f.z;
                r[4 * e4 + 3] *= f.w;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (j0 + e < L_t) mx = fmaxf(mx, r[e]);
            const float m_new = fmaxf(m, mx * qinv);
            const bool none = (m_new == -INFINITY);  // no key visible to this row yet
            const float corr = none ? 1.0f : ex2_approx(m - m_new);
            // one P buffer: O_t(i-1) must have read P(i-1) before it is overwritten
            if (NP == 1 && i > 0 && !mbar_wait(&sm.bar_o[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag, a.err)) {
                ok = false;
                break;
            }
            float ps = 0.0f;
            unsigned char *pph = reinterpret_cast<unsigned char *>(sm.ph[i % NP][0]);
            unsigned char *ppl = reinterpret_cast<unsigned char *>(sm.pl[i % NP][0]);
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
                float4 wh, wl;
                float *whv = reinterpret_cast<float *>(&wh), *wlv = reinterpret_cast<float *>(&wl);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = j0 + 4 * e4 + e;
                    const float pe = (!none && j < L_t) ? ex2_approx(fmaf(r[4 * e4 + e], qinv, -m_new)) : 0.0f;
                    split_tf32(pe, whv[e], wlv[e]);
                    ps += pe;
                }
                *reinterpret_cast<float4 *>(pph + sw128_off(tid, 4 * e4)) = wh;
                *reinterpret_cast<float4 *>(ppl + sw128_off(tid, 4 * e4)) = wl;
            }
            l = fmaf(l, corr, ps);
            m = m_new;
            fence_async_smem();  // P hi/lo -> visible to the tensor cores
            tc_fence_before();
            mbar_arrive(&sm.bar_p[i & 1]);
            if (i > 0) {
                if (!mbar_wait(&sm.bar_o[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                fold_o(i - 1, corr_prev);
                tc_fence_before();  // the O buffer is read before the next P lets O_t(i+1) overwrite it
            }
            corr_prev = corr;
        }
        if (ok) {  // the last tile's O_t
            const int j = n_tiles - 1;
            if (mbar_wait(&sm.bar_o[j & 1], (j >> 1) & 1, abort_flag, a.err)) {
                tc_fence_after();
                fold_o(j, corr_prev);
            }
        }
        bool write_out = true;
        if (n_act > 1) {
            // more than one chunk of keys: publish this chunk's (m, l, o) per row; the last
            // chunk of the (query tile, head) to arrive folds them (an atomic ticket, no wait)
            const size_t blk = (static_cast<size_t>(qt) * a.nh + h) * a.n_kc;
            float *po = a.ws_o + (blk + kc) * HDKV * BM;
            float *pml = a.ws_ml + (blk + kc) * 2 * BM;
#pragma unroll
            for (int d4 = 0; d4 < HDKV / 4; ++d4)  // float4 of dims, rows adjacent: coalesced vector access
                reinterpret_cast<float4 *>(po)[d4 * BM + tid] =
                    make_float4(o[4 * d4], o[4 * d4 + 1], o[4 * d4 + 2], o[4 * d4 + 3]);
            pml[tid] = m;
            pml[BM + tid] = l;
            named_sync(1, kSoftThreads);
            if (tid == 0) {
                if (it.ws_tag == 0 || it.ws_tag == a.ws_key) {
                    if (it.ws_tag == 0) atomicCAS(a.ws_tag, 0, a.ws_key);  // a fresh workspace takes this layout
                    int old;
                    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                                 : "=r"(old)
                                 : "l"(a.ws_ticket + static_cast<size_t>(qt) * a.nh + h)
                                 : "memory");
                    sm.lmax = (old == n_act - 1) ? -1 : 0;  // reuse as the "last" flag
                } else {
                    // another layout's workspace: its tickets are not this call's to trust
                    flag_error(a.err, MINF_ERRBIT_WORKSPACE);
                    sm.lmax = 0;
                }
            }
            named_sync(1, kSoftThreads);
            write_out = sm.lmax == -1;
            if (write_out) {
                // The other chunks' partial outputs are bulk-copied into the free shared memory,
                // kN chunks at a time, all copies of a batch in flight together; meanwhile the
                // (max, sum) pairs of every chunk come in one round trip, so the combined max and
                // every chunk's factor are known when the outputs land.  Then each chunk's
                // outputs, scaled, are added in chunk order (at most 16 chunks a tile).
                using MS = MergeSlots<HDKV>;
                constexpr int kMaxKc = 16;
                unsigned char *slots = reinterpret_cast<unsigned char *>(&sm.qh[0][0]) + MS::kStg;
                auto issue_batch = [&](int c0) {  // chunks c0 .. c0 + kN - 1 other than kc
                    if (tid != 0 || *abort_flag) return;
                    uint32_t bytes = 0;
                    for (int c = c0; c < c0 + MS::kN && c < n_act; ++c)
                        if (c != kc) bytes += static_cast<uint32_t>(MS::kPart);
                    if (bytes == 0) return;
                    fence_async_global();  // the partials acquired through the ticket, to the copy engine
                    mbar_expect_tx(&sm.bar_m, bytes);
                    for (int c = c0; c < c0 + MS::kN && c < n_act; ++c)
                        if (c != kc)
                            bulk_load(slots + (c - c0) * MS::kPart, a.ws_o + (blk + c) * HDKV * BM,
                                      static_cast<uint32_t>(MS::kPart), &sm.bar_m);
                };
                issue_batch(0);
                float mcs[kMaxKc], lcs[kMaxKc];
#pragma unroll
                for (int c = 0; c < kMaxKc; ++c) {
                    const bool use = c < n_act && c != kc;
                    const float *qml = a.ws_ml + (blk + c) * 2 * BM;
                    mcs[c] = use ? __ldcg(qml + tid) : -INFINITY;
                    lcs[c] = use ? __ldcg(qml + BM + tid) : 0.0f;
                }
                float M = m;
#pragma unroll
                for (int c = 0; c < kMaxKc; ++c) M = fmaxf(M, mcs[c]);
                const float fa = m == -INFINITY ? 0.0f : ex2_approx(m - M);
                l *= fa;
                float fbs[kMaxKc];  // every chunk's factor (the sum takes them in chunk order)
#pragma unroll
                for (int c = 0; c < kMaxKc; ++c) {
                    fbs[c] = mcs[c] == -INFINITY ? 0.0f : ex2_approx(mcs[c] - M);
                    if (c < n_act && c != kc) l = fmaf(lcs[c], fbs[c], l);
                }
#pragma unroll
                for (int d = 0; d < HDKV; ++d) o[d] *= fa;
                uint32_t mph = 0;  // phase of bar_m
#pragma unroll 1
                for (int c0 = 0; c0 < kMaxKc; c0 += MS::kN) {
                    if (c0 >= n_act) break;
                    const int cnt = min(MS::kN, n_act - c0);
                    if (cnt > 1 || c0 != kc) {  // the batch holds a chunk other than kc: copies to wait for
                        // (one decision for every row: the threads meet at named barriers below)
                        if (!named_all(1, kSoftThreads, mbar_wait(&sm.bar_m, mph, abort_flag, a.err))) break;
                        mph ^= 1u;
                    }
#pragma unroll
                    for (int cc = 0; cc < MS::kN; ++cc) {
                        const int c = c0 + cc;
                        if (c < kMaxKc && c < n_act && c != kc) {
                            const float fb = fbs[c];
                            const float4 *qo = reinterpret_cast<const float4 *>(slots + cc * MS::kPart);
#pragma unroll
                            for (int d4 = 0; d4 < HDKV / 4; ++d4) {
                                const float4 x = qo[d4 * BM + tid];
                                o[4 * d4] = fmaf(x.x, fb, o[4 * d4]);
                                o[4 * d4 + 1] = fmaf(x.y, fb, o[4 * d4 + 1]);
                                o[4 * d4 + 2] = fmaf(x.z, fb, o[4 * d4 + 2]);
                                o[4 * d4 + 3] = fmaf(x.w, fb, o[4 * d4 + 3]);
                            }
                        }
                    }
                    if (c0 + MS::kN < n_act) {  // every row has read the slots before they refill
                        named_sync(1, kSoftThreads);
                        issue_batch(c0 + MS::kN);
                    }
                }
                m = M;
                if (tid == 0) a.ws_ticket[static_cast<size_t>(qt) * a.nh + h] = 0;  // ready for reuse
            }
        }
        if (write_out) {  // the same in every softmax thread
            // Rows pass through shared memory (the Q slabs: every S has completed) so that each
            // warp writes whole output rows, which lie n_head*hd_kv floats apart.
            constexpr int kRS = MergeSlots<HDKV>::kRS;
            static_assert(BM * kRS <= 2 * HDKV * BM, "staging fits the Q slabs");
            float *stg = &sm.qh[0][0];
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
            for (int d4 = 0; d4 < HDKV / 4; ++d4)
                reinterpret_cast<float4 *>(stg + tid * kRS)[d4] =
                    make_float4(o[4 * d4] * inv, o[4 * d4 + 1] * inv, o[4 * d4 + 2] * inv, o[4 * d4 + 3] * inv);
            named_sync(1, kSoftThreads);
            constexpr int kF4 = HDKV / 4;       // float4 of a row
            constexpr int kRowsPer = 32 / kF4;  // rows a warp writes per instruction
            if (!*abort_flag)
#pragma unroll 4
                for (int r0 = warp * 32; r0 < warp * 32 + 32; r0 += kRowsPer) {
                    const int r = r0 + lane / kF4, c = lane % kF4;
                    if (t0 + r < a.nt)
                        reinterpret_cast<float4 *>(a.out + (static_cast<size_t>(t0 + r) * a.nh + h) * HDKV)[c] =
                            reinterpret_cast<const float4 *>(stg + r * kRS)[c];
                }
        }
    }
}

// One CTA per (query tile, key chunk, head) item.
template <int HDKV, typename T>
__global__ void __launch_bounds__(kThreadsP, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const PParams a) {
    extern __shared__ unsigned char smem_raw[];
    Smem<HDKV> &sm = *reinterpret_cast<Smem<HDKV> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTA -> (query tile, key chunk) pair and head, the head fastest (chunks past a tile's
    // widest window leave at once)
    const int h = blockIdx.x % a.nh;
    int qt, kc;
    pair_of(blockIdx.x / a.nh, a.n_qt, a.n_kc, qt, kc);
    const int t0 = qt * BM;
    const int g = a.nh / a.nk;
    const int hk = h / g;
    volatile int *abort_flag = &sm.abort_flag;

    if (tid == 0) {
        // One barrier per buffer, so that no role can complete a phase twice before another
        // role waits on it (every refill of a buffer waits on the consumer of its last phase).
        mbar_init(&sm.bar_q, 1);
        mbar_init(&sm.bar_qs, kSoftThreads);
        for (int b = 0; b < Smem<HDKV>::NB; ++b) {
            mbar_init(&sm.bar_k[b], 1);
            mbar_init(&sm.bar_kk[b], kStageThreads);
            mbar_init(&sm.bar_vv[b], kStageThreads);
        }
        for (int b = 0; b < 4; ++b) mbar_init(&sm.bar_ks[b], kStageThreads);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.bar_s[b], 1);
            mbar_init(&sm.bar_p[b], kSoftThreads);
            mbar_init(&sm.bar_o[b], 1);
        }
        mbar_init(&sm.bar_m, 1);
        sm.abort_flag = 0;
        sm.lmax = 0;
        mbar_init_fence();
    }
    // Nothing is read before the launch ahead of this one has finished: pos, q, the regions, the
    // workspace and the output may all be its outputs (a no-op without programmatic launch).
    gdc_wait();
    // The workspace's tag, checked before a ticket is taken (the load is in flight meanwhile).
    const int ws_tag0 = (tid == 0 && a.ws_tag) ? ld_relaxed(a.ws_tag) : 0;
    // this row's window ("11 . Attention...", §3.2.4: vl = min(pos[t] + 1, nkv), nkv <= n_ctx)
    int L_t = 0;
    const int t = t0 + tid;
    if (tid < kSoftThreads && t < a.nt) {
        const int p = __ldg(a.pos + t);
        L_t = p < 0 ? 0 : (p + 1 < a.cap ? p + 1 : a.cap);
        if ((p < 0 || p >= a.cap) && h == 0 && kc == 0) flag_error(a.err, MINF_ERRBIT_ATTN_POS);
    }
    __syncthreads();
    if (tid < kSoftThreads) {
        int mx = L_t;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) atomicMax(&sm.lmax, mx);
    }
    __syncthreads();
    const int lmax = sm.lmax;
    const int n_tiles_all = (lmax + BN - 1) / BN;
    const int n_act = (n_tiles_all + a.kc_tiles - 1) / a.kc_tiles;  // chunks with keys for this tile
    if (kc > 0 && kc >= n_act) return;  // nothing to do (chunk 0 always runs: it writes the output)
    const int tile0 = kc * a.kc_tiles;
    const int n_tiles = min(n_tiles_all - tile0, a.kc_tiles) > 0 ? min(n_tiles_all - tile0, a.kc_tiles) : 0;
    if (warp == kProducerWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(&sm.tmem_base)),
                     "r"(tmem_cols<HDKV>())
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    // The launch that follows may start now: this kernel writes no K/V rows (a following decode
    // kernel streams cached rows before its own wait), and every launch before it has completed.
    gdc_launch_dependents();
    const Item it = {h, hk, qt, kc, t0, L_t, lmax, n_act, tile0, n_tiles, tmem, nullptr, ws_tag0};
    attend<HDKV, T>(sm, tm_q, tm_k, a, it);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kProducerWarp) {
        if (*abort_flag && lane == 0) {
            // let copies and MMAs that may still be in flight finish before TMEM and shared memory go away
            const unsigned long long t0n = gtimer();
            while (gtimer() - t0n < kWaitBudgetNs / 4) {
            }
            if (a.ws_tag) *a.ws_tag = kWsPoison;  // a wait expired: refused until zero-filled
        }
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols<HDKV>())
                     : "memory");
    }
}

// ----------------------------------------------------------------------------- fused step
// The prefill layer step in one launch ("11 . Attention, vec ops, and the KV cache", §3.2.1 -
// §3.2.4: RMSNorm, RoPE on q and k at the tokens' positions, the K/V store, then the causal
// attention over the regions).  A grid of at most one CTA an SM, all resident together (a
// cooperative launch), first does the step's row work split over every thread of the grid; a
// grid barrier makes the rotated q and the stored rows visible to every CTA; then the CTAs take
// the (query tile, key chunk, head) items that have keys in turn, each as the per-item kernel
// does.  No second launch sits between two layer steps, and no CTA is spent on an empty item.

// Shared memory of the step beyond the items' own: the query tiles' widest windows and the
// prefix sums of their chunk counts (the item enumeration).
struct StepSmem {
    int lmq[kStepMaxQt];
    int pref[kStepMaxQt + 1];
};

// The row work of the step, spread over every thread of the grid.  The first warps take the
// RMSNorm rows (a warp a row); every other thread takes one unit at a time: a RoPE unit -- pair
// group j (pairs 4j .. 4j+3) of token t in up to kRopeHeads q heads or k heads, rotated in place,
// the k rows also stored at pos -- or kVPerUnit float4 of v, stored at pos.  A RoPE unit computes its
// four angles' sines and cosines once for its heads and loads all of its heads before it stores
// any, so that those loads are in flight together.  A pair group is two float4: elements
// i..i+3 and i+hd/2.. (style 0) or 8j..8j+7 (style 1).  The error bits are those of the
// separate RoPE + store launch.
constexpr int kRopeHeads = 8;
// float4 of v a unit copies: few enough units that a grid of one CTA an SM takes every RoPE and
// v unit of a 512-token step in one pass (a second unit a thread was the slowest CTAs' tail)
constexpr int kVPerUnit = 4;

struct RopeGroup {
    float4 u0[kRopeHeads], u1[kRopeHeads];
};

__device__ __forceinline__ void rope_group_load(RopeGroup &g, const StepParams &x, const float *base, int nheads,
                                                int hd, int j) {
    const int i0 = x.style == 0 ? 4 * j : 8 * j;
    const int i1 = x.style == 0 ? 4 * j + (hd >> 1) : 8 * j + 4;
#pragma unroll
    for (int e = 0; e < kRopeHeads; ++e)
        if (e < nheads) {
            const float *row = base + static_cast<size_t>(e) * hd;
            g.u0[e] = *reinterpret_cast<const float4 *>(row + i0);
            g.u1[e] = *reinterpret_cast<const float4 *>(row + i1);
        }
}

template <typename T>
__device__ __forceinline__ void rope_group_store(const RopeGroup &g, const StepParams &x, float *base, int nheads,
                                                 int hd, int j, const float *sn, const float *cs, T *reg_row) {
    const int i0 = x.style == 0 ? 4 * j : 8 * j;
    const int i1 = x.style == 0 ? 4 * j + (hd >> 1) : 8 * j + 4;
#pragma unroll
    for (int e = 0; e < kRopeHeads; ++e)
        if (e < nheads) {
            float4 w0 = g.u0[e], w1 = g.u1[e];
            if (x.style == 0) {  // pair c: (w0[c], w1[c])
                rope_pair_sc(w0.x, w1.x, sn[0], cs[0]);
                rope_pair_sc(w0.y, w1.y, sn[1], cs[1]);
                rope_pair_sc(w0.z, w1.z, sn[2], cs[2]);
                rope_pair_sc(w0.w, w1.w, sn[3], cs[3]);
            } else {  // pairs (w0.x, w0.y), (w0.z, w0.w), (w1.x, w1.y), (w1.z, w1.w)
                rope_pair_sc(w0.x, w0.y, sn[0], cs[0]);
                rope_pair_sc(w0.z, w0.w, sn[1], cs[1]);
                rope_pair_sc(w1.x, w1.y, sn[2], cs[2]);
                rope_pair_sc(w1.z, w1.w, sn[3], cs[3]);
            }
            float *row = base + static_cast<size_t>(e) * hd;
            *reinterpret_cast<float4 *>(row + i0) = w0;
            *reinterpret_cast<float4 *>(row + i1) = w1;
            if (reg_row) {
                const size_t b4 = static_cast<size_t>(e) * (hd >> 2);
                put4(reg_row, b4 + (i0 >> 2), w0);
                put4(reg_row, b4 + (i1 >> 2), w1);
            }
        }
}

template <typename T>
__device__ __forceinline__ void step_rows(const PParams &a, const StepParams &x, const float *fq, const float *fk) {
    const int warps = gridDim.x * (blockDim.x >> 5);
    const int norm_warps = a.nt < warps / 2 ? a.nt : warps / 2;
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw < norm_warps) {
        for (int r = gw; r < a.nt; r += norm_warps) {  // RMSNorm: a warp per row
            if (x.norm_vec)
                rms_norm_row<true>(x.xn, x.hx, x.gain, r, x.n_embd, x.eps);
            else
                rms_norm_row<false>(x.xn, x.hx, x.gain, r, x.n_embd, x.eps);
        }
        return;
    }
    const int G = (warps - norm_warps) * 32;
    const int gt = (gw - norm_warps) * 32 + (threadIdx.x & 31);
    const int hd_kv = a.W / a.nk;
    const int gq = a.hd >> 3, gk = hd_kv >> 3;  // pair groups of a head
    const int bq = (a.nh + kRopeHeads - 1) / kRopeHeads, bk = (a.nk + kRopeHeads - 1) / kRopeHeads;
    const int per_tok = gq * bq + gk * bk;  // RoPE units of a token
    const int nvu = a.W >> 2;                          // float4 of a v row
    const int nvg = (nvu + kVPerUnit - 1) / kVPerUnit;  // v units of a token
    const int n_rope = a.nt * per_tok;  // the host keeps nt * (per_tok + nvu) below 2^30
    const int total = n_rope + a.nt * nvg;
    for (int u = gt; u < total; u += G) {
        if (u >= n_rope) {  // kVPerUnit float4 of v (loaded together with their position)
            const int w = u - n_rope;
            const int t = w / nvg, c0 = (w - t * nvg) * kVPerUnit;
            const int p = __ldg(a.pos + t);
            const float4 *vr = reinterpret_cast<const float4 *>(x.v) + static_cast<size_t>(t) * nvu;
            float4 vv[kVPerUnit];
#pragma unroll
            for (int e = 0; e < kVPerUnit; ++e)
                if (c0 + e < nvu) vv[e] = vr[c0 + e];
            if (p < 0 || p >= a.cap) {
                if (c0 == 0) flag_error(a.err, MINF_ERRBIT_STORE_POS);
                continue;
            }
#pragma unroll
            for (int e = 0; e < kVPerUnit; ++e)
                if (c0 + e < nvu) put4(static_cast<T *>(x.v_st), static_cast<size_t>(p) * nvu + c0 + e, vv[e]);
            continue;
        }
        const int t = u / per_tok;
        int r = u - t * per_tok;
        const bool is_q = r < gq * bq;
        if (!is_q) r -= gq * bq;
        const int ng = is_q ? gq : gk;
        const int b = r / ng, j = r - b * ng;  // head batch, pair group
        const int nheads = is_q ? a.nh : a.nk, hd = is_q ? a.hd : hd_kv;
        const int h0 = b * kRopeHeads;
        const int nb = nheads - h0 < kRopeHeads ? nheads - h0 : kRopeHeads;
        float *base = (is_q ? x.q + static_cast<size_t>(t) * a.nh * a.hd : x.k + static_cast<size_t>(t) * a.W) +
                      static_cast<size_t>(h0) * hd;
        // the heads' pairs and the position in flight together
        const int p = __ldg(a.pos + t);
        RopeGroup grp;
        rope_group_load(grp, x, base, nb, hd, j);
        if (p < 0) {
            if (is_q && r == 0) flag_error(a.err, MINF_ERRBIT_ROPE_POS);
            continue;
        }
        const float pf = static_cast<float>(p);
        const float *f = is_q ? fq : fk;
        float sn[4], cs[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) sincosf(__fmul_rn(pf, f[4 * j + c]), &sn[c], &cs[c]);
        T *reg = (!is_q && p < a.cap) ? static_cast<T *>(x.k_st) + static_cast<size_t>(p) * a.W + h0 * hd : nullptr;
        rope_group_store<T>(grp, x, base, nb, hd, j, sn, cs, reg);
    }
}

template <int HDKV, typename T>
__global__ void __launch_bounds__(kThreadsP, 1)
    prefill_step_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const PParams a, const StepParams x, const RopeTable tq, const RopeTable tk) {
    extern __shared__ unsigned char smem_raw[];
    Smem<HDKV> &sm = *reinterpret_cast<Smem<HDKV> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    StepSmem &ss = *reinterpret_cast<StepSmem *>(reinterpret_cast<unsigned char *>(&sm) + sizeof(Smem<HDKV>));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort_flag = &sm.abort_flag;
    auto init_barriers = [&](bool again) {  // thread 0
        unsigned long long *bars[] = {&sm.bar_q, &sm.bar_qs, &sm.bar_m};
        for (unsigned long long *b : bars)
            if (again) mbar_inval(b);
        if (again) {
            for (int b = 0; b < Smem<HDKV>::NB; ++b) {
                mbar_inval(&sm.bar_k[b]);
                mbar_inval(&sm.bar_kk[b]);
                mbar_inval(&sm.bar_vv[b]);
            }
            for (int b = 0; b < 4; ++b) mbar_inval(&sm.bar_ks[b]);
            for (int b = 0; b < 2; ++b) {
                mbar_inval(&sm.bar_s[b]);
                mbar_inval(&sm.bar_p[b]);
                mbar_inval(&sm.bar_o[b]);
            }
        }
        mbar_init(&sm.bar_q, 1);
        mbar_init(&sm.bar_qs, kSoftThreads);
        for (int b = 0; b < Smem<HDKV>::NB; ++b) {
            mbar_init(&sm.bar_k[b], 1);
            mbar_init(&sm.bar_kk[b], kStageThreads);
            mbar_init(&sm.bar_vv[b], kStageThreads);
        }
        for (int b = 0; b < 4; ++b) mbar_init(&sm.bar_ks[b], kStageThreads);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.bar_s[b], 1);
            mbar_init(&sm.bar_p[b], kSoftThreads);
            mbar_init(&sm.bar_o[b], 1);
        }
        mbar_init(&sm.bar_m, 1);
        mbar_init_fence();
    };
    if (tid == 0) {
        init_barriers(false);
        sm.abort_flag = 0;
    }
    // the angular-speed tables, into shared memory the items overwrite later
    float *fq = &sm.kh[0][0][0], *fk = fq + kMaxHalf;
    for (int i = tid; i < kMaxHalf; i += kThreadsP) {
        fq[i] = tq.f[i];
        fk[i] = tk.f[i];
    }
    if (warp == kProducerWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(&sm.tmem_base)),
                     "r"(tmem_cols<HDKV>())
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    gdc_wait();  // every input (pos included) and the workspace, only after the launch before this one
    // The workspace's control block as the call found it (checked before the grid barrier, the
    // loads in flight meanwhile): the tag of any layout will do -- this step zeroes its own
    // tickets -- but not a poisoned or garbage one, and no CTA can have departed yet.
    int ctl_tag = 0, ctl_dep = 0;
    if (tid == 0) {
        ctl_tag = ld_relaxed(x.bar + kWsTag);
        ctl_dep = ld_relaxed(x.bar + kWsBarDepart);
    }
    // This call's merge tickets start at zero whatever an earlier call of another shape left in
    // their words (its partial outputs, say): no item takes a ticket before the grid barrier.
    if (a.ws_ticket)
        for (int i = blockIdx.x * kThreadsP + tid; i < a.n_qt * a.nh; i += gridDim.x * kThreadsP) a.ws_ticket[i] = 0;

    // Every query tile's widest window ("11 . Attention...", §3.2.4: vl = min(pos[t] + 1, nkv)),
    // in every CTA (the positions are few): the first tiles' positions are loaded before the row
    // work and folded after it, so that the loads are in flight meanwhile.
    if (tid < a.n_qt) ss.lmq[tid] = 0;
    constexpr int kEarly = 8;
    int pw[kEarly];
#pragma unroll
    for (int k = 0; k < kEarly; ++k) {  // (volatile: issued here, not sunk past the row work)
        const int t = k * BM + tid;
        pw[k] = 0;
        if (tid < BM && k < a.n_qt && t < a.nt)
            asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(pw[k]) : "l"(a.pos + t) : "memory");
    }
    step_rows<T>(a, x, fq, fk);

    // Grid barrier: every CTA's row work before any item reads it.  Arrivals are counted; a CTA
    // leaves once all have arrived and later counts its departure; the last to depart zeroes both
    // counts for the next launch (every CTA has left the wait by then).  The tiles' windows and
    // the item enumeration are computed between the arrival and the wait.  Every CTA reads the
    // same control block before any arrival, so on a refused workspace none arrives or waits.
    if (tid == 0) {
        sm.lmax = (ctl_tag == 0 || ws_key_valid(ctl_tag)) && ctl_dep == 0 ? 0 : 1;  // 1: refused
        if (sm.lmax && blockIdx.x == 0) flag_error(a.err, MINF_ERRBIT_WORKSPACE);
    }
    __syncthreads();
    const bool ws_refused = sm.lmax != 0;
    // release: the CTA's writes (ordered before by the barrier above) before the arrival; it
    // waits for those writes to complete, so a thread outside the window loop below makes it
    if (tid == kProducerWarp * 32 && !ws_refused)
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(x.bar) : "memory");
    if (tid < BM) {
        for (int qt = 0; qt < a.n_qt; ++qt) {
            const int t = qt * BM + tid;
            int p = 0;
#pragma unroll
            for (int k = 0; k < kEarly; ++k)
                if (k == qt) p = pw[k];
            if (qt >= kEarly && t < a.nt) p = __ldg(a.pos + t);
            int L = 0;
            if (t < a.nt) {
                L = p < 0 ? 0 : (p + 1 < a.cap ? p + 1 : a.cap);
                if ((p < 0 || p >= a.cap) && blockIdx.x == 0) flag_error(a.err, MINF_ERRBIT_ATTN_POS);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) L = max(L, __shfl_xor_sync(0xffffffffu, L, o));
            if (lane == 0) atomicMax(&ss.lmq[qt], L);
        }
    }
    __syncthreads();
    if (tid == 0) {
        // the items: chunks with keys of every tile (chunk 0 always: it writes the output)
        int acc = 0;
        for (int q = 0; q < a.n_qt; ++q) {
            ss.pref[q] = acc;
            const int nta = (ss.lmq[q] + BN - 1) / BN;
            const int na = (nta + a.kc_tiles - 1) / a.kc_tiles;
            acc += na > 1 ? na : 1;
        }
        ss.pref[a.n_qt] = acc;
        // acquire: every other CTA's writes before this CTA's reads after the wait
        const unsigned long long t0n = gtimer();
        while (!ws_refused) {
            int n;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(n) : "l"(x.bar) : "memory");
            if (n >= static_cast<int>(gridDim.x)) break;
            if (gtimer() - t0n > kWaitBudgetNs) {
                sm.abort_flag = 1;
                flag_error(a.err, MINF_ERRBIT_TIMEOUT);
                x.bar[kWsTag] = kWsPoison;  // its counts are left non-zero: refused until zero-filled
                break;
            }
        }
    }
    __syncthreads();
    // the rows stored by other CTAs are read next by bulk tensor copies (the async proxy), which
    // the producer thread issues
    if (warp == kProducerWarp && lane == 0) fence_async_global();
    // The launch after this one may start: the rows it may stream before its own wait are stored.
    gdc_launch_dependents();

    const int g = a.nh / a.nk;
    const int n_items = (*abort_flag || ws_refused) ? 0 : ss.pref[a.n_qt] * a.nh;
    // the departure: by the first item's P*V thread while it waits for P(0), else here
    if (static_cast<int>(blockIdx.x) >= n_items && tid == 0 && !ws_refused) step_depart(x, a.ws_key);
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int h = item % a.nh, pr = item / a.nh;
        int qt = 0;
        while (qt + 1 < a.n_qt && ss.pref[qt + 1] <= pr) ++qt;
        const int kc = pr - ss.pref[qt];
        const int lmax = ss.lmq[qt];
        const int t0 = qt * BM;
        if (tid == 0) {
            if (item != static_cast<int>(blockIdx.x)) init_barriers(true);
            sm.lmax = 0;  // the merge's "last chunk" flag
        }
        const int n_tiles_all = (lmax + BN - 1) / BN;
        const int n_act = (n_tiles_all + a.kc_tiles - 1) / a.kc_tiles;
        const int tile0 = kc * a.kc_tiles;
        const int n_tiles = min(n_tiles_all - tile0, a.kc_tiles) > 0 ? min(n_tiles_all - tile0, a.kc_tiles) : 0;
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const Item it = {h, h / g, qt, kc, t0, -1, lmax, n_act, tile0, n_tiles, tmem,
                         item == static_cast<int>(blockIdx.x) ? &x : nullptr, a.ws_key};
        attend<HDKV, T>(sm, tm_q, tm_k, a, it);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (*abort_flag) break;
    }
    __syncthreads();
    if (warp == kProducerWarp) {
        if (*abort_flag && lane == 0) {
            // let copies and MMAs that may still be in flight finish before TMEM and shared memory go away
            const unsigned long long t0n = gtimer();
            while (gtimer() - t0n < kWaitBudgetNs / 4) {
            }
            x.bar[kWsTag] = kWsPoison;  // a wait expired: refused until zero-filled
        }
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols<HDKV>())
                     : "memory");
    }
}

static_assert(sizeof(Smem<128>) + sizeof(StepSmem) + 1024 <= 232448, "the fused step fits 227 KB of shared memory");

struct PrefillPlan {
    int n_qt, n_kc, kc_tiles;
    size_t step_off, o_off, ml_off, ticket_off, total;  // step: the fused step's barrier counts
};

size_t align256p(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Key chunks: at least 128 keys each and at most 16 per query tile (so the launch never
// depends on the positions and stays small for long regions).
PrefillPlan prefill_plan(int nt, int nh, int hd_kv, int cap) {
    PrefillPlan p;
    p.n_qt = (nt + BM - 1) / BM;
    long long kc_keys = (static_cast<long long>(cap) + 15) / 16;
    kc_keys = ((kc_keys + BN - 1) / BN) * BN;
    if (kc_keys < 128) kc_keys = 128;
    p.kc_tiles = static_cast<int>(kc_keys / BN);
    p.n_kc = static_cast<int>((cap + kc_keys - 1) / kc_keys);
    const size_t parts = static_cast<size_t>(p.n_qt) * nh * p.n_kc;
    p.step_off = 0;          // the control block: the step's barrier counts and the layout tag
    p.o_off = kWsCtlBytes;
    p.ml_off = p.o_off + (p.n_kc > 1 ? align256p(parts * hd_kv * BM * sizeof(float)) : 0);
    p.ticket_off = p.ml_off + (p.n_kc > 1 ? align256p(parts * 2 * BM * sizeof(float)) : 0);
    p.total = p.ticket_off + (p.n_kc > 1 ? align256p(static_cast<size_t>(p.n_qt) * nh * sizeof(int)) : 0);
    return p;
}

// Tensor maps and kernel parameters of a prefill launch, shared by both kernels.
template <int HDKV, typename T>
int prefill_setup(const PrefillArgs &pa, CUtensorMap *tq, CUtensorMap *tk, PParams *out, PrefillPlan *plan) {
    if (!make_tensor_map_2d(tq, pa.q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, static_cast<uint64_t>(pa.nh) * pa.hd, pa.nt,
                            32, BM, true))
        return MINF_ERR_CUDA;
    if (!std::is_same<T, float>::value)
        *tk = *tq;  // binary16 and Q8_0 K are read by the staging warps: the map argument goes unused
    else if (!make_tensor_map_2d(tk, pa.k_reg, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                                 static_cast<uint64_t>(pa.nk) * HDKV, pa.cap, 32, BN, true))
        return MINF_ERR_CUDA;
    PParams a;
    a.out = pa.out;
    a.k_reg = pa.k_reg;
    a.v_reg = pa.v_reg;
    a.row_bytes = q8_row_bytes(pa.nk * HDKV);
    a.pos = pa.pos;
    a.err = pa.err;
    a.nt = pa.nt;
    a.nh = pa.nh;
    a.nk = pa.nk;
    a.hd = pa.hd;
    a.cap = pa.cap;
    a.W = pa.nk * HDKV;
    a.scale_log2 = pa.scale * kLog2e;
    const PrefillPlan pl = prefill_plan(pa.nt, pa.nh, HDKV, pa.cap);
    a.n_qt = pl.n_qt;
    a.n_kc = pl.n_kc;
    a.kc_tiles = pl.kc_tiles;
    if (pl.n_kc > 1 && (!pa.ws || pa.ws_bytes < pl.total || !aligned16(pa.ws))) return MINF_ERR_WORKSPACE;
    char *ws = static_cast<char *>(pa.ws);
    a.ws_o = pl.n_kc > 1 ? reinterpret_cast<float *>(ws + pl.o_off) : nullptr;
    a.ws_ml = pl.n_kc > 1 ? reinterpret_cast<float *>(ws + pl.ml_off) : nullptr;
    a.ws_ticket = pl.n_kc > 1 ? reinterpret_cast<int *>(ws + pl.ticket_off) : nullptr;
    a.ws_tag = pl.n_kc > 1 ? reinterpret_cast<int *>(ws) + kWsTag : nullptr;
    a.ws_key = ws_key(kWsKindPrefill, pl.o_off, pl.ml_off, pl.ticket_off, pl.total);
    *out = a;
    *plan = pl;
    return MINF_OK;
}

template <int HDKV, typename T>
int launch_t(const PrefillArgs &pa, cudaStream_t s) {
    CUtensorMap tq, tk;
    PParams a;
    PrefillPlan pl;
    const int st = prefill_setup<HDKV, T>(pa, &tq, &tk, &a, &pl);
    if (st != MINF_OK) return st;
    const size_t smem = sizeof(Smem<HDKV>) + 1024;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MINF_ERR_CUDA;
    static std::atomic<bool> attr_set[64];
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(prefill_kernel<HDKV, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return MINF_ERR_CUDA;
        attr_set[dev].store(true, std::memory_order_release);
    }
    const long long ctas = static_cast<long long>(pl.n_qt) * pa.nh * pl.n_kc;
    if (ctas > 0x7fffffffLL) return MINF_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kThreadsP);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pa.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prefill_kernel<HDKV, T>, tq, tk, a) == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

// The fused step: MINF_ERR_UNSUPPORTED (nothing launched) where its conditions do not hold.
template <int HDKV, typename T>
int launch_step_t(const PrefillArgs &pa, const PrefillStepExtra &xs, cudaStream_t s) {
    const PrefillPlan plan = prefill_plan(pa.nt, pa.nh, HDKV, pa.cap);
    if (plan.n_qt > kStepMaxQt || pa.hd % 8 != 0 || pa.hd > 2 * kMaxHalf || !pa.ws || pa.ws_bytes < plan.total ||
        !aligned16(pa.ws) || !aligned16(xs.q) || !aligned16(xs.k) || !aligned16(xs.v) || !aligned16(pa.k_reg) ||
        !aligned16(pa.v_reg))
        return MINF_ERR_UNSUPPORTED;
    const long long units =
        static_cast<long long>(pa.nt) * ((pa.hd / 8) * ((pa.nh + kRopeHeads - 1) / kRopeHeads) +
                                         (HDKV / 8) * ((pa.nk + kRopeHeads - 1) / kRopeHeads) + pa.nk * HDKV / 4);
    if (units >= (1ll << 30)) return MINF_ERR_UNSUPPORTED;
    CUtensorMap tq, tk;
    PParams a;
    PrefillPlan pl;
    int st = prefill_setup<HDKV, T>(pa, &tq, &tk, &a, &pl);
    if (st != MINF_OK) return st;
    StepParams x;
    x.q = xs.q;
    x.k = xs.k;
    x.v = xs.v;
    x.k_st = const_cast<void *>(pa.k_reg);
    x.v_st = const_cast<void *>(pa.v_reg);
    x.style = xs.style;
    x.xn = xs.xn;
    x.hx = xs.h;
    x.gain = xs.gain;
    x.n_embd = xs.n_embd;
    x.norm_vec = (xs.n_embd % 4 == 0) && aligned16(xs.h) && aligned16(xs.xn) && (!xs.gain || aligned16(xs.gain));
    x.eps = xs.eps;
    char *ws = static_cast<char *>(pa.ws);
    x.bar = reinterpret_cast<int *>(ws + pl.step_off);
    RopeTable rq, rk;
    rope_table(&rq, pa.hd, xs.theta, xs.freq_scale);
    rope_table(&rk, HDKV, xs.theta, xs.freq_scale);
    const size_t smem = sizeof(Smem<HDKV>) + sizeof(StepSmem) + 1024;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MINF_ERR_CUDA;
    // per device, shared by host threads: CTAs that can be resident at once (0: not yet known),
    // and whether the runtime refused the cooperative launch with early start
    static std::atomic<int> resident[64];
    static std::atomic<bool> no_pdl[64];
    int res = resident[dev].load(std::memory_order_acquire);
    if (!res) {
        if (cudaFuncSetAttribute(prefill_step_kernel<HDKV, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return MINF_ERR_CUDA;
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prefill_step_kernel<HDKV, T>, kThreadsP, smem) !=
                cudaSuccess ||
            per_sm < 1)
            return MINF_ERR_UNSUPPORTED;
        res = per_sm * sm_count();
        resident[dev].store(res, std::memory_order_release);
    }
    const long long items = static_cast<long long>(pl.n_qt) * pa.nh * pl.n_kc;
    const int grid = static_cast<int>(items < res ? items : res);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreadsP);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every CTA resident
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    const bool pdl = !no_pdl[dev].load(std::memory_order_relaxed);
    cfg.numAttrs = pdl ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_step_kernel<HDKV, T>, tq, tk, a, x, rq, rk);
    if (e != cudaSuccess && pdl) {
        // Retried without early start; only when that launch succeeds was the refusal the
        // attribute's, and later calls on this device skip it.  Any other failure is returned.
        (void)cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, prefill_step_kernel<HDKV, T>, tq, tk, a, x, rq, rk);
        if (e == cudaSuccess) no_pdl[dev].store(true, std::memory_order_relaxed);
    }
    return e == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

}  // namespace

size_t prefill_workspace_bytes(int nt, int nh, int hd_kv, int cap) {
    if (nt <= 0 || nh <= 0 || hd_kv <= 0 || cap <= 0) return 0;
    return prefill_plan(nt, nh, hd_kv, cap).total;
}

int launch_prefill_step(const PrefillArgs &pa, const PrefillStepExtra &x, cudaStream_t s) {
    if (pa.nt == 0) return MINF_OK;
    if ((static_cast<long long>(pa.nh) * pa.hd) % 4 != 0) return MINF_ERR_UNSUPPORTED;
    if (pa.kv == kKvF16) {
        if (pa.hd_kv == 64) return launch_step_t<64, __half>(pa, x, s);
        if (pa.hd_kv == 128) return launch_step_t<128, __half>(pa, x, s);
    } else if (pa.kv == kKvF32) {
        if (pa.hd_kv == 64) return launch_step_t<64, float>(pa, x, s);
        if (pa.hd_kv == 128) return launch_step_t<128, float>(pa, x, s);
    }
    return MINF_ERR_UNSUPPORTED;
}

int launch_prefill(const PrefillArgs &pa, cudaStream_t s) {
    if (pa.nt == 0) return MINF_OK;
    if ((static_cast<long long>(pa.nh) * pa.hd) % 4 != 0) return MINF_ERR_UNSUPPORTED;
    if (pa.kv == kKvF16) {
        if (pa.hd_kv == 64) return launch_t<64, __half>(pa, s);
        if (pa.hd_kv == 128) return launch_t<128, __half>(pa, s);
        return MINF_ERR_UNSUPPORTED;
    }
    if (pa.kv == kKvQ8) {
        if (pa.hd_kv == 64) return launch_t<64, Q8>(pa, s);
        if (pa.hd_kv == 128) return launch_t<128, Q8>(pa, s);
        return MINF_ERR_UNSUPPORTED;
    }
    if (pa.hd_kv == 64) return launch_t<64, float>(pa, s);
    if (pa.hd_kv == 128) return launch_t<128, float>(pa, s);
    return MINF_ERR_UNSUPPORTED;
}

}  // namespace minf
