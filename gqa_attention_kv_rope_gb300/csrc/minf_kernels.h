// minf_kernels.h -- internal launcher declarations (between the C ABI and the kernels).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace minf {

// Storage of the K/V regions: fp32, IEEE binary16 (converted on the store with round to
// nearest even, read back exactly), or Q8_0 blocks; the arithmetic stays fp32.
enum KvKind : int { kKvF32 = 0, kKvF16 = 1, kKvQ8 = 2 };

// Q8_0 storage ("11 . Attention, vec ops, and the KV cache", §2.5): a row of W values is W int8
// quants, then W/32 binary16 block scales, then zero padding to a multiple of 16 bytes; the
// store quantizes each 32-value block with d = max|x|/127, q = round(x * (1/d)) (halves away
// from zero), and a value reads back as f16(d) * q.
inline long long q8_row_bytes(int W) { return W + ((static_cast<long long>(W / 32) * 2 + 15) / 16) * 16; }

struct RopeKvArgs {
    float *q;               // [nt, nh, hd], rotated in place
    float *k;               // [nt, nk, hd_kv], rotated in place
    const float *v;         // [nt, nk*hd_kv]
    const int32_t *pos;     // [nt]
    void *k_reg, *v_reg;    // regions / arena [rows, nk*hd_kv] of `kv` elements
    int kv;                 // KvKind
    const int64_t *row_off; // per token arena row offset (nullable: 0)
    const int32_t *caps;    // per token capacity (nullable: cap)
    int cap;
    int nt, nh, nk, hd, hd_kv, style;
    int32_t *err;
    // paged regions (table non-null): token t is sequence t's token; its row p is pool row
    // table[t*max_blocks + p/block_rows]*block_rows + p%block_rows; cap = max_blocks*block_rows
    const int32_t *table;
    int max_blocks, block_rows, pool_blocks;
};

struct DecodeArgs {
    float *out;              // [n_seq, nh*hd_kv]
    const float *q;          // [n_seq, nh, hd]
    const void *k_reg, *v_reg;  // of `kv` elements
    int kv;                  // KvKind
    const int64_t *row_off;  // per sequence (nullable)
    const int32_t *caps;     // per sequence (nullable)
    int cap;                 // capacity when caps is null; also the host bound max_cap
    long long arena_rows;    // rows of the K/V arena when row_off is given
    const int32_t *pos;      // [n_seq]
    int n_seq, nh, nk, hd, hd_kv;
    float scale;
    int32_t *err;
    void *ws;
    size_t ws_bytes;
    // paged regions (table non-null): the pool has arena_rows rows in blocks of block_rows;
    // sequence s's row j is pool row table[s*max_blocks + j/block_rows]*block_rows + j%block_rows,
    // and cap = max_blocks*block_rows
    const int32_t *table;
    int max_blocks, block_rows;
};

int launch_rms_norm(float *y, const float *x, const float *w, int rows, int n, float eps,
                    cudaStream_t s);
int launch_rope(float *x, const int32_t *pos, int nt, int nh, int hd, float theta,
                float freq_scale, int style, int32_t *err, cudaStream_t s);
int launch_kv_append(void *k_reg, void *v_reg, int kv, int cap, int W, const float *k_rows,
                     const float *v_rows, const int32_t *pos, int nt, int32_t *err,
                     cudaStream_t s);
// Q8_0 store (one row per token at pos, at row_off[t] + pos with caps[t] when given; with a
// table, token t is sequence t's token and its row goes through the table).
int launch_kv_append_q8(void *k_reg, void *v_reg, int cap, int W, const float *k_rows, const float *v_rows,
                        const int32_t *pos, int nt, const int64_t *row_off, const int32_t *caps,
                        const int32_t *table, int max_blocks, int block_rows, int pool_blocks, int32_t *err,
                        cudaStream_t s);
// One row per sequence through a block table (the pool has pool_blocks blocks).
int launch_kv_append_paged(void *k_pool, void *v_pool, int kv, int pool_blocks, int block_rows, int W,
                           const int32_t *table, int max_blocks, const float *k_rows, const float *v_rows,
                           const int32_t *pos, int n_seq, int32_t *err, cudaStream_t s);
int launch_rope_kv_append(const RopeKvArgs &a, float theta, float freq_scale, cudaStream_t s);

struct NormArgs {
    float *y;
    const float *x, *w;
    int rows, n;
    float eps;
};
// RMSNorm rows and RoPE + KV store in one launch (the layer step's prologue when the
// attention is a separate launch); it releases the next launch at once.
int launch_layer_prologue(const RopeKvArgs &a, float theta, float freq_scale, const NormArgs &nrm, cudaStream_t s);
int launch_silu_mul(float *y, const float *g, const float *u, long long n, cudaStream_t s);

// The fused QKV decode op (RMSNorm, q/k/v projections with biases, RoPE, K/V store) for up to
// kQkvMaxTok tokens of one sequence.
constexpr int kQkvMaxTok = 16;
struct QkvArgs {
    float *xn;                 // [nt, n_embd] RMSNorm output
    const float *h, *gain;     // [nt, n_embd], [n_embd] (gain nullable)
    float eps;
    int n_embd;
    const float *w, *b;        // [n_out, n_embd] (q rows, k rows, v rows), [n_out] (nullable)
    const int32_t *pos;        // [nt]
    int nt;
    float *q, *k, *v;          // [nt, nh*hd] rotated, [nt, W] rotated, [nt, W]
    float *k_reg, *v_reg;      // regions [cap, W]
    int cap, nh, nk, hd, hd_kv, style;
    int32_t *err;
};
int launch_fused_qkv(const QkvArgs &a, float theta, float freq_scale, cudaStream_t s);

// The rest of a decode layer step, fused into the attention launch (one token per sequence).
struct DecodeStepExtra {
    float *k;             // [n_seq, nk, hd_kv] rotated in place
    const float *v;       // [n_seq, W]
    float *xn;            // [n_seq, n_embd] RMSNorm output
    const float *h, *gain;
    float eps, theta, freq_scale;
    int n_embd, style;
    bool pdl;             // launch with programmatic stream serialization
    bool early;           // with pdl: read the positions and stream cached rows before the
                          // dependency wait (the launch before writes neither)
};

struct PrefillArgs {
    float *out;               // [nt, nh*hd_kv]
    const float *q;           // [nt, nh, hd] (rotated)
    const void *k_reg, *v_reg;  // regions [cap, nk*hd_kv] of `kv` elements
    int kv;                   // KvKind
    const int32_t *pos;       // [nt]
    int32_t *err;
    int nt, nh, nk, hd, hd_kv, cap;
    float scale;
    void *ws;                 // key-chunk partials (prefill_workspace_bytes)
    size_t ws_bytes;
    bool pdl;                 // launch with programmatic stream serialization
};

size_t prefill_workspace_bytes(int nt, int nh, int hd_kv, int cap);
int launch_prefill(const PrefillArgs &a, cudaStream_t s);

// The rest of a prefill layer step, fused into the attention launch (one sequence, contiguous
// fp32 or binary16 regions).  launch_prefill_step returns MINF_ERR_UNSUPPORTED, launching
// nothing, where the fused kernel does not apply (the caller then runs the prologue launch and
// launch_prefill).
struct PrefillStepExtra {
    float *q, *k;         // [nt, nh, hd], [nt, nk, hd_kv] rotated in place (q: the PrefillArgs q)
    const float *v;       // [nt, W]
    float *xn;            // [nt, n_embd] RMSNorm output
    const float *h, *gain;
    float eps, theta, freq_scale;
    int n_embd, style;
};
int launch_prefill_step(const PrefillArgs &a, const PrefillStepExtra &x, cudaStream_t s);

size_t decode_workspace_bytes(int n_seq, int nh, int nk, int hd_kv, int max_cap);
bool decode_supported(int nh, int nk, int hd, int hd_kv);
bool fused_step_supported(int nh, int nk, int hd, int hd_kv, int n_embd);
int launch_decode(const DecodeArgs &a, cudaStream_t s);
int launch_decode_step(const DecodeArgs &a, const DecodeStepExtra &x, cudaStream_t s);

}  // namespace minf
