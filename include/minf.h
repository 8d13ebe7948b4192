/*
 * minf.h -- C ABI of the GB300 attention-stage library (libminf.so).
 *
 * One layer's attention stage of a small decoder-only LLM: RMSNorm, rotary
 * position embedding at positions passed in as data, an in-place append of the
 * step's K/V rows into persistent per-layer regions addressed by position, and
 * grouped-query attention over the causal window [0, pos].
 *
 * Sources (page title, section):
 *   "11 . Attention, vec ops, and the KV cache" (minfer walkthrough)  [P1]
 *   "IV.2: Zero-copy KV cache"                                         [P2]
 *   "13 . The decode loop and graph reuse" (minfer walkthrough)        [P3]
 *
 * Conventions for every entry point:
 *   - The caller owns all memory.  The library never allocates or frees device
 *     memory and never synchronises; every call is enqueued on `stream`.
 *   - All float tensors are fp32, row-major, contiguous, 16-byte aligned, in
 *     device memory (unless stated otherwise).  int32 positions are device arrays,
 *     so a captured CUDA graph can be replayed with only the positions changed
 *     ([P3] §2.3: positions and n_past are data, not topology).
 *   - Host-detectable problems return a status without launching anything.
 *   - Problems only the device can see (a position outside a region) are never
 *     clamped into a write: the kernel skips the write and ORs a bit into the
 *     caller's device word `*err` ([P1] §3.2.3: an out-of-range KV position is a
 *     hard error).  Check it after synchronising.  Kernels never trap.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Shapes: nh = n_head, nk = n_kv_head, g = nh/nk, hd = query head dim,
 *     hd_kv = key/value head dim, W = nk*hd_kv (the K/V row width).
 */
#ifndef MINF_H
#define MINF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *minf_stream_t; /* identical to cudaStream_t */

#if defined(__GNUC__)
#define MINF_API __attribute__((visibility("default")))
#else
#define MINF_API
#endif

/* Status codes returned by every entry point. */
enum {
    MINF_OK = 0,
    MINF_ERR_ARG = 1,         /* null/misaligned pointer, size out of range, bad style */
    MINF_ERR_GEOMETRY = 2,    /* hd < hd_kv ([P1] §1: refused) or n_head % n_kv_head != 0 */
    MINF_ERR_UNSUPPORTED = 3, /* valid geometry the kernels do not implement */
    MINF_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required */
    MINF_ERR_CUDA = 6         /* a kernel launch failed */
};

/* Bits OR-ed into the device error word *err. */
#define MINF_ERRBIT_STORE_POS 0x1  /* KV store: pos < 0 or pos >= cap; that row was not written */
#define MINF_ERRBIT_ROPE_POS 0x2   /* RoPE: pos < 0; that token was left unrotated */
#define MINF_ERRBIT_ATTN_POS 0x4   /* attention: pos < 0 (empty window, zero output) or
                                      pos >= cap (window clamped to cap, as [P1] §3.2.4's
                                      nkv = min(max pos + 1, n_ctx) does) */
#define MINF_ERRBIT_TIMEOUT 0x8    /* an internal pipeline wait exceeded its time budget (200 ms);
                                      the call's outputs are invalid.  Kernels bound every wait
                                      so that a fault in the pipeline returns instead of hanging. */
#define MINF_ERRBIT_BLOCK 0x10     /* paged regions: a block the window or the store needs is
                                      missing from the table (id < 0 or past the pool); its rows
                                      read as zeros, the store is skipped, the outputs of that
                                      sequence are invalid */
#define MINF_ERRBIT_WORKSPACE 0x20 /* the workspace was last used by a call of another layout
                                      (a decode call of another shape, a prefill after a decode
                                      or the reverse: its merge tickets may not be zero), was
                                      never zero-filled, or held the workspace of a call whose
                                      bounded wait expired.  Nothing that depends on the
                                      workspace was computed (the attention output is not
                                      written); zero-fill it and call again.  The test reads a
                                      tag in the workspace's first 256 bytes (its control block:
                                      the counters every call leaves at zero, and the layout of
                                      the last call that used it). */

/* Human-readable name of a status code (static storage). */
MINF_API const char *minf_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
MINF_API int minf_version(void);

/*
 * RoPE angular speeds, host-side.  [P1] §2.3 and §3.2.2: freq_i =
 * freq_scale / theta^(2i/hd) for i < hd/2.  Evaluated as the exact quotient in
 * double and rounded once to float (so the table does not depend on a
 * particular powf).  `freqs` is a HOST array of hd/2 floats.
 * Errors: MINF_ERR_ARG if freqs is NULL, hd is odd, hd <= 0 or hd > 256.
 */
MINF_API int minf_rope_freqs(float *freqs, int hd, float theta, float freq_scale);

/*
 * RMSNorm with gains.  [P1] §3.2.1: y = x / sqrt(mean(x^2) + eps) * w, no mean
 * subtraction.  x, y: [rows, n]; w: [n] (NULL = unit gains).  y may equal x.
 * Errors: MINF_ERR_ARG for null x/y, rows < 0, n <= 0.  rows == 0 is a no-op.
 */
MINF_API int minf_rms_norm(float *y, const float *x, const float *w, int rows, int n, float eps,
                  minf_stream_t stream);

/*
 * Rotary position embedding, in place.  [P1] §3.2.2: for token t, head h and
 * i < hd/2, th = (float)pos[t] * freq_i; the pair (i, i+hd/2) (style 0,
 * NonInterleaved: Qwen, NEOX) or (2i, 2i+1) (style 1, Interleaved: Llama) is
 * rotated by +th.  x: [nt, n_head, hd]; pos: int32[nt] (device).
 * Device errors: pos[t] < 0 -> MINF_ERRBIT_ROPE_POS, token left unchanged.
 * Errors: MINF_ERR_ARG for null x/pos/err, nt < 0, n_head <= 0, odd hd,
 * hd > 256, style not in {0, 1}.
 */
MINF_API int minf_rope(float *x, const int32_t *pos, int nt, int n_head, int hd, float theta,
              float freq_scale, int style, int32_t *err, minf_stream_t stream);

/*
 * KV store: a pure copy, bit-exact.  [P1] §3.2.3 and [P2] (in-place append):
 * for each token t with p = pos[t] in [0, cap): K region row p = k_rows[t],
 * V region row p = v_rows[t].  Regions: [cap, row_width]; rows: [nt, row_width].
 * Device errors: p < 0 or p >= cap -> MINF_ERRBIT_STORE_POS and that token's
 * rows are not written (other tokens still are).
 * Errors: MINF_ERR_ARG for null pointers, cap <= 0, nt < 0, row_width <= 0 or
 * not a multiple of 4.
 */
MINF_API int minf_kv_append(float *k_reg, float *v_reg, int cap, int row_width, const float *k_rows,
                   const float *v_rows, const int32_t *pos, int nt, int32_t *err,
                   minf_stream_t stream);

/*
 * Fused RoPE on q and k plus the KV store ([P1] §3.2.2 and §3.2.3, store
 * before attention per [P1] §3.4).  q: [nt, n_head, hd] and k: [nt, n_kv_head,
 * hd_kv] are rotated in place; the rotated k rows and the v rows [nt, W] are
 * then written to row pos[t] of the regions [cap, W].  The appended K row is
 * bit-identical to minf_rope's output for the same k.
 * Device errors: as minf_rope and minf_kv_append.
 * Errors: MINF_ERR_ARG / MINF_ERR_GEOMETRY as above.
 */
MINF_API int minf_rope_kv_append(float *q, float *k, const float *v, const int32_t *pos, int nt,
                        int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                        float freq_scale, int style, float *k_reg, float *v_reg, int cap,
                        int32_t *err, minf_stream_t stream);

/*
 * Bytes of device workspace minf_gqa_attn_decode needs for n_seq sequences
 * whose regions hold at most max_cap rows.  Returns 0 for invalid arguments.
 * The workspace must be zero-filled before its first use.  Every call leaves its
 * counters and merge tickets at zero, so calls of the same shape (n_seq, heads,
 * hd_kv, max_cap) can reuse it, and be captured in a CUDA graph, without clearing.
 * Its first 256 bytes are a control block that also records the layout of the last
 * call that used it: a call of another layout (another shape, or a prefill) leaves
 * partials where this one's tickets are, so the call refuses such a workspace with
 * MINF_ERRBIT_WORKSPACE until it is zero-filled again.  Two calls that run
 * concurrently must not share it.
 */
MINF_API size_t minf_attn_decode_workspace_bytes(int n_seq, int n_head, int n_kv_head, int hd_kv,
                                        int max_cap);

/*
 * Decode attention (one query token per sequence), split-KV.  [P1] §3.2.4 with
 * [P1] §2.5 (split the KV axis across blocks, then reduce) and [P2] (the
 * attention reads the cache through a view, never a copy):
 *   for sequence s and query head h, hk = h / g, L = min(pos[s] + 1, cap_s),
 *   out[s, h] = sum_{j < L} softmax_j(scale * q[s,h][0:hd_kv] . K[j, hk]) V[j, hk]
 * where K[j] is row seq_row_off[s] + j of the arena.  Arena: k_reg/v_reg
 * [arena_rows, W]; q: [n_seq, n_head, hd]; out: [n_seq, n_head*hd_kv].
 * seq_row_off: int64[n_seq] device (NULL = all 0, and the arena is then
 * max_cap rows); seq_cap: int32[n_seq] device (NULL = max_cap for all);
 * max_cap: host upper bound of every cap_s (it sizes the split grid and the
 * workspace; the grid never depends on pos, so the call can be graph-captured
 * and replayed with new positions); arena_rows: rows of the arena when
 * seq_row_off is given (the kernels read rows only inside it; ignored
 * otherwise).  The cached rows stream through a TMA pipeline, so the K/V
 * regions must stay in device memory that the tensor map can address.
 * Device errors: MINF_ERRBIT_ATTN_POS (see above).
 * Errors: MINF_ERR_ARG, MINF_ERR_GEOMETRY, MINF_ERR_UNSUPPORTED (hd_kv not 64
 * or 128, g > 8, hd > 256), MINF_ERR_WORKSPACE.
 */
MINF_API int minf_gqa_attn_decode(float *out, const float *q, const float *k_reg, const float *v_reg,
                         const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap,
                         int64_t arena_rows, const int32_t *pos, int n_seq, int n_head,
                         int n_kv_head, int hd, int hd_kv, float scale, void *ws,
                         size_t ws_bytes, int32_t *err, minf_stream_t stream);

/*
 * Decode attention without a caller-provided workspace.  None of the source pages has a
 * counterpart: this entry point exists for callers that cannot allocate device memory --
 * code embedded where it is handed only its input and output buffers, or callers that must
 * not call the device allocator on their hot path (it can synchronise the device or
 * fragment a memory pool they do not own).  It computes exactly what minf_gqa_attn_decode
 * computes, with the same arguments minus ws/ws_bytes, and allocates nothing: the split
 * partials and merge tickets live in a fixed 8 MiB array of device memory that the library
 * owns (every GPU that loads the library holds it until the process exits).
 *   - A call that would need more than 8 MiB of workspace (see
 *     minf_attn_decode_workspace_bytes) returns MINF_ERR_WORKSPACE and launches nothing.
 *   - The first call in a CUDA context looks up that context's copy of the array (with the
 *     context current; one entry per context, so a caller that switches contexts on a device
 *     is served too); make that first call before any stream capture in the context.
 *   - Each call clears the part of the array it uses (an asynchronous memset on `stream`)
 *     before its kernel.
 *   - Every call shares the one array: calls whose work overlaps on the GPU (different
 *     streams, or concurrent host threads) race on it and must be serialised by the caller.
 * Device errors and other statuses: as minf_gqa_attn_decode.
 */
MINF_API int minf_gqa_attn_decode_static_ws(float *out, const float *q, const float *k_reg,
                                   const float *v_reg, const int64_t *seq_row_off,
                                   const int32_t *seq_cap, int max_cap, int64_t arena_rows,
                                   const int32_t *pos, int n_seq, int n_head, int n_kv_head,
                                   int hd, int hd_kv, float scale, int32_t *err,
                                   minf_stream_t stream);

/*
 * Causal prefill attention over one sequence's regions.  [P1] §3.2.4: token t
 * attends over rows [0, min(pos[t] + 1, cap)) of the K/V regions [cap, W]
 * (store before attention: the tokens' own rows must already be appended).
 * q: [nt, n_head, hd]; out: [nt, n_head*hd_kv].  Positions are arbitrary
 * (a prefill that continues an existing cache passes pos = n_past..).
 * The QK^T and PV products run on the tensor cores with split-precision operands
 * (hi + lo halves, three MMAs per product: binary16 halves of power-of-two-scaled
 * q and k rows for QK^T, TF32 halves for PV) and fp32 accumulation, which matches
 * an fp32 evaluation to a few 1e-6; max, exp and sums run in fp32.
 * The keys of a query tile are cut into chunks processed by separate CTAs whose
 * partials are folded at the end: ws must hold minf_attn_prefill_workspace_bytes
 * (zero-filled before its first use; every call leaves its counters and tickets at
 * zero, the partial outputs not, so a workspace last used by a call of another
 * shape, or by decode, is refused with MINF_ERRBIT_WORKSPACE until it is zero-filled
 * again; concurrent calls must not share it); it may be NULL when no query tile has
 * more than one key chunk.  The call reads pos only after the launch before it on
 * the stream has finished.
 * Device errors: MINF_ERRBIT_ATTN_POS, MINF_ERRBIT_TIMEOUT, MINF_ERRBIT_WORKSPACE.
 * Errors: as minf_gqa_attn_decode.
 */
MINF_API int minf_gqa_attn_prefill(float *out, const float *q, const float *k_reg, const float *v_reg,
                          int cap, const int32_t *pos, int nt, int n_head, int n_kv_head, int hd,
                          int hd_kv, float scale, void *ws, size_t ws_bytes, int32_t *err,
                          minf_stream_t stream);

/* Workspace bytes minf_gqa_attn_prefill (and a layer step with nt > 1) needs for
 * nt tokens over regions of cap rows (at least 256 for nt > 0; 0 for nt <= 0). */
MINF_API size_t minf_attn_prefill_workspace_bytes(int nt, int n_head, int n_kv_head, int hd_kv, int cap);

/*
 * One layer's attention stage for one sequence ([P1] §1, the decoder-layer
 * picture, minus the weight matmuls): xn = RMSNorm(h) * gain ([nt, n_embd]);
 * q [nt, n_head, hd] and k [nt, n_kv_head, hd_kv] rotated in place at pos;
 * rotated k and v appended at pos into the regions [cap, W]; out [nt, n_head*hd_kv]
 * = attention with scale 1/sqrt(hd) ([P1] §2.4).  nt == 1 runs the split-KV
 * decode path (a single launch for the supported geometries), nt > 1 the
 * tensor-core prefill path: a single cooperative launch (the row work over the
 * whole grid, a grid barrier, then the attention) when hd % 8 == 0, hd <= 256,
 * nt <= 8192, q, k, v and the regions are 16-byte aligned and ws is given, else
 * a launch for RMSNorm, RoPE and the store followed by the attention launch.
 * ws/ws_bytes: for nt == 1 at least
 * minf_attn_decode_workspace_bytes(1, n_head, n_kv_head, hd_kv, cap), for nt > 1
 * at least minf_attn_prefill_workspace_bytes(nt, n_head, n_kv_head, hd_kv, cap);
 * zero-filled before its first use.  Every call leaves the workspace's first
 * 256 bytes (its control block: counters and the tag of the last layout that used
 * it) ready for the next: consecutive nt > 1 steps of any shape may share one
 * workspace, a single-launch prefill step may follow a decode step on it, and a
 * decode step may follow decode steps of the same shape.  Any other reuse (a decode
 * step after a prefill, or after a decode of another shape) is refused on the
 * device with MINF_ERRBIT_WORKSPACE until the workspace is zero-filled again.
 * Ordering: safe after any launch.  Every launch of the step is a programmatic
 * dependent launch -- its blocks may be scheduled while the launch just before it on the
 * stream finishes -- but it reads nothing (pos included) before that launch has
 * finished, so a kernel that writes pos or the cached rows right before the call (an
 * eager pos.fill_, a copy kernel) is safe.  For early start use the _chained form below.
 * A launch after an nt > 1 step may start early once the step's rows are stored (its
 * grid barrier).
 * Device errors: any of the bits above.
 */
MINF_API int minf_layer_attn_step(float *xn, const float *h, const float *gain, float eps, int n_embd,
                         float *q, float *k, const float *v, const int32_t *pos, int nt,
                         float *k_reg, float *v_reg, int cap, int n_head, int n_kv_head, int hd,
                         int hd_kv, float theta, float freq_scale, int style, float *out,
                         void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream);

/*
 * minf_layer_attn_step with early start: the same arguments, results and errors, but the
 * nt == 1 (decode) launch reads pos and begins streaming the cached rows [0, pos) of the
 * regions before the launch just before it on the stream has finished (h, gain, q, k, v,
 * ws and every output only after it).  Use it when that launch writes neither pos nor
 * those rows -- the previous layer's step, a projection kernel -- so the row stream
 * overlaps its end; a host-to-device copy of pos is not a launch and is always safe.  If a
 * kernel writes pos or the rows just before, the call may read the old values: use
 * minf_layer_attn_step.  nt > 1 runs exactly as minf_layer_attn_step.  The _f16 and _q8
 * forms take the regions of minf_layer_attn_step_f16 and minf_layer_attn_step_q8.
 */
MINF_API int minf_layer_attn_step_chained(float *xn, const float *h, const float *gain, float eps, int n_embd,
                                          float *q, float *k, const float *v, const int32_t *pos, int nt,
                                          float *k_reg, float *v_reg, int cap, int n_head, int n_kv_head, int hd,
                                          int hd_kv, float theta, float freq_scale, int style, float *out,
                                          void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream);
MINF_API int minf_layer_attn_step_chained_f16(float *xn, const float *h, const float *gain, float eps, int n_embd,
                                              float *q, float *k, const float *v, const int32_t *pos, int nt,
                                              uint16_t *k_reg, uint16_t *v_reg, int cap, int n_head, int n_kv_head,
                                              int hd, int hd_kv, float theta, float freq_scale, int style,
                                              float *out, void *ws, size_t ws_bytes, int32_t *err,
                                              minf_stream_t stream);
MINF_API int minf_layer_attn_step_chained_q8(float *xn, const float *h, const float *gain, float eps, int n_embd,
                                             float *q, float *k, const float *v, const int32_t *pos, int nt,
                                             uint8_t *k_reg, uint8_t *v_reg, int cap, int n_head, int n_kv_head,
                                             int hd, int hd_kv, float theta, float freq_scale, int style,
                                             float *out, void *ws, size_t ws_bytes, int32_t *err,
                                             minf_stream_t stream);

/*
 * One layer's attention stage for a batch of n_seq independent sequences, one
 * token each ([P2] batched decode; [P1] §2.2).  h: [n_seq, n_embd];
 * q: [n_seq, n_head, hd]; k, v: [n_seq, W]; pos: int32[n_seq]; sequence s owns
 * arena rows [seq_row_off[s], seq_row_off[s] + seq_cap[s]) and appends at
 * row seq_row_off[s] + pos[s].  Both descriptor arrays are device memory and
 * required; arena_rows is the arena's row count.
 * ws: minf_attn_decode_workspace_bytes(n_seq, ..., max_cap).
 */
MINF_API int minf_layer_attn_step_batched(float *xn, const float *h, const float *gain, float eps,
                                 int n_embd, float *q, float *k, const float *v,
                                 const int32_t *pos, int n_seq, float *k_arena, float *v_arena,
                                 const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap,
                                 int64_t arena_rows, int n_head, int n_kv_head, int hd, int hd_kv,
                                 float theta,
                                 float freq_scale, int style, float *out, void *ws,
                                 size_t ws_bytes, int32_t *err, minf_stream_t stream);

/*
 * The f16 cache ([P1] §2.5: the GPU backends may keep the K/V regions in f16,
 * halving the bytes every attention read moves).  These entry points are the
 * ones above with the regions (or arena) holding IEEE binary16 values instead of
 * fp32, passed as uint16_t bit patterns, 16-byte aligned, row width W a multiple
 * of 8.  The store converts each element with round to nearest, ties to even
 * (the pages name no rounding; this is the format's default); the attention read
 * converts back exactly and computes in fp32 as before, so the result is the
 * fp32 attention over the values the regions hold.  q, k, v, out, h, xn stay
 * fp32, and the rotated k written back to `k` is the unrounded fp32 value.
 * Workspace sizes are the same functions as for fp32 regions.  Device errors and
 * statuses: as the fp32 entry points (MINF_ERR_ARG also for W not a multiple of 8).
 */
MINF_API int minf_kv_append_f16(uint16_t *k_reg, uint16_t *v_reg, int cap, int row_width, const float *k_rows,
                                const float *v_rows, const int32_t *pos, int nt, int32_t *err,
                                minf_stream_t stream);
MINF_API int minf_rope_kv_append_f16(float *q, float *k, const float *v, const int32_t *pos, int nt, int n_head,
                                     int n_kv_head, int hd, int hd_kv, float theta, float freq_scale, int style,
                                     uint16_t *k_reg, uint16_t *v_reg, int cap, int32_t *err,
                                     minf_stream_t stream);
MINF_API int minf_gqa_attn_decode_f16(float *out, const float *q, const uint16_t *k_reg, const uint16_t *v_reg,
                                      const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap,
                                      int64_t arena_rows, const int32_t *pos, int n_seq, int n_head,
                                      int n_kv_head, int hd, int hd_kv, float scale, void *ws, size_t ws_bytes,
                                      int32_t *err, minf_stream_t stream);
MINF_API int minf_gqa_attn_prefill_f16(float *out, const float *q, const uint16_t *k_reg, const uint16_t *v_reg,
                                       int cap, const int32_t *pos, int nt, int n_head, int n_kv_head, int hd,
                                       int hd_kv, float scale, void *ws, size_t ws_bytes, int32_t *err,
                                       minf_stream_t stream);
MINF_API int minf_layer_attn_step_f16(float *xn, const float *h, const float *gain, float eps, int n_embd,
                                      float *q, float *k, const float *v, const int32_t *pos, int nt,
                                      uint16_t *k_reg, uint16_t *v_reg, int cap, int n_head, int n_kv_head, int hd,
                                      int hd_kv, float theta, float freq_scale, int style, float *out, void *ws,
                                      size_t ws_bytes, int32_t *err, minf_stream_t stream);
MINF_API int minf_layer_attn_step_batched_f16(float *xn, const float *h, const float *gain, float eps,
                                              int n_embd, float *q, float *k, const float *v, const int32_t *pos,
                                              int n_seq, uint16_t *k_arena, uint16_t *v_arena,
                                              const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap,
                                              int64_t arena_rows, int n_head, int n_kv_head, int hd, int hd_kv,
                                              float theta, float freq_scale, int style, float *out, void *ws,
                                              size_t ws_bytes, int32_t *err, minf_stream_t stream);

/*
 * The Q8_0 cache ([P1] §2.5: the store quantizes each row into Q8_0 blocks --
 * 32 consecutive values kept as one binary16 scale and 32 int8 quants -- and
 * the attention read dequantizes the window it uses).  These entry points are
 * the fp32 ones with the regions (or arena, or pool) holding Q8_0 rows as bytes:
 * a row of W values is W int8 quants, then W/32 binary16 scales, then zero
 * padding to a multiple of 16 bytes -- minf_q8_row_bytes(W) bytes (1088 for
 * W = 1024, the pages' 3.76x).  The store quantizes each block with
 * d = max|x|/127 and q = round(x * (1/d)), halves away from zero (the pages
 * name the format, not the rounding); a value reads back as f16(d) * q, exactly
 * in fp32, and the attention is the fp32 attention over those values.  q, k, v,
 * out, h, xn stay fp32; the rotated k written back to `k` is not quantized.
 * W must be a multiple of 32.  Workspace sizes: the same functions as for fp32.
 * Device errors and statuses: as the fp32 entry points.
 */
MINF_API size_t minf_q8_row_bytes(int row_width); /* 0 when row_width is not a positive multiple of 32 */
MINF_API int minf_kv_append_q8(uint8_t *k_reg, uint8_t *v_reg, int cap, int row_width, const float *k_rows,
                               const float *v_rows, const int32_t *pos, int nt, int32_t *err, minf_stream_t stream);
MINF_API int minf_rope_kv_append_q8(float *q, float *k, const float *v, const int32_t *pos, int nt, int n_head,
                                    int n_kv_head, int hd, int hd_kv, float theta, float freq_scale, int style,
                                    uint8_t *k_reg, uint8_t *v_reg, int cap, int32_t *err, minf_stream_t stream);
MINF_API int minf_gqa_attn_decode_q8(float *out, const float *q, const uint8_t *k_reg, const uint8_t *v_reg,
                                     const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap,
                                     int64_t arena_rows, const int32_t *pos, int n_seq, int n_head, int n_kv_head,
                                     int hd, int hd_kv, float scale, void *ws, size_t ws_bytes, int32_t *err,
                                     minf_stream_t stream);
MINF_API int minf_gqa_attn_prefill_q8(float *out, const float *q, const uint8_t *k_reg, const uint8_t *v_reg,
                                      int cap, const int32_t *pos, int nt, int n_head, int n_kv_head, int hd,
                                      int hd_kv, float scale, void *ws, size_t ws_bytes, int32_t *err,
                                      minf_stream_t stream);
MINF_API int minf_layer_attn_step_q8(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q,
                                     float *k, const float *v, const int32_t *pos, int nt, uint8_t *k_reg,
                                     uint8_t *v_reg, int cap, int n_head, int n_kv_head, int hd, int hd_kv,
                                     float theta, float freq_scale, int style, float *out, void *ws,
                                     size_t ws_bytes, int32_t *err, minf_stream_t stream);
MINF_API int minf_layer_attn_step_batched_q8(float *xn, const float *h, const float *gain, float eps, int n_embd,
                                             float *q, float *k, const float *v, const int32_t *pos, int n_seq,
                                             uint8_t *k_arena, uint8_t *v_arena, const int64_t *seq_row_off,
                                             const int32_t *seq_cap, int max_cap, int64_t arena_rows, int n_head,
                                             int n_kv_head, int hd, int hd_kv, float theta, float freq_scale,
                                             int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                                             minf_stream_t stream);

/*
 * Paged regions ([P2]: the paged cache keeps a sequence as scattered fixed-size
 * blocks, so it has no contiguous view to lend; [P3] §2.2: the window the
 * attention reads is an explicit input).  A pool k_pool / v_pool of pool_rows
 * rows of width W (fp32, or binary16 for the _f16 forms) is cut into blocks of
 * block_rows rows; block_table is an int32 device array [n_seq, max_blocks] of
 * block ids: logical row j of sequence s is pool row
 *   block_table[s * max_blocks + j / block_rows] * block_rows + j % block_rows,
 * and the sequence's capacity is cap = max_blocks * block_rows.  One token per
 * sequence, at pos[s]: the window is rows [0, min(pos[s] + 1, cap)) as for
 * contiguous regions, and the store writes logical row pos[s].  Block ids may
 * differ per call (a graph replays with a new table as with new positions).
 * block_rows: a power of two in [16, 4096]; pool_rows a multiple of it.
 * Workspace: minf_attn_decode_workspace_bytes(n_seq, ..., cap).
 * Device errors: as the contiguous forms, plus MINF_ERRBIT_BLOCK when a block
 * the window or the store needs has an id < 0 or past the pool (its rows read
 * as zeros and the store is skipped; that sequence's outputs are invalid).
 * Errors: MINF_ERR_UNSUPPORTED for block_rows outside the above; otherwise as the
 * contiguous forms.
 */
MINF_API int minf_kv_append_paged(float *k_pool, float *v_pool, int64_t pool_rows, int row_width,
                                  const int32_t *block_table, int max_blocks, int block_rows, const float *k_rows,
                                  const float *v_rows, const int32_t *pos, int n_seq, int32_t *err,
                                  minf_stream_t stream);
MINF_API int minf_kv_append_paged_f16(uint16_t *k_pool, uint16_t *v_pool, int64_t pool_rows, int row_width,
                                      const int32_t *block_table, int max_blocks, int block_rows,
                                      const float *k_rows, const float *v_rows, const int32_t *pos, int n_seq,
                                      int32_t *err, minf_stream_t stream);
MINF_API int minf_gqa_attn_decode_paged(float *out, const float *q, const float *k_pool, const float *v_pool,
                                        int64_t pool_rows, const int32_t *block_table, int max_blocks,
                                        int block_rows, const int32_t *pos, int n_seq, int n_head, int n_kv_head,
                                        int hd, int hd_kv, float scale, void *ws, size_t ws_bytes, int32_t *err,
                                        minf_stream_t stream);
MINF_API int minf_gqa_attn_decode_paged_f16(float *out, const float *q, const uint16_t *k_pool,
                                            const uint16_t *v_pool, int64_t pool_rows, const int32_t *block_table,
                                            int max_blocks, int block_rows, const int32_t *pos, int n_seq,
                                            int n_head, int n_kv_head, int hd, int hd_kv, float scale, void *ws,
                                            size_t ws_bytes, int32_t *err, minf_stream_t stream);
MINF_API int minf_layer_attn_step_paged(float *xn, const float *h, const float *gain, float eps, int n_embd,
                                        float *q, float *k, const float *v, const int32_t *pos, int n_seq,
                                        float *k_pool, float *v_pool, int64_t pool_rows, const int32_t *block_table,
                                        int max_blocks, int block_rows, int n_head, int n_kv_head, int hd,
                                        int hd_kv, float theta, float freq_scale, int style, float *out, void *ws,
                                        size_t ws_bytes, int32_t *err, minf_stream_t stream);
MINF_API int minf_kv_append_paged_q8(uint8_t *k_pool, uint8_t *v_pool, int64_t pool_rows, int row_width,
                                     const int32_t *block_table, int max_blocks, int block_rows, const float *k_rows,
                                     const float *v_rows, const int32_t *pos, int n_seq, int32_t *err,
                                     minf_stream_t stream);
MINF_API int minf_gqa_attn_decode_paged_q8(float *out, const float *q, const uint8_t *k_pool,
                                           const uint8_t *v_pool, int64_t pool_rows, const int32_t *block_table,
                                           int max_blocks, int block_rows, const int32_t *pos, int n_seq,
                                           int n_head, int n_kv_head, int hd, int hd_kv, float scale, void *ws,
                                           size_t ws_bytes, int32_t *err, minf_stream_t stream);
MINF_API int minf_layer_attn_step_paged_q8(float *xn, const float *h, const float *gain, float eps, int n_embd,
                                           float *q, float *k, const float *v, const int32_t *pos, int n_seq,
                                           uint8_t *k_pool, uint8_t *v_pool, int64_t pool_rows,
                                           const int32_t *block_table, int max_blocks, int block_rows, int n_head,
                                           int n_kv_head, int hd, int hd_kv, float theta, float freq_scale,
                                           int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                                           minf_stream_t stream);
MINF_API int minf_layer_attn_step_paged_f16(float *xn, const float *h, const float *gain, float eps, int n_embd,
                                            float *q, float *k, const float *v, const int32_t *pos, int n_seq,
                                            uint16_t *k_pool, uint16_t *v_pool, int64_t pool_rows,
                                            const int32_t *block_table, int max_blocks, int block_rows, int n_head,
                                            int n_kv_head, int hd, int hd_kv, float theta, float freq_scale,
                                            int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                                            minf_stream_t stream);

/*
 * The fused QKV decode op ([P3] §2.3: for a single token the three projection
 * matmuls, their biases, the two RoPEs and the two KV stores become one op),
 * here with the RMSNorm in front, for nt <= 16 tokens of one sequence:
 *   xn = RMSNorm(h) * gain                    ([P1] §3.2.1; xn [nt, n_embd])
 *   y  = w_qkv xn + b_qkv                     (w_qkv [n_out, n_embd] fp32, rows: the
 *        n_head*hd q outputs, then n_kv_head*hd_kv k outputs, then as many v outputs;
 *        b_qkv [n_out] or NULL)
 *   q [nt, n_head*hd] and k [nt, W] written rotated at pos ([P1] §3.2.2), v [nt, W];
 *   the rotated k and v stored at row pos of the regions [cap, W] ([P1] §3.2.3).
 * Each output is an fp32 dot product over n_embd (within 1e-5 + 1e-4|y| of an exact
 * one for unit-variance inputs and weights scaled by 1/sqrt(n_embd)).
 * Device errors: pos < 0 -> MINF_ERRBIT_ROPE_POS (q, k left unrotated) and
 * MINF_ERRBIT_STORE_POS; pos >= cap -> MINF_ERRBIT_STORE_POS (not stored).
 * Errors: MINF_ERR_UNSUPPORTED for nt > 16 or nt * n_embd * 4 > 227 KB (the normalized
 * tokens are held in shared memory); MINF_ERR_ARG for n_embd not a multiple of 4 or
 * unaligned pointers; MINF_ERR_GEOMETRY as elsewhere.
 * Early start: the op is a programmatic dependent launch and begins reading w_qkv and
 * b_qkv before the launch just before it on the stream has finished (h, gain, pos and
 * every output only after): the weights must not be written by that launch.
 *
 * minf_layer_attn_step_qkv: one decode token (nt = 1) from the hidden state h to the
 * attention output: the fused QKV op, then the split-KV decode attention over
 * [0, pos] (out [1, n_head*hd_kv]); ws as for minf_gqa_attn_decode with n_seq = 1.
 */
MINF_API int minf_fused_qkv(float *xn, const float *h, const float *gain, float eps, int n_embd,
                            const float *w_qkv, const float *b_qkv, const int32_t *pos, int nt, float *q, float *k,
                            float *v, float *k_reg, float *v_reg, int cap, int n_head, int n_kv_head, int hd,
                            int hd_kv, float theta, float freq_scale, int style, int32_t *err,
                            minf_stream_t stream);
MINF_API int minf_layer_attn_step_qkv(float *xn, const float *h, const float *gain, float eps, int n_embd,
                                      const float *w_qkv, const float *b_qkv, const int32_t *pos, float *q,
                                      float *k, float *v, float *k_reg, float *v_reg, int cap, int n_head,
                                      int n_kv_head, int hd, int hd_kv, float theta, float freq_scale, int style,
                                      float *out, void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream);

/*
 * SiLU times up ([P1] §3.2.5): y = gate / (1 + e^-gate) * up over n elements.
 * Errors: MINF_ERR_ARG for null pointers or n < 0.
 */
MINF_API int minf_silu_mul(float *y, const float *gate, const float *up, int64_t n, minf_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MINF_H */
