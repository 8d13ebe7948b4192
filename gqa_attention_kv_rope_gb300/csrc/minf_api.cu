// minf_api.cu -- the C ABI: argument validation, then the stream-ordered launches.
#include <cmath>

#include "minf_common.cuh"
#include "minf_kernels.h"

using namespace minf;

namespace {

inline cudaStream_t cs(minf_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

bool ok_f(const void *p) { return p != nullptr && aligned16(p); }

// Head geometry shared by every attention entry point.
int check_heads(int nh, int nk, int hd, int hd_kv) {
    if (nh <= 0 || nk <= 0 || hd <= 0 || hd_kv <= 0) return MINF_ERR_ARG;
    if (hd < hd_kv || nh % nk != 0) return MINF_ERR_GEOMETRY;  // hd < hd_kv is refused
    if ((hd & 1) || (hd_kv & 1)) return MINF_ERR_ARG;
    if (hd > 2 * kMaxHalf || hd_kv > 2 * kMaxHalf) return MINF_ERR_UNSUPPORTED;
    return MINF_OK;
}

int check_attn(int nh, int nk, int hd, int hd_kv) {
    int st = check_heads(nh, nk, hd, hd_kv);
    if (st != MINF_OK) return st;
    return decode_supported(nh, nk, hd, hd_kv) ? MINF_OK : MINF_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" {

const char *minf_status_string(int status) {
    switch (status) {
        case MINF_OK: return "ok";
        case MINF_ERR_ARG: return "invalid argument";
        case MINF_ERR_GEOMETRY: return "invalid head geometry (hd < hd_kv or n_head % n_kv_head != 0)";
        case MINF_ERR_UNSUPPORTED: return "shape not implemented by the kernels";
        case MINF_ERR_WORKSPACE: return "workspace missing or too small";
        case MINF_ERR_CUDA: return "CUDA launch failed";
        default: return "unknown status";
    }
}

int minf_version(void) { return 100; }

int minf_rope_freqs(float *freqs, int hd, float theta, float freq_scale) {
    if (!freqs || hd <= 0 || (hd & 1) || hd > 2 * kMaxHalf) return MINF_ERR_ARG;
    RopeTable t;
    rope_table(&t, hd, theta, freq_scale);
    for (int i = 0; i < hd / 2; ++i) freqs[i] = t.f[i];
    return MINF_OK;
}

int minf_rms_norm(float *y, const float *x, const float *w, int rows, int n, float eps,
                  minf_stream_t stream) {
    if (!y || !x || rows < 0 || n <= 0) return MINF_ERR_ARG;
    return launch_rms_norm(y, x, w, rows, n, eps, cs(stream));
}

int minf_rope(float *x, const int32_t *pos, int nt, int n_head, int hd, float theta,
              float freq_scale, int style, int32_t *err, minf_stream_t stream) {
    if (!x || !pos || !err || nt < 0 || n_head <= 0 || hd <= 0 || (hd & 1) || hd > 2 * kMaxHalf)
        return MINF_ERR_ARG;
    if (style != 0 && style != 1) return MINF_ERR_ARG;
    return launch_rope(x, pos, nt, n_head, hd, theta, freq_scale, style, err, cs(stream));
}

// Row widths each storage kind accepts: fp32 in float4s, binary16 in 16-byte pieces, Q8_0 in
// whole 32-value blocks.
static int row_multiple(int kv) { return kv == kKvQ8 ? 32 : (kv == kKvF16 ? 8 : 4); }

static int kv_append(void *k_reg, void *v_reg, int kv, int cap, int row_width, const float *k_rows,
                     const float *v_rows, const int32_t *pos, int nt, int32_t *err, minf_stream_t stream) {
    if (!ok_f(k_reg) || !ok_f(v_reg) || !ok_f(k_rows) || !ok_f(v_rows) || !pos || !err)
        return MINF_ERR_ARG;
    if (cap <= 0 || nt < 0 || row_width <= 0 || row_width % row_multiple(kv)) return MINF_ERR_ARG;
    if (kv == kKvQ8)
        return launch_kv_append_q8(k_reg, v_reg, cap, row_width, k_rows, v_rows, pos, nt, nullptr, nullptr, nullptr,
                                   0, 0, 0, err, cs(stream));
    return launch_kv_append(k_reg, v_reg, kv, cap, row_width, k_rows, v_rows, pos, nt, err, cs(stream));
}

int minf_kv_append_q8(uint8_t *k_reg, uint8_t *v_reg, int cap, int row_width, const float *k_rows,
                      const float *v_rows, const int32_t *pos, int nt, int32_t *err, minf_stream_t stream) {
    return kv_append(k_reg, v_reg, kKvQ8, cap, row_width, k_rows, v_rows, pos, nt, err, stream);
}

size_t minf_q8_row_bytes(int row_width) {
    return row_width > 0 && row_width % 32 == 0 ? static_cast<size_t>(q8_row_bytes(row_width)) : 0;
}

int minf_kv_append(float *k_reg, float *v_reg, int cap, int row_width, const float *k_rows,
                   const float *v_rows, const int32_t *pos, int nt, int32_t *err,
                   minf_stream_t stream) {
    return kv_append(k_reg, v_reg, kKvF32, cap, row_width, k_rows, v_rows, pos, nt, err, stream);
}

int minf_kv_append_f16(uint16_t *k_reg, uint16_t *v_reg, int cap, int row_width, const float *k_rows,
                       const float *v_rows, const int32_t *pos, int nt, int32_t *err, minf_stream_t stream) {
    return kv_append(k_reg, v_reg, kKvF16, cap, row_width, k_rows, v_rows, pos, nt, err, stream);
}

static int rope_kv(float *q, float *k, const float *v, const int32_t *pos, int nt, int nh, int nk,
                   int hd, int hd_kv, float theta, float freq_scale, int style, void *k_reg,
                   void *v_reg, int kv, const int64_t *row_off, const int32_t *caps, int cap,
                   int32_t *err, cudaStream_t s) {
    RopeKvArgs a = {};
    a.q = q;
    a.k = k;
    a.v = v;
    a.pos = pos;
    a.k_reg = k_reg;
    a.v_reg = v_reg;
    a.kv = kv;
    a.row_off = row_off;
    a.caps = caps;
    a.cap = cap;
    a.nt = nt;
    a.nh = nh;
    a.nk = nk;
    a.hd = hd;
    a.hd_kv = hd_kv;
    a.style = style;
    a.err = err;
    if (kv == kKvQ8) {  // rotate here, then quantize the rotated rows into the regions
        a.k_reg = a.v_reg = nullptr;
        const int st = launch_rope_kv_append(a, theta, freq_scale, s);
        if (st != MINF_OK) return st;
        return launch_kv_append_q8(k_reg, v_reg, cap, nk * hd_kv, k, v, pos, nt, row_off, caps, nullptr, 0, 0, 0, err,
                                   s);
    }
    return launch_rope_kv_append(a, theta, freq_scale, s);
}

static int rope_kv_append(float *q, float *k, const float *v, const int32_t *pos, int nt, int n_head,
                          int n_kv_head, int hd, int hd_kv, float theta, float freq_scale, int style,
                          void *k_reg, void *v_reg, int kv, int cap, int32_t *err, minf_stream_t stream) {
    int st = check_heads(n_head, n_kv_head, hd, hd_kv);
    if (st != MINF_OK) return st;
    if (!ok_f(q) || !ok_f(k) || !ok_f(v) || !ok_f(k_reg) || !ok_f(v_reg) || !pos || !err)
        return MINF_ERR_ARG;
    if (nt < 0 || cap <= 0 || (style != 0 && style != 1) || (n_kv_head * hd_kv) % row_multiple(kv))
        return MINF_ERR_ARG;
    return rope_kv(q, k, v, pos, nt, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style,
                   k_reg, v_reg, kv, nullptr, nullptr, cap, err, cs(stream));
}

// A block table over a pool of K/V rows (paged regions).
struct Paged {
    const int32_t *table;
    int max_blocks, block_rows, pool_blocks;
};

static int layer_prologue(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q, float *k,
                          const float *v, const int32_t *pos, int nt, int nh, int nk, int hd, int hd_kv, float theta,
                          float freq_scale, int style, void *k_reg, void *v_reg, int kv, const int64_t *row_off,
                          const int32_t *caps, int cap, int32_t *err, cudaStream_t s, const Paged *pg = nullptr) {
    RopeKvArgs a = {};
    if (pg) {
        a.table = pg->table;
        a.max_blocks = pg->max_blocks;
        a.block_rows = pg->block_rows;
        a.pool_blocks = pg->pool_blocks;
    }
    a.q = q;
    a.k = k;
    a.v = v;
    a.pos = pos;
    a.k_reg = k_reg;
    a.v_reg = v_reg;
    a.kv = kv;
    a.row_off = row_off;
    a.caps = caps;
    a.cap = cap;
    a.nt = nt;
    a.nh = nh;
    a.nk = nk;
    a.hd = hd;
    a.hd_kv = hd_kv;
    a.style = style;
    a.err = err;
    NormArgs nrm = {xn, h, gain, nt, n_embd, eps};
    if (kv == kKvQ8) {  // rotate in the prologue, then quantize the rotated rows into the regions
        a.k_reg = a.v_reg = nullptr;
        const int st = launch_layer_prologue(a, theta, freq_scale, nrm, s);
        if (st != MINF_OK) return st;
        return launch_kv_append_q8(k_reg, v_reg, cap, nk * hd_kv, k, v, pos, nt, row_off, caps,
                                   pg ? pg->table : nullptr, pg ? pg->max_blocks : 0, pg ? pg->block_rows : 0,
                                   pg ? pg->pool_blocks : 0, err, s);
    }
    return launch_layer_prologue(a, theta, freq_scale, nrm, s);
}

int minf_rope_kv_append(float *q, float *k, const float *v, const int32_t *pos, int nt,
                        int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                        float freq_scale, int style, float *k_reg, float *v_reg, int cap,
                        int32_t *err, minf_stream_t stream) {
    return rope_kv_append(q, k, v, pos, nt, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, k_reg,
                          v_reg, kKvF32, cap, err, stream);
}

int minf_rope_kv_append_q8(float *q, float *k, const float *v, const int32_t *pos, int nt, int n_head, int n_kv_head,
                           int hd, int hd_kv, float theta, float freq_scale, int style, uint8_t *k_reg, uint8_t *v_reg,
                           int cap, int32_t *err, minf_stream_t stream) {
    return rope_kv_append(q, k, v, pos, nt, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, k_reg, v_reg,
                          kKvQ8, cap, err, stream);
}

int minf_rope_kv_append_f16(float *q, float *k, const float *v, const int32_t *pos, int nt, int n_head,
                            int n_kv_head, int hd, int hd_kv, float theta, float freq_scale, int style,
                            uint16_t *k_reg, uint16_t *v_reg, int cap, int32_t *err, minf_stream_t stream) {
    return rope_kv_append(q, k, v, pos, nt, n_head, n_kv_head, hd, hd_kv, theta, freq_scale, style, k_reg,
                          v_reg, kKvF16, cap, err, stream);
}

size_t minf_attn_decode_workspace_bytes(int n_seq, int n_head, int n_kv_head, int hd_kv,
                                        int max_cap) {
    return decode_workspace_bytes(n_seq, n_head, n_kv_head, hd_kv, max_cap);
}

size_t minf_attn_prefill_workspace_bytes(int nt, int n_head, int n_kv_head, int hd_kv, int cap) {
    (void)n_kv_head;
    return prefill_workspace_bytes(nt, n_head, hd_kv, cap);
}

static PrefillArgs prefill_args(float *out, const float *q, const void *k_reg, const void *v_reg, int kv, int cap,
                                const int32_t *pos, int nt, int nh, int nk, int hd, int hd_kv, float scale,
                                void *ws, size_t ws_bytes, int32_t *err, bool pdl) {
    PrefillArgs a = {};
    a.pdl = pdl;
    a.ws = ws;
    a.ws_bytes = ws_bytes;
    a.out = out;
    a.q = q;
    a.k_reg = k_reg;
    a.v_reg = v_reg;
    a.kv = kv;
    a.pos = pos;
    a.err = err;
    a.nt = nt;
    a.nh = nh;
    a.nk = nk;
    a.hd = hd;
    a.hd_kv = hd_kv;
    a.cap = cap;
    a.scale = scale;
    return a;
}

static int prefill(float *out, const float *q, const void *k_reg, const void *v_reg, int kv, int cap,
                   const int32_t *pos, int nt, int nh, int nk, int hd, int hd_kv, float scale,
                   void *ws, size_t ws_bytes, int32_t *err, cudaStream_t s, bool pdl = false) {
    return launch_prefill(
        prefill_args(out, q, k_reg, v_reg, kv, cap, pos, nt, nh, nk, hd, hd_kv, scale, ws, ws_bytes, err, pdl), s);
}

static DecodeArgs decode_args(float *out, const float *q, const void *k_reg,
                              const void *v_reg, int kv, const int64_t *row_off, const int32_t *caps,
                              int cap, const int32_t *pos, int n_seq, int nh, int nk, int hd,
                              int hd_kv, float scale, void *ws, size_t ws_bytes, int32_t *err,
                              long long arena_rows = 0) {
    DecodeArgs d = {};
    d.arena_rows = arena_rows;
    d.out = out;
    d.q = q;
    d.k_reg = k_reg;
    d.v_reg = v_reg;
    d.kv = kv;
    d.row_off = row_off;
    d.caps = caps;
    d.cap = cap;
    d.pos = pos;
    d.n_seq = n_seq;
    d.nh = nh;
    d.nk = nk;
    d.hd = hd;
    d.hd_kv = hd_kv;
    d.scale = scale;
    d.err = err;
    d.ws = ws;
    d.ws_bytes = ws_bytes;
    return d;
}

static int decode(float *out, const float *q, const void *k_reg, const void *v_reg, int kv,
                  const int64_t *row_off, const int32_t *caps, int cap, const int32_t *pos,
                  int n_seq, int nh, int nk, int hd, int hd_kv, float scale, void *ws,
                  size_t ws_bytes, int32_t *err, cudaStream_t s, long long arena_rows = 0) {
    return launch_decode(decode_args(out, q, k_reg, v_reg, kv, row_off, caps, cap, pos, n_seq, nh, nk,
                                     hd, hd_kv, scale, ws, ws_bytes, err, arena_rows),
                         s);
}

static int gqa_attn_decode(float *out, const float *q, const void *k_reg, const void *v_reg, int kv,
                           const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap, int64_t arena_rows,
                           const int32_t *pos, int n_seq, int n_head, int n_kv_head, int hd, int hd_kv,
                           float scale, void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    int st = check_attn(n_head, n_kv_head, hd, hd_kv);
    if (st != MINF_OK) return st;
    if (!ok_f(out) || !ok_f(q) || !ok_f(k_reg) || !ok_f(v_reg) || !pos || !err) return MINF_ERR_ARG;
    if (n_seq < 0 || max_cap <= 0 || (seq_row_off && arena_rows <= 0)) return MINF_ERR_ARG;
    return decode(out, q, k_reg, v_reg, kv, seq_row_off, seq_cap, max_cap, pos, n_seq, n_head,
                  n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err, cs(stream), arena_rows);
}

int minf_gqa_attn_decode(float *out, const float *q, const float *k_reg, const float *v_reg,
                         const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap,
                         int64_t arena_rows, const int32_t *pos, int n_seq, int n_head,
                         int n_kv_head, int hd, int hd_kv, float scale, void *ws,
                         size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    return gqa_attn_decode(out, q, k_reg, v_reg, kKvF32, seq_row_off, seq_cap, max_cap, arena_rows, pos, n_seq,
                           n_head, n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err, stream);
}

int minf_gqa_attn_decode_q8(float *out, const float *q, const uint8_t *k_reg, const uint8_t *v_reg,
                            const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap, int64_t arena_rows,
                            const int32_t *pos, int n_seq, int n_head, int n_kv_head, int hd, int hd_kv, float scale,
                            void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    if ((n_kv_head * hd_kv) % 32) return MINF_ERR_ARG;
    return gqa_attn_decode(out, q, k_reg, v_reg, kKvQ8, seq_row_off, seq_cap, max_cap, arena_rows, pos, n_seq, n_head,
                           n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err, stream);
}

int minf_gqa_attn_decode_f16(float *out, const float *q, const uint16_t *k_reg, const uint16_t *v_reg,
                             const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap, int64_t arena_rows,
                             const int32_t *pos, int n_seq, int n_head, int n_kv_head, int hd, int hd_kv,
                             float scale, void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    return gqa_attn_decode(out, q, k_reg, v_reg, kKvF16, seq_row_off, seq_cap, max_cap, arena_rows, pos, n_seq,
                           n_head, n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err, stream);
}

static int gqa_attn_prefill(float *out, const float *q, const void *k_reg, const void *v_reg, int kv, int cap,
                            const int32_t *pos, int nt, int n_head, int n_kv_head, int hd, int hd_kv, float scale,
                            void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    int st = check_attn(n_head, n_kv_head, hd, hd_kv);
    if (st != MINF_OK) return st;
    if (!ok_f(out) || !ok_f(q) || !ok_f(k_reg) || !ok_f(v_reg) || !pos || !err) return MINF_ERR_ARG;
    if (nt < 0 || cap <= 0) return MINF_ERR_ARG;
    return prefill(out, q, k_reg, v_reg, kv, cap, pos, nt, n_head, n_kv_head, hd, hd_kv, scale, ws,
                   ws_bytes, err, cs(stream));
}

int minf_gqa_attn_prefill(float *out, const float *q, const float *k_reg, const float *v_reg,
                          int cap, const int32_t *pos, int nt, int n_head, int n_kv_head, int hd,
                          int hd_kv, float scale, void *ws, size_t ws_bytes, int32_t *err,
                          minf_stream_t stream) {
    return gqa_attn_prefill(out, q, k_reg, v_reg, kKvF32, cap, pos, nt, n_head, n_kv_head, hd, hd_kv, scale, ws,
                            ws_bytes, err, stream);
}

int minf_gqa_attn_prefill_q8(float *out, const float *q, const uint8_t *k_reg, const uint8_t *v_reg, int cap,
                             const int32_t *pos, int nt, int n_head, int n_kv_head, int hd, int hd_kv, float scale,
                             void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    if ((n_kv_head * hd_kv) % 32) return MINF_ERR_ARG;
    return gqa_attn_prefill(out, q, k_reg, v_reg, kKvQ8, cap, pos, nt, n_head, n_kv_head, hd, hd_kv, scale, ws,
                            ws_bytes, err, stream);
}

int minf_gqa_attn_prefill_f16(float *out, const float *q, const uint16_t *k_reg, const uint16_t *v_reg, int cap,
                              const int32_t *pos, int nt, int n_head, int n_kv_head, int hd, int hd_kv, float scale,
                              void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    return gqa_attn_prefill(out, q, k_reg, v_reg, kKvF16, cap, pos, nt, n_head, n_kv_head, hd, hd_kv, scale, ws,
                            ws_bytes, err, stream);
}

static int layer_attn_step(float *xn, const float *h, const float *gain, float eps, int n_embd,
                           float *q, float *k, const float *v, const int32_t *pos, int nt,
                           void *k_reg, void *v_reg, int kv, int cap, int n_head, int n_kv_head, int hd,
                           int hd_kv, float theta, float freq_scale, int style, float *out,
                           void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream,
                           bool chained = false) {
    int st = check_attn(n_head, n_kv_head, hd, hd_kv);
    if (st != MINF_OK) return st;
    if (!xn || !h || n_embd <= 0 || nt < 0 || cap <= 0 || (style != 0 && style != 1))
        return MINF_ERR_ARG;
    if (!ok_f(q) || !ok_f(k) || !ok_f(v) || !ok_f(k_reg) || !ok_f(v_reg) || !ok_f(out) || !pos ||
        !err)
        return MINF_ERR_ARG;
    if (nt == 0) return MINF_OK;
    const size_t need = nt == 1 ? decode_workspace_bytes(1, n_head, n_kv_head, hd_kv, cap)
                                : prefill_workspace_bytes(nt, n_head, hd_kv, cap);
    if (need && (!ws || ws_bytes < need)) return MINF_ERR_WORKSPACE;
    cudaStream_t s = cs(stream);
    const float scale = 1.0f / sqrtf(static_cast<float>(hd));
    if (nt == 1 && fused_step_supported(n_head, n_kv_head, hd, hd_kv, n_embd) && aligned16(h) &&
        aligned16(xn) && (!gain || aligned16(gain))) {
        // one launch: RMSNorm, RoPE on q and k, the K/V append and split-KV attention
        DecodeArgs d = decode_args(out, q, k_reg, v_reg, kv, nullptr, nullptr, cap, pos, 1, n_head,
                                   n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err);
        // a programmatic dependent launch either way (its start overlaps the launch before it);
        // chained: positions and cached rows read before the dependency wait
        DecodeStepExtra x = {k, v, xn, h, gain, eps, theta, freq_scale, n_embd, style, true, chained};
        return launch_decode_step(d, x, s);
    }
    if (nt > 1 && kv != kKvQ8) {
        // one launch: the row work, a grid barrier, then the attention items
        const PrefillArgs pa = prefill_args(out, q, k_reg, v_reg, kv, cap, pos, nt, n_head, n_kv_head, hd, hd_kv,
                                            scale, ws, ws_bytes, err, true);
        const PrefillStepExtra x = {q, k, v, xn, h, gain, eps, theta, freq_scale, n_embd, style};
        st = launch_prefill_step(pa, x, s);
        if (st != MINF_ERR_UNSUPPORTED) return st;
    }
    // one launch for RMSNorm, RoPE and the store, then the attention
    st = layer_prologue(xn, h, gain, eps, n_embd, q, k, v, pos, nt, n_head, n_kv_head, hd, hd_kv, theta,
                        freq_scale, style, k_reg, v_reg, kv, nullptr, nullptr, cap, err, s);
    if (st != MINF_OK) return st;
    if (nt == 1)  // the decode kernel streams cached rows before its wait: no early start after a store
        return decode(out, q, k_reg, v_reg, kv, nullptr, nullptr, cap, pos, 1, n_head, n_kv_head, hd,
                      hd_kv, scale, ws, ws_bytes, err, s);
    return prefill(out, q, k_reg, v_reg, kv, cap, pos, nt, n_head, n_kv_head, hd, hd_kv, scale, ws, ws_bytes,
                   err, s, true);
}

int minf_layer_attn_step(float *xn, const float *h, const float *gain, float eps, int n_embd,
                         float *q, float *k, const float *v, const int32_t *pos, int nt,
                         float *k_reg, float *v_reg, int cap, int n_head, int n_kv_head, int hd,
                         int hd_kv, float theta, float freq_scale, int style, float *out,
                         void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    return layer_attn_step(xn, h, gain, eps, n_embd, q, k, v, pos, nt, k_reg, v_reg, kKvF32, cap, n_head,
                           n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, ws_bytes, err, stream);
}

int minf_layer_attn_step_q8(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q, float *k,
                            const float *v, const int32_t *pos, int nt, uint8_t *k_reg, uint8_t *v_reg, int cap,
                            int n_head, int n_kv_head, int hd, int hd_kv, float theta, float freq_scale, int style,
                            float *out, void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    if ((n_kv_head * hd_kv) % 32) return MINF_ERR_ARG;
    return layer_attn_step(xn, h, gain, eps, n_embd, q, k, v, pos, nt, k_reg, v_reg, kKvQ8, cap, n_head, n_kv_head,
                           hd, hd_kv, theta, freq_scale, style, out, ws, ws_bytes, err, stream);
}

int minf_layer_attn_step_f16(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q,
                             float *k, const float *v, const int32_t *pos, int nt, uint16_t *k_reg,
                             uint16_t *v_reg, int cap, int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                             float freq_scale, int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                             minf_stream_t stream) {
    return layer_attn_step(xn, h, gain, eps, n_embd, q, k, v, pos, nt, k_reg, v_reg, kKvF16, cap, n_head,
                           n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, ws_bytes, err, stream);
}

// The same steps with early start (the launch before writes neither pos nor cached rows).
int minf_layer_attn_step_chained(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q,
                                 float *k, const float *v, const int32_t *pos, int nt, float *k_reg, float *v_reg,
                                 int cap, int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                                 float freq_scale, int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                                 minf_stream_t stream) {
    return layer_attn_step(xn, h, gain, eps, n_embd, q, k, v, pos, nt, k_reg, v_reg, kKvF32, cap, n_head,
                           n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, ws_bytes, err, stream, true);
}

int minf_layer_attn_step_chained_f16(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q,
                                     float *k, const float *v, const int32_t *pos, int nt, uint16_t *k_reg,
                                     uint16_t *v_reg, int cap, int n_head, int n_kv_head, int hd, int hd_kv,
                                     float theta, float freq_scale, int style, float *out, void *ws,
                                     size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    return layer_attn_step(xn, h, gain, eps, n_embd, q, k, v, pos, nt, k_reg, v_reg, kKvF16, cap, n_head,
                           n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, ws_bytes, err, stream, true);
}

int minf_layer_attn_step_chained_q8(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q,
                                    float *k, const float *v, const int32_t *pos, int nt, uint8_t *k_reg,
                                    uint8_t *v_reg, int cap, int n_head, int n_kv_head, int hd, int hd_kv,
                                    float theta, float freq_scale, int style, float *out, void *ws,
                                    size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    if ((n_kv_head * hd_kv) % 32) return MINF_ERR_ARG;
    return layer_attn_step(xn, h, gain, eps, n_embd, q, k, v, pos, nt, k_reg, v_reg, kKvQ8, cap, n_head,
                           n_kv_head, hd, hd_kv, theta, freq_scale, style, out, ws, ws_bytes, err, stream, true);
}

static int layer_attn_step_batched(float *xn, const float *h, const float *gain, float eps,
                                   int n_embd, float *q, float *k, const float *v,
                                   const int32_t *pos, int n_seq, void *k_arena, void *v_arena, int kv,
                                   const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap,
                                   int64_t arena_rows,
                                   int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                                   float freq_scale, int style, float *out, void *ws,
                                   size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    int st = check_attn(n_head, n_kv_head, hd, hd_kv);
    if (st != MINF_OK) return st;
    if (!xn || !h || n_embd <= 0 || n_seq < 0 || max_cap <= 0 || (style != 0 && style != 1))
        return MINF_ERR_ARG;
    if (!ok_f(q) || !ok_f(k) || !ok_f(v) || !ok_f(k_arena) || !ok_f(v_arena) || !ok_f(out) ||
        !pos || !err || !seq_row_off || !seq_cap || arena_rows <= 0)
        return MINF_ERR_ARG;
    if (n_seq == 0) return MINF_OK;
    cudaStream_t s = cs(stream);
    const float scale = 1.0f / sqrtf(static_cast<float>(hd));
    if (fused_step_supported(n_head, n_kv_head, hd, hd_kv, n_embd) && aligned16(h) &&
        aligned16(xn) && (!gain || aligned16(gain))) {
        DecodeArgs d = decode_args(out, q, k_arena, v_arena, kv, seq_row_off, seq_cap, max_cap, pos,
                                   n_seq, n_head, n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err,
                                   arena_rows);
        DecodeStepExtra x = {k, v, xn, h, gain, eps, theta, freq_scale, n_embd, style, false, false};
        return launch_decode_step(d, x, s);
    }
    st = layer_prologue(xn, h, gain, eps, n_embd, q, k, v, pos, n_seq, n_head, n_kv_head, hd, hd_kv, theta,
                        freq_scale, style, k_arena, v_arena, kv, seq_row_off, seq_cap, max_cap, err, s);
    if (st != MINF_OK) return st;
    return decode(out, q, k_arena, v_arena, kv, seq_row_off, seq_cap, max_cap, pos, n_seq, n_head,
                  n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err, s, arena_rows);
}

int minf_layer_attn_step_batched(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q,
                                 float *k, const float *v, const int32_t *pos, int n_seq, float *k_arena,
                                 float *v_arena, const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap,
                                 int64_t arena_rows, int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                                 float freq_scale, int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                                 minf_stream_t stream) {
    return layer_attn_step_batched(xn, h, gain, eps, n_embd, q, k, v, pos, n_seq, k_arena, v_arena, kKvF32,
                                   seq_row_off, seq_cap, max_cap, arena_rows, n_head, n_kv_head, hd, hd_kv, theta,
                                   freq_scale, style, out, ws, ws_bytes, err, stream);
}

int minf_layer_attn_step_batched_q8(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q,
                                    float *k, const float *v, const int32_t *pos, int n_seq, uint8_t *k_arena,
                                    uint8_t *v_arena, const int64_t *seq_row_off, const int32_t *seq_cap, int max_cap,
                                    int64_t arena_rows, int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                                    float freq_scale, int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                                    minf_stream_t stream) {
    if ((n_kv_head * hd_kv) % 32) return MINF_ERR_ARG;
    return layer_attn_step_batched(xn, h, gain, eps, n_embd, q, k, v, pos, n_seq, k_arena, v_arena, kKvQ8,
                                   seq_row_off, seq_cap, max_cap, arena_rows, n_head, n_kv_head, hd, hd_kv, theta,
                                   freq_scale, style, out, ws, ws_bytes, err, stream);
}

int minf_layer_attn_step_batched_f16(float *xn, const float *h, const float *gain, float eps, int n_embd,
                                     float *q, float *k, const float *v, const int32_t *pos, int n_seq,
                                     uint16_t *k_arena, uint16_t *v_arena, const int64_t *seq_row_off,
                                     const int32_t *seq_cap, int max_cap, int64_t arena_rows, int n_head,
                                     int n_kv_head, int hd, int hd_kv, float theta, float freq_scale, int style,
                                     float *out, void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    return layer_attn_step_batched(xn, h, gain, eps, n_embd, q, k, v, pos, n_seq, k_arena, v_arena, kKvF16,
                                   seq_row_off, seq_cap, max_cap, arena_rows, n_head, n_kv_head, hd, hd_kv, theta,
                                   freq_scale, style, out, ws, ws_bytes, err, stream);
}

int minf_silu_mul(float *y, const float *gate, const float *up, int64_t n, minf_stream_t stream) {
    if (!y || !gate || !up || n < 0) return MINF_ERR_ARG;
    return launch_silu_mul(y, gate, up, n, cs(stream));
}

// ----------------------------------------------------------------------------- paged regions
// "IV.2: Zero-copy KV cache": the paged cache keeps a sequence as scattered fixed-size blocks
// of a shared pool; a table per sequence names them ("13 . The decode loop and graph reuse",
// §2.2: the window the attention reads is an explicit input).

static int check_paged(const void *k_pool, const void *v_pool, int kv, int64_t pool_rows, const int32_t *table,
                       int max_blocks, int block_rows, Paged *pg) {
    if (!ok_f(k_pool) || !ok_f(v_pool) || !table || pool_rows <= 0 || max_blocks <= 0) return MINF_ERR_ARG;
    if (block_rows < 16 || block_rows > 4096 || (block_rows & (block_rows - 1))) return MINF_ERR_UNSUPPORTED;
    if (pool_rows % block_rows || static_cast<long long>(max_blocks) * block_rows > 0x7fffffffLL - 4096 ||
        pool_rows > 0x7fffffffLL - 4096)
        return MINF_ERR_UNSUPPORTED;
    (void)kv;
    pg->table = table;
    pg->max_blocks = max_blocks;
    pg->block_rows = block_rows;
    pg->pool_blocks = static_cast<int>(pool_rows / block_rows);
    return MINF_OK;
}

static void set_paged(DecodeArgs &d, const Paged &pg, int64_t pool_rows) {
    d.table = pg.table;
    d.max_blocks = pg.max_blocks;
    d.block_rows = pg.block_rows;
    d.arena_rows = pool_rows;
}

static int kv_append_paged(void *k_pool, void *v_pool, int kv, int64_t pool_rows, int row_width,
                           const int32_t *table, int max_blocks, int block_rows, const float *k_rows,
                           const float *v_rows, const int32_t *pos, int n_seq, int32_t *err, minf_stream_t stream) {
    Paged pg;
    int st = check_paged(k_pool, v_pool, kv, pool_rows, table, max_blocks, block_rows, &pg);
    if (st != MINF_OK) return st;
    if (!ok_f(k_rows) || !ok_f(v_rows) || !pos || !err || n_seq < 0 || row_width <= 0 ||
        row_width % row_multiple(kv))
        return MINF_ERR_ARG;
    if (kv == kKvQ8)
        return launch_kv_append_q8(k_pool, v_pool, 0, row_width, k_rows, v_rows, pos, n_seq, nullptr, nullptr, table,
                                   max_blocks, block_rows, pg.pool_blocks, err, cs(stream));
    return launch_kv_append_paged(k_pool, v_pool, kv, pg.pool_blocks, block_rows, row_width, table, max_blocks,
                                  k_rows, v_rows, pos, n_seq, err, cs(stream));
}

int minf_kv_append_paged(float *k_pool, float *v_pool, int64_t pool_rows, int row_width, const int32_t *block_table,
                         int max_blocks, int block_rows, const float *k_rows, const float *v_rows, const int32_t *pos,
                         int n_seq, int32_t *err, minf_stream_t stream) {
    return kv_append_paged(k_pool, v_pool, kKvF32, pool_rows, row_width, block_table, max_blocks, block_rows, k_rows,
                           v_rows, pos, n_seq, err, stream);
}

int minf_kv_append_paged_q8(uint8_t *k_pool, uint8_t *v_pool, int64_t pool_rows, int row_width,
                            const int32_t *block_table, int max_blocks, int block_rows, const float *k_rows,
                            const float *v_rows, const int32_t *pos, int n_seq, int32_t *err, minf_stream_t stream) {
    return kv_append_paged(k_pool, v_pool, kKvQ8, pool_rows, row_width, block_table, max_blocks, block_rows, k_rows,
                           v_rows, pos, n_seq, err, stream);
}

int minf_kv_append_paged_f16(uint16_t *k_pool, uint16_t *v_pool, int64_t pool_rows, int row_width,
                             const int32_t *block_table, int max_blocks, int block_rows, const float *k_rows,
                             const float *v_rows, const int32_t *pos, int n_seq, int32_t *err, minf_stream_t stream) {
    return kv_append_paged(k_pool, v_pool, kKvF16, pool_rows, row_width, block_table, max_blocks, block_rows, k_rows,
                           v_rows, pos, n_seq, err, stream);
}

static int gqa_attn_decode_paged(float *out, const float *q, const void *k_pool, const void *v_pool, int kv,
                                 int64_t pool_rows, const int32_t *table, int max_blocks, int block_rows,
                                 const int32_t *pos, int n_seq, int n_head, int n_kv_head, int hd, int hd_kv,
                                 float scale, void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    int st = check_attn(n_head, n_kv_head, hd, hd_kv);
    if (st != MINF_OK) return st;
    Paged pg;
    st = check_paged(k_pool, v_pool, kv, pool_rows, table, max_blocks, block_rows, &pg);
    if (st != MINF_OK) return st;
    if (!ok_f(out) || !ok_f(q) || !pos || !err || n_seq < 0) return MINF_ERR_ARG;
    DecodeArgs d = decode_args(out, q, k_pool, v_pool, kv, nullptr, nullptr, max_blocks * block_rows, pos, n_seq,
                               n_head, n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err);
    set_paged(d, pg, pool_rows);
    return launch_decode(d, cs(stream));
}

int minf_gqa_attn_decode_paged(float *out, const float *q, const float *k_pool, const float *v_pool,
                               int64_t pool_rows, const int32_t *block_table, int max_blocks, int block_rows,
                               const int32_t *pos, int n_seq, int n_head, int n_kv_head, int hd, int hd_kv,
                               float scale, void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    return gqa_attn_decode_paged(out, q, k_pool, v_pool, kKvF32, pool_rows, block_table, max_blocks, block_rows, pos,
                                 n_seq, n_head, n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err, stream);
}

int minf_gqa_attn_decode_paged_q8(float *out, const float *q, const uint8_t *k_pool, const uint8_t *v_pool,
                                  int64_t pool_rows, const int32_t *block_table, int max_blocks, int block_rows,
                                  const int32_t *pos, int n_seq, int n_head, int n_kv_head, int hd, int hd_kv,
                                  float scale, void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    if ((n_kv_head * hd_kv) % 32) return MINF_ERR_ARG;
    return gqa_attn_decode_paged(out, q, k_pool, v_pool, kKvQ8, pool_rows, block_table, max_blocks, block_rows, pos,
                                 n_seq, n_head, n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err, stream);
}

int minf_gqa_attn_decode_paged_f16(float *out, const float *q, const uint16_t *k_pool, const uint16_t *v_pool,
                                   int64_t pool_rows, const int32_t *block_table, int max_blocks, int block_rows,
                                   const int32_t *pos, int n_seq, int n_head, int n_kv_head, int hd, int hd_kv,
                                   float scale, void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    return gqa_attn_decode_paged(out, q, k_pool, v_pool, kKvF16, pool_rows, block_table, max_blocks, block_rows, pos,
                                 n_seq, n_head, n_kv_head, hd, hd_kv, scale, ws, ws_bytes, err, stream);
}

static int layer_attn_step_paged(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q,
                                 float *k, const float *v, const int32_t *pos, int n_seq, void *k_pool, void *v_pool,
                                 int kv, int64_t pool_rows, const int32_t *table, int max_blocks, int block_rows,
                                 int n_head, int n_kv_head, int hd, int hd_kv, float theta, float freq_scale,
                                 int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                                 minf_stream_t stream) {
    int st = check_attn(n_head, n_kv_head, hd, hd_kv);
    if (st != MINF_OK) return st;
    Paged pg;
    st = check_paged(k_pool, v_pool, kv, pool_rows, table, max_blocks, block_rows, &pg);
    if (st != MINF_OK) return st;
    if (!xn || !h || n_embd <= 0 || n_seq < 0 || (style != 0 && style != 1)) return MINF_ERR_ARG;
    if (!ok_f(q) || !ok_f(k) || !ok_f(v) || !ok_f(out) || !pos || !err) return MINF_ERR_ARG;
    if (n_seq == 0) return MINF_OK;
    cudaStream_t s = cs(stream);
    const float scale = 1.0f / sqrtf(static_cast<float>(hd));
    const int cap = max_blocks * block_rows;
    DecodeArgs d = decode_args(out, q, k_pool, v_pool, kv, nullptr, nullptr, cap, pos, n_seq, n_head, n_kv_head, hd,
                               hd_kv, scale, ws, ws_bytes, err);
    set_paged(d, pg, pool_rows);
    if (fused_step_supported(n_head, n_kv_head, hd, hd_kv, n_embd) && aligned16(h) && aligned16(xn) &&
        (!gain || aligned16(gain))) {
        DecodeStepExtra x = {k, v, xn, h, gain, eps, theta, freq_scale, n_embd, style, false, false};
        return launch_decode_step(d, x, s);
    }
    st = layer_prologue(xn, h, gain, eps, n_embd, q, k, v, pos, n_seq, n_head, n_kv_head, hd, hd_kv, theta,
                        freq_scale, style, k_pool, v_pool, kv, nullptr, nullptr, cap, err, s, &pg);
    if (st != MINF_OK) return st;
    return launch_decode(d, s);
}

int minf_layer_attn_step_paged(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q, float *k,
                               const float *v, const int32_t *pos, int n_seq, float *k_pool, float *v_pool,
                               int64_t pool_rows, const int32_t *block_table, int max_blocks, int block_rows,
                               int n_head, int n_kv_head, int hd, int hd_kv, float theta, float freq_scale, int style,
                               float *out, void *ws, size_t ws_bytes, int32_t *err, minf_stream_t stream) {
    return layer_attn_step_paged(xn, h, gain, eps, n_embd, q, k, v, pos, n_seq, k_pool, v_pool, kKvF32, pool_rows,
                                 block_table, max_blocks, block_rows, n_head, n_kv_head, hd, hd_kv, theta, freq_scale,
                                 style, out, ws, ws_bytes, err, stream);
}

int minf_layer_attn_step_paged_q8(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q,
                                  float *k, const float *v, const int32_t *pos, int n_seq, uint8_t *k_pool,
                                  uint8_t *v_pool, int64_t pool_rows, const int32_t *block_table, int max_blocks,
                                  int block_rows, int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                                  float freq_scale, int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                                  minf_stream_t stream) {
    if ((n_kv_head * hd_kv) % 32) return MINF_ERR_ARG;
    return layer_attn_step_paged(xn, h, gain, eps, n_embd, q, k, v, pos, n_seq, k_pool, v_pool, kKvQ8, pool_rows,
                                 block_table, max_blocks, block_rows, n_head, n_kv_head, hd, hd_kv, theta, freq_scale,
                                 style, out, ws, ws_bytes, err, stream);
}

int minf_layer_attn_step_paged_f16(float *xn, const float *h, const float *gain, float eps, int n_embd, float *q,
                                   float *k, const float *v, const int32_t *pos, int n_seq, uint16_t *k_pool,
                                   uint16_t *v_pool, int64_t pool_rows, const int32_t *block_table, int max_blocks,
                                   int block_rows, int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                                   float freq_scale, int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                                   minf_stream_t stream) {
    return layer_attn_step_paged(xn, h, gain, eps, n_embd, q, k, v, pos, n_seq, k_pool, v_pool, kKvF16, pool_rows,
                                 block_table, max_blocks, block_rows, n_head, n_kv_head, hd, hd_kv, theta, freq_scale,
                                 style, out, ws, ws_bytes, err, stream);
}

// ----------------------------------------------------------------------------- fused QKV op
// "13 . The decode loop and graph reuse", §2.3: the decode step's three projections, biases,
// RoPEs and KV stores as one op (here with the RMSNorm in front).

static int fused_qkv(float *xn, const float *h, const float *gain, float eps, int n_embd, const float *w_qkv,
                     const float *b_qkv, const int32_t *pos, int nt, float *q, float *k, float *v, float *k_reg,
                     float *v_reg, int cap, int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                     float freq_scale, int style, int32_t *err, cudaStream_t s) {
    int st = check_heads(n_head, n_kv_head, hd, hd_kv);
    if (st != MINF_OK) return st;
    if (!ok_f(xn) || !ok_f(h) || (gain && !ok_f(gain)) || !ok_f(w_qkv) || !ok_f(q) || !ok_f(k) || !ok_f(v) ||
        !ok_f(k_reg) || !ok_f(v_reg) || !pos || !err)
        return MINF_ERR_ARG;
    if (n_embd <= 0 || n_embd % 4 || nt < 0 || cap <= 0 || (style != 0 && style != 1)) return MINF_ERR_ARG;
    if (nt > kQkvMaxTok) return MINF_ERR_UNSUPPORTED;
    QkvArgs a = {};
    a.xn = xn;
    a.h = h;
    a.gain = gain;
    a.eps = eps;
    a.n_embd = n_embd;
    a.w = w_qkv;
    a.b = b_qkv;
    a.pos = pos;
    a.nt = nt;
    a.q = q;
    a.k = k;
    a.v = v;
    a.k_reg = k_reg;
    a.v_reg = v_reg;
    a.cap = cap;
    a.nh = n_head;
    a.nk = n_kv_head;
    a.hd = hd;
    a.hd_kv = hd_kv;
    a.style = style;
    a.err = err;
    return launch_fused_qkv(a, theta, freq_scale, s);
}

int minf_fused_qkv(float *xn, const float *h, const float *gain, float eps, int n_embd, const float *w_qkv,
                   const float *b_qkv, const int32_t *pos, int nt, float *q, float *k, float *v, float *k_reg,
                   float *v_reg, int cap, int n_head, int n_kv_head, int hd, int hd_kv, float theta, float freq_scale,
                   int style, int32_t *err, minf_stream_t stream) {
    return fused_qkv(xn, h, gain, eps, n_embd, w_qkv, b_qkv, pos, nt, q, k, v, k_reg, v_reg, cap, n_head, n_kv_head,
                     hd, hd_kv, theta, freq_scale, style, err, cs(stream));
}

int minf_layer_attn_step_qkv(float *xn, const float *h, const float *gain, float eps, int n_embd, const float *w_qkv,
                             const float *b_qkv, const int32_t *pos, float *q, float *k, float *v, float *k_reg,
                             float *v_reg, int cap, int n_head, int n_kv_head, int hd, int hd_kv, float theta,
                             float freq_scale, int style, float *out, void *ws, size_t ws_bytes, int32_t *err,
                             minf_stream_t stream) {
    int st = check_attn(n_head, n_kv_head, hd, hd_kv);
    if (st != MINF_OK) return st;
    if (!ok_f(out)) return MINF_ERR_ARG;
    const size_t need = decode_workspace_bytes(1, n_head, n_kv_head, hd_kv, cap);
    if (!ws || ws_bytes < need) return MINF_ERR_WORKSPACE;
    cudaStream_t s = cs(stream);
    st = fused_qkv(xn, h, gain, eps, n_embd, w_qkv, b_qkv, pos, 1, q, k, v, k_reg, v_reg, cap, n_head, n_kv_head, hd,
                   hd_kv, theta, freq_scale, style, err, s);
    if (st != MINF_OK) return st;
    const float scale = 1.0f / sqrtf(static_cast<float>(hd));
    return decode(out, q, k_reg, v_reg, kKvF32, nullptr, nullptr, cap, pos, 1, n_head, n_kv_head, hd, hd_kv, scale,
                  ws, ws_bytes, err, s);
}

}  // extern "C"
