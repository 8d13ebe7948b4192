/*
 * minf_oracle.c -- the CPU oracle for the attention stage (TEST INFRASTRUCTURE).
 *
 * This file is test infrastructure, not part of the product.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library: every
 * formula below is written out again, plainly, from the pages it cites.
 *
 * Sources (page title, section):
 *   [P1] "11 . Attention, vec ops, and the KV cache" (minfer walkthrough)
 *   [P2] "IV.2: Zero-copy KV cache"
 *   [P3] "13 . The decode loop and graph reuse" (minfer walkthrough)
 *
 * Precision follows what [P1] fixes: fp32 data, fp32 dot products and fp32
 * weighted sums, an f64 sum of squares in RMSNorm and an f64 softmax
 * denominator.  The brute-force reference (orc_attn_bruteforce_f64) is fp64
 * throughout and is an independent formulation used to pin this one.
 *
 * Build with -ffp-contract=off so that x86-64 and aarch64 round every product
 * separately (no fused multiply-add), giving identical results on both hosts.
 *
 * Parity status per function (what pins it is in tests/test_oracle_*.py):
 *   orc_rope_freqs, orc_rms_norm, orc_rope, orc_kv_append, orc_gqa_attn,
 *   orc_attn_bruteforce_f64, orc_silu_mul, orc_layer_attn_step,
 *   orc_f32_to_f16, orc_f16_to_f32, orc_kv_append_f16,
 *   orc_layer_attn_step_f16, orc_kv_append_paged, orc_gqa_attn_paged,
 *   orc_q8_quantize_row, orc_q8_dequant_row, orc_kv_append_q8, orc_fused_qkv -- all pinned.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status codes (the oracle's own; numerically chosen to match the library's
 * public enum so tests can compare statuses, but not shared as a header). */
#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_GEOMETRY 2
#define ORC_ERR_POS 4

uint16_t orc_f32_to_f16(float f);
float orc_f16_to_f32(uint16_t h);

#define ORC_MAX_HALF 128 /* [P1] §3.2.2: the angular-speed table holds hd/2 <= 128 entries */

/* ------------------------------------------------------------------------ */
/* RoPE angular speeds.  [P1] §2.3 and §3.2.2: freq_i = freq_scale / base^(2i/hd).
 * The page evaluates this in f32 with powf, whose last bit differs between math
 * libraries; the reading taken here is the exact quotient evaluated in double and
 * rounded once to float, so any implementation can reproduce the table bit for bit. */
void orc_rope_freqs(float *freqs, int hd, float theta, float freq_scale)
{
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double expo = (double)(2 * i) / (double)hd;
        freqs[i] = (float)((double)freq_scale / pow((double)theta, expo));
    }
}

/* ------------------------------------------------------------------------ */
/* RMSNorm with gains.  [P1] §3.2.1: sum of squares in f64, mean rounded to f32,
 * scale = 1/sqrt(mean + eps) in f32, y = x * scale, then y *= weight.  No mean
 * subtraction.  y may alias x.  w == NULL means unit gains. */
void orc_rms_norm(float *y, const float *x, const float *w, int rows, int n, float eps)
{
    for (int r = 0; r < rows; ++r) {
        const float *xr = x + (size_t)r * n;
        float *yr = y + (size_t)r * n;
        double sum_sq = 0.0;
        for (int i = 0; i < n; ++i)
            sum_sq += (double)xr[i] * (double)xr[i];
        float mean = (float)(sum_sq / (double)n);
        float scale = 1.0f / sqrtf(mean + eps);
        for (int i = 0; i < n; ++i) {
            float v = xr[i] * scale;
            yr[i] = w ? v * w[i] : v;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Rotary position embedding, in place.  [P1] §3.2.2 (the cpu_rope core loop):
 * per token t, head h and subspace i < hd/2, angle th = pos[t] * freq_i (f32
 * product); the pair is (i, i+hd/2) for the NonInterleaved (Qwen/NEOX) style
 * and (2i, 2i+1) for the Interleaved (Llama) style; the pair is rotated by
 * +th: x0' = x0 cos - x1 sin, x1' = x0 sin + x1 cos.  sin and cos are taken
 * in double and rounded to float (the reading for large positions).
 * x is [nt, nh, hd] row-major.  style: 0 = NonInterleaved, 1 = Interleaved. */
int orc_rope(float *x, const int32_t *pos, int nt, int nh, int hd,
             float theta, float freq_scale, int style)
{
    if (hd <= 0 || (hd & 1) || hd / 2 > ORC_MAX_HALF || nh <= 0 || nt < 0)
        return ORC_ERR_ARG;
    if (style != 0 && style != 1)
        return ORC_ERR_ARG;
    int half = hd / 2;
    float freqs[ORC_MAX_HALF];
    orc_rope_freqs(freqs, hd, theta, freq_scale);
    for (int t = 0; t < nt; ++t) {
        if (pos[t] < 0)
            return ORC_ERR_POS;
        float p = (float)pos[t];
        for (int h = 0; h < nh; ++h) {
            size_t b = ((size_t)t * nh + h) * hd;
            for (int i = 0; i < half; ++i) {
                float th = p * freqs[i];
                float sn = (float)sin((double)th);
                float cs = (float)cos((double)th);
                size_t i0 = style == 0 ? b + i : b + 2 * (size_t)i;
                size_t i1 = style == 0 ? b + i + half : b + 2 * (size_t)i + 1;
                float x0 = x[i0], x1 = x[i1];
                x[i0] = x0 * cs - x1 * sn;
                x[i1] = x0 * sn + x1 * cs;
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* KV store.  [P1] §3.2.3 (the KvcacheStore arm): for each token in order,
 * p = pos[t]; p >= n_ctx is a hard error (return, never clamp); otherwise the
 * K row and the V row (W floats each) are copied to offset p*W of the layer's
 * persistent regions.  Like the page, the first bad position returns at once,
 * after the rows before it were written.  [P2] (the in-place append with
 * headroom) is the same copy with the region's row capacity as n_ctx. */
int orc_kv_append(float *k_reg, float *v_reg, int cap, int W,
                  const float *k_rows, const float *v_rows, const int32_t *pos, int nt)
{
    if (cap < 0 || W <= 0 || nt < 0)
        return ORC_ERR_ARG;
    for (int t = 0; t < nt; ++t) {
        int p = pos[t];
        if (p < 0 || p >= cap)
            return ORC_ERR_POS;
        memcpy(k_reg + (size_t)p * W, k_rows + (size_t)t * W, sizeof(float) * (size_t)W);
        memcpy(v_reg + (size_t)p * W, v_rows + (size_t)t * W, sizeof(float) * (size_t)W);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Grouped-query attention.  [P1] §3.2.4 (the Attn arm and the per-head worker)
 * and §3.2.5 (softmax):
 *   nkv = min(max_t pos[t] + 1, cap)                      (the window is data)
 *   query head h reads kv head hk = h / (nh / nk)
 *   vl  = min(pos[t] + 1, nkv)                            (causal by length)
 *   s_j = dot_f32(q[t,h][0:hdkv], K[j, hk]) * scale for j < vl, -inf after
 *   softmax over all nkv entries: exp(s - max) with an f64 sum, then scaled
 *   by (float)(1/sum); out = sum_j w_j V[j, hk] over all nkv rows, ascending.
 * q is [nt, nh, hd] (query head stride hd; the dot uses its first hdkv
 * entries), the regions are [cap, nk*hdkv], out is [nt, nh*hdkv].
 * Heads are split over n_threads workers; heads never reduce against each
 * other, so the result is bit-identical at any thread count ([P1] §3.2.4). */
typedef struct {
    float *out;
    const float *q, *k_reg, *v_reg;
    const int32_t *pos;
    int nt, nh, nk, hd, hdkv, nkv, h0, h1;
    float scale;
    int status;
} orc_attn_job;

static void *orc_attn_heads(void *arg)
{
    orc_attn_job *c = (orc_attn_job *)arg;
    int gqa = c->nh / c->nk;
    int W = c->nk * c->hdkv;
    float *scrs = (float *)malloc(sizeof(float) * (size_t)(c->nkv > 0 ? c->nkv : 1));
    if (!scrs) {
        c->status = ORC_ERR_ARG;
        return NULL;
    }
    for (int h = c->h0; h < c->h1; ++h) {
        int hk = h / gqa;
        for (int t = 0; t < c->nt; ++t) {
            const float *q_row = c->q + ((size_t)t * c->nh + h) * c->hd;
            float *out_row = c->out + ((size_t)t * c->nh + h) * c->hdkv;
            int vl = c->pos[t] + 1 < c->nkv ? c->pos[t] + 1 : c->nkv;
            float mx = -INFINITY;
            for (int kv = 0; kv < vl; ++kv) {
                const float *k_row = c->k_reg + (size_t)kv * W + (size_t)hk * c->hdkv;
                float dot = 0.0f;
                for (int d = 0; d < c->hdkv; ++d)
                    dot += q_row[d] * k_row[d];
                float s = dot * c->scale;
                scrs[kv] = s;
                if (s > mx)
                    mx = s;
            }
            for (int kv = vl; kv < c->nkv; ++kv)
                scrs[kv] = -INFINITY;
            double sum = 0.0;
            for (int kv = 0; kv < c->nkv; ++kv) {
                float e = expf(scrs[kv] - mx);
                scrs[kv] = e;
                sum += (double)e;
            }
            float inv = (float)(1.0 / sum);
            for (int kv = 0; kv < c->nkv; ++kv)
                scrs[kv] *= inv;
            for (int d = 0; d < c->hdkv; ++d)
                out_row[d] = 0.0f;
            for (int kv = 0; kv < c->nkv; ++kv) {
                const float *v_row = c->v_reg + (size_t)kv * W + (size_t)hk * c->hdkv;
                float wgt = scrs[kv];
                for (int d = 0; d < c->hdkv; ++d)
                    out_row[d] += wgt * v_row[d];
            }
        }
    }
    free(scrs);
    return NULL;
}

int orc_gqa_attn(float *out, const float *q, const float *k_reg, const float *v_reg, int cap,
                 const int32_t *pos, int nt, int nh, int nk, int hd, int hdkv, float scale,
                 int n_threads)
{
    if (nt < 0 || nh <= 0 || nk <= 0 || hd <= 0 || hdkv <= 0 || cap < 0)
        return ORC_ERR_ARG;
    if (hd < hdkv || nh % nk != 0) /* [P1] §1: hd < hd_kv is refused */
        return ORC_ERR_GEOMETRY;
    if (nt == 0)
        return ORC_OK;
    long mx_pos1 = 0;
    for (int t = 0; t < nt; ++t) {
        if (pos[t] < 0)
            return ORC_ERR_POS;
        if ((long)pos[t] + 1 > mx_pos1)
            mx_pos1 = (long)pos[t] + 1;
    }
    int nkv = (int)(mx_pos1 < cap ? mx_pos1 : cap);
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > nh)
        n_threads = nh;
    orc_attn_job jobs[256];
    pthread_t tids[256];
    if (n_threads > 256)
        n_threads = 256;
    for (int w = 0; w < n_threads; ++w) {
        orc_attn_job *j = &jobs[w];
        j->out = out; j->q = q; j->k_reg = k_reg; j->v_reg = v_reg; j->pos = pos;
        j->nt = nt; j->nh = nh; j->nk = nk; j->hd = hd; j->hdkv = hdkv; j->nkv = nkv;
        j->h0 = (int)((long)nh * w / n_threads);
        j->h1 = (int)((long)nh * (w + 1) / n_threads);
        j->scale = scale;
        j->status = ORC_OK;
    }
    if (n_threads == 1) {
        orc_attn_heads(&jobs[0]);
    } else {
        for (int w = 0; w < n_threads; ++w)
            pthread_create(&tids[w], NULL, orc_attn_heads, &jobs[w]);
        for (int w = 0; w < n_threads; ++w)
            pthread_join(tids[w], NULL);
    }
    for (int w = 0; w < n_threads; ++w)
        if (jobs[w].status != ORC_OK)
            return jobs[w].status;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* The Q8_0 cache.  [P1] §2.5: the store quantizes each K/V row into Q8_0 block
 * rows -- blocks of 32 consecutive values, each one f16 scale and 32 int8
 * quants (34 bytes per 32 values, 3.76x smaller than f32) -- and the attention
 * read dequantizes the window it uses.  The pages give the block format but not
 * the quantizer; the reading taken is the symmetric absolute-maximum one the
 * format is built for: d = max|x| / 127, q = round(x / d) (nearest, halves away
 * from zero, so |q| <= 127), computed as x * (1/d) in fp32 with d = 0 giving
 * q = 0; the block keeps f16(d) and reads back x' = f16(d) * q.
 * Row layout (bytes): the W quants of the row in order, then its W/32 scales
 * (binary16, block order), then zero padding to a multiple of 16 bytes. */
long orc_q8_row_bytes(int W)
{
    long scales = (long)(W / 32) * 2;
    return (long)W + ((scales + 15) / 16) * 16;
}

void orc_q8_quantize_row(uint8_t *dst, const float *x, int W)
{
    int nb = W / 32;
    long rb = orc_q8_row_bytes(W);
    memset(dst, 0, (size_t)rb);
    for (int b = 0; b < nb; ++b) {
        float amax = 0.0f;
        for (int j = 0; j < 32; ++j) {
            float a = fabsf(x[32 * b + j]);
            if (a > amax)
                amax = a;
        }
        float d = amax / 127.0f;
        float id = d != 0.0f ? 1.0f / d : 0.0f;
        for (int j = 0; j < 32; ++j) {
            float qf = roundf(x[32 * b + j] * id);
            int8_t qi = (int8_t)qf;
            memcpy(dst + 32 * b + j, &qi, 1);
        }
        uint16_t h = orc_f32_to_f16(d);
        memcpy(dst + W + 2 * b, &h, 2);
    }
}

void orc_q8_dequant_row(float *x, const uint8_t *src, int W)
{
    int nb = W / 32;
    for (int b = 0; b < nb; ++b) {
        uint16_t h;
        memcpy(&h, src + W + 2 * b, 2);
        float d = orc_f16_to_f32(h);
        for (int j = 0; j < 32; ++j) {
            int8_t qi;
            memcpy(&qi, src + 32 * b + j, 1);
            x[32 * b + j] = d * (float)qi;
        }
    }
}

void orc_q8_quantize_rows(uint8_t *dst, const float *x, long rows, int W)
{
    long rb = orc_q8_row_bytes(W);
    for (long r = 0; r < rows; ++r)
        orc_q8_quantize_row(dst + r * rb, x + r * W, W);
}

void orc_q8_dequant_rows(float *x, const uint8_t *src, long rows, int W)
{
    long rb = orc_q8_row_bytes(W);
    for (long r = 0; r < rows; ++r)
        orc_q8_dequant_row(x + r * W, src + r * rb, W);
}

/* The KV store into Q8_0 regions ([cap, row_bytes] bytes): the same placement
 * as orc_kv_append, each row quantized on the way in. */
int orc_kv_append_q8(uint8_t *k_reg, uint8_t *v_reg, int cap, int W, const float *k_rows, const float *v_rows,
                     const int32_t *pos, int nt)
{
    if (cap < 0 || W <= 0 || W % 32 || nt < 0)
        return ORC_ERR_ARG;
    long rb = orc_q8_row_bytes(W);
    for (int t = 0; t < nt; ++t) {
        int p = pos[t];
        if (p < 0 || p >= cap)
            return ORC_ERR_POS;
        orc_q8_quantize_row(k_reg + (size_t)p * rb, k_rows + (size_t)t * W, W);
        orc_q8_quantize_row(v_reg + (size_t)p * rb, v_rows + (size_t)t * W, W);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Paged regions.  [P2] "IV.2: Zero-copy KV cache" (the paged cache stores a
 * sequence as scattered fixed-size blocks, so it cannot lend one contiguous
 * view) and [P3] §2.2 (the attention reads the cells an explicit window
 * names).  A pool holds pool_blocks blocks of block_rows rows of width W;
 * sequence s owns the blocks its table row names: logical row j of s is pool
 * row table[s*max_blocks + j/block_rows]*block_rows + j%block_rows, so its
 * capacity is max_blocks*block_rows rows.  A block id outside the pool (or
 * negative: not allocated) is an error wherever a row of it is needed. */
static int orc_paged_row(const int32_t *table, int max_blocks, int block_rows, int pool_blocks, int s,
                         long j, long *row)
{
    long blk = j / block_rows;
    if (j < 0 || blk >= max_blocks)
        return ORC_ERR_POS;
    int b = table[(size_t)s * max_blocks + blk];
    if (b < 0 || b >= pool_blocks)
        return ORC_ERR_POS;
    *row = (long)b * block_rows + j % block_rows;
    return ORC_OK;
}

/* The KV store through the table: one token per sequence, at pos[s]. */
int orc_kv_append_paged(float *k_pool, float *v_pool, int pool_blocks, int block_rows, int W,
                        const int32_t *table, int max_blocks, const float *k_rows, const float *v_rows,
                        const int32_t *pos, int n_seq)
{
    if (pool_blocks < 0 || block_rows <= 0 || W <= 0 || max_blocks <= 0 || n_seq < 0)
        return ORC_ERR_ARG;
    for (int s = 0; s < n_seq; ++s) {
        long row;
        int st = orc_paged_row(table, max_blocks, block_rows, pool_blocks, s, pos[s], &row);
        if (st != ORC_OK)
            return st;
        memcpy(k_pool + (size_t)row * W, k_rows + (size_t)s * W, sizeof(float) * (size_t)W);
        memcpy(v_pool + (size_t)row * W, v_rows + (size_t)s * W, sizeof(float) * (size_t)W);
    }
    return ORC_OK;
}

/* Decode attention through the table: for each sequence, the rows of its window
 * [0, min(pos+1, max_blocks*block_rows)) are gathered in logical order and the
 * attention above runs over them.  q is [n_seq, nh, hd], out [n_seq, nh*hdkv]. */
int orc_gqa_attn_paged(float *out, const float *q, const float *k_pool, const float *v_pool, int pool_blocks,
                       int block_rows, const int32_t *table, int max_blocks, const int32_t *pos, int n_seq,
                       int nh, int nk, int hd, int hdkv, float scale)
{
    if (pool_blocks < 0 || block_rows <= 0 || max_blocks <= 0 || n_seq < 0 || nk <= 0 || hdkv <= 0)
        return ORC_ERR_ARG;
    int W = nk * hdkv;
    long cap = (long)max_blocks * block_rows;
    for (int s = 0; s < n_seq; ++s) {
        if (pos[s] < 0)
            return ORC_ERR_POS;
        long L = (long)pos[s] + 1 < cap ? (long)pos[s] + 1 : cap;
        float *kb = malloc(sizeof(float) * (size_t)L * W);
        float *vb = malloc(sizeof(float) * (size_t)L * W);
        if (!kb || !vb) {
            free(kb);
            free(vb);
            return ORC_ERR_ARG;
        }
        int st = ORC_OK;
        for (long j = 0; j < L && st == ORC_OK; ++j) {
            long row;
            st = orc_paged_row(table, max_blocks, block_rows, pool_blocks, s, j, &row);
            if (st == ORC_OK) {
                memcpy(kb + (size_t)j * W, k_pool + (size_t)row * W, sizeof(float) * (size_t)W);
                memcpy(vb + (size_t)j * W, v_pool + (size_t)row * W, sizeof(float) * (size_t)W);
            }
        }
        if (st == ORC_OK)
            st = orc_gqa_attn(out + (size_t)s * nh * hdkv, q + (size_t)s * nh * hd, kb, vb, (int)L, pos + s, 1,
                              nh, nk, hd, hdkv, scale, 1);
        free(kb);
        free(vb);
        if (st != ORC_OK)
            return st;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Brute-force masked attention in fp64: an independent formulation of [P1] §2.1
 * steps 1-4 used only to pin orc_gqa_attn on small inputs.  It builds the
 * explicit [nt x nkv] additive mask matrix (0 where key j <= pos[t], -inf
 * elsewhere) that the pages deliberately avoid, maps query head h to kv head
 * floor(h * nk / nh), takes a full softmax in double and a double weighted
 * sum.  out is [nt, nh*hdkv] in double. */
int orc_attn_bruteforce_f64(double *out, const float *q, const float *k_reg, const float *v_reg,
                            int cap, const int32_t *pos, int nt, int nh, int nk, int hd, int hdkv,
                            double scale)
{
    if (nt <= 0 || nh <= 0 || nk <= 0 || hd < hdkv || nh % nk != 0)
        return ORC_ERR_GEOMETRY;
    int W = nk * hdkv;
    long nkv = 0;
    for (int t = 0; t < nt; ++t)
        if ((long)pos[t] + 1 > nkv)
            nkv = (long)pos[t] + 1;
    if (nkv > cap)
        nkv = cap;
    double *mask = (double *)malloc(sizeof(double) * (size_t)nt * (size_t)nkv);
    double *logit = (double *)malloc(sizeof(double) * (size_t)nkv);
    if (!mask || !logit) {
        free(mask);
        free(logit);
        return ORC_ERR_ARG;
    }
    for (int t = 0; t < nt; ++t)
        for (long j = 0; j < nkv; ++j)
            mask[(size_t)t * nkv + j] = (j <= pos[t]) ? 0.0 : -INFINITY;
    for (int t = 0; t < nt; ++t) {
        for (int h = 0; h < nh; ++h) {
            int hk = (int)(((long)h * nk) / nh);
            const float *qr = q + ((size_t)t * nh + h) * hd;
            double best = -INFINITY;
            for (long j = 0; j < nkv; ++j) {
                const float *kr = k_reg + (size_t)j * W + (size_t)hk * hdkv;
                double acc = 0.0;
                for (int d = 0; d < hdkv; ++d)
                    acc += (double)qr[d] * (double)kr[d];
                logit[j] = acc * scale + mask[(size_t)t * nkv + j];
                if (logit[j] > best)
                    best = logit[j];
            }
            double z = 0.0;
            for (long j = 0; j < nkv; ++j) {
                logit[j] = exp(logit[j] - best);
                z += logit[j];
            }
            double *o = out + ((size_t)t * nh + h) * hdkv;
            for (int d = 0; d < hdkv; ++d) {
                double acc = 0.0;
                for (long j = 0; j < nkv; ++j)
                    acc += logit[j] * (double)v_reg[(size_t)j * W + (size_t)hk * hdkv + d];
                o[d] = acc / z;
            }
        }
    }
    free(mask);
    free(logit);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* The f16 cache.  [P1] §2.5 ("What changes on the GPU"): the GPU backends may
 * keep the K/V regions in f16, halving the bytes each attention read moves;
 * the store converts and the attention read converts back.  The pages do not
 * name a rounding, so the store takes IEEE 754 binary16 with round to nearest,
 * ties to even (the format's default), written out here from the format's
 * definition: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;
 * subnormals are m * 2^-24; magnitudes that round past 65504 become infinity;
 * NaN stays NaN.  Reading back is exact (every binary16 value is an fp32). */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint32_t sign = (x >> 16) & 0x8000u;
    int exp = (int)((x >> 23) & 0xffu);
    uint32_t frac = x & 0x7fffffu;
    if (exp == 0xff) /* infinity, or NaN (kept quiet, payload truncated) */
        return (uint16_t)(sign | 0x7c00u | (frac ? 0x200u | (frac >> 13) : 0u));
    int e = exp - 127 + 15; /* the binary16 biased exponent of a normal result */
    if (e >= 1) {
        uint32_t m = frac >> 13, rest = frac & 0x1fffu;
        if (rest > 0x1000u || (rest == 0x1000u && (m & 1u)))
            ++m;
        if (m == 0x400u) { /* the fraction overflowed into the exponent */
            m = 0;
            ++e;
        }
        if (e >= 31)
            return (uint16_t)(sign | 0x7c00u);
        return (uint16_t)(sign | ((uint32_t)e << 10) | m);
    }
    /* subnormal (or zero) result: value / 2^-24, rounded to an integer */
    if (exp == 0)
        return (uint16_t)sign; /* fp32 subnormals are far below 2^-25 */
    uint32_t full = frac | 0x800000u; /* 24 significant bits, value = full * 2^(exp-150) */
    int shift = 126 - exp;            /* value / 2^-24 = full >> shift */
    if (shift > 24)
        return (uint16_t)sign;
    uint32_t m = full >> shift, rest = full & ((1u << shift) - 1u), half = 1u << (shift - 1);
    if (rest > half || (rest == half && (m & 1u)))
        ++m; /* m == 0x400 is the smallest normal, which the bits already spell */
    return (uint16_t)(sign | m);
}

float orc_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    int e = (h >> 10) & 0x1f;
    uint32_t m = h & 0x3ffu;
    float v;
    if (e == 0) {
        v = ldexpf((float)m, -24);
        if (sign)
            v = -v;
        return v;
    }
    uint32_t x;
    if (e == 31)
        x = sign | 0x7f800000u | (m << 13);
    else
        x = sign | ((uint32_t)(e - 15 + 127) << 23) | (m << 13);
    memcpy(&v, &x, sizeof v);
    return v;
}

void orc_f32_to_f16_array(uint16_t *dst, const float *src, long n)
{
    for (long i = 0; i < n; ++i)
        dst[i] = orc_f32_to_f16(src[i]);
}

void orc_f16_to_f32_array(float *dst, const uint16_t *src, long n)
{
    for (long i = 0; i < n; ++i)
        dst[i] = orc_f16_to_f32(src[i]);
}

/* The KV store into f16 regions: the same placement as orc_kv_append, each
 * element converted on the way in ([P1] §2.5: the store converts). */
int orc_kv_append_f16(uint16_t *k_reg, uint16_t *v_reg, int cap, int W,
                      const float *k_rows, const float *v_rows, const int32_t *pos, int nt)
{
    if (cap < 0 || W <= 0 || nt < 0)
        return ORC_ERR_ARG;
    for (int t = 0; t < nt; ++t) {
        int p = pos[t];
        if (p < 0 || p >= cap)
            return ORC_ERR_POS;
        orc_f32_to_f16_array(k_reg + (size_t)p * W, k_rows + (size_t)t * W, W);
        orc_f32_to_f16_array(v_reg + (size_t)p * W, v_rows + (size_t)t * W, W);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* The fused QKV decode op.  [P3] §2.3: for a single token, a GPU build merges the
 * three projection matmuls, their three biases, the two RoPEs and the two KV
 * stores into one op.  Here, per token t: xn = RMSNorm(h) * gain ([P1] §3.2.1);
 * y = W xn + b with W [n_out, n_embd] whose rows are the nh*hd q outputs, then
 * the nk*hdkv k outputs, then the nk*hdkv v outputs, and b [n_out] (NULL: no
 * bias), every output a dot product accumulated in double and rounded once to
 * fp32 before the bias is added in fp32; then q and k rotated at pos ([P1]
 * §3.2.2) and the rotated k and v stored at pos ([P1] §3.2.3). */
int orc_fused_qkv(float *xn, float *q, float *k, float *v, const float *h, const float *gain, float eps,
                  int n_embd, const float *w, const float *b, const int32_t *pos, int nt, float *k_reg,
                  float *v_reg, int cap, int nh, int nk, int hd, int hdkv, float theta, float freq_scale, int style)
{
    if (hd < hdkv || nh <= 0 || nk <= 0 || nh % nk != 0)
        return ORC_ERR_GEOMETRY;
    if (n_embd <= 0 || nt < 0)
        return ORC_ERR_ARG;
    orc_rms_norm(xn, h, gain, nt, n_embd, eps);
    int nq = nh * hd, W = nk * hdkv, n_out = nq + 2 * W;
    for (int t = 0; t < nt; ++t) {
        const float *x = xn + (size_t)t * n_embd;
        for (int j = 0; j < n_out; ++j) {
            const float *wr = w + (size_t)j * n_embd;
            double acc = 0.0;
            for (int i = 0; i < n_embd; ++i)
                acc += (double)wr[i] * (double)x[i];
            float y = (float)acc;
            if (b)
                y = y + b[j];
            if (j < nq)
                q[(size_t)t * nq + j] = y;
            else if (j < nq + W)
                k[(size_t)t * W + (j - nq)] = y;
            else
                v[(size_t)t * W + (j - nq - W)] = y;
        }
    }
    int st = orc_rope(q, pos, nt, nh, hd, theta, freq_scale, style);
    if (st != ORC_OK)
        return st;
    st = orc_rope(k, pos, nt, nk, hdkv, theta, freq_scale, style);
    if (st != ORC_OK)
        return st;
    return orc_kv_append(k_reg, v_reg, cap, W, k, v, pos, nt);
}

/* ------------------------------------------------------------------------ */
/* SiLU times up.  [P1] §3.2.5: silu(x) = x / (1 + e^-x); SwiGLU multiplies it
 * by the up projection element-wise. */
void orc_silu_mul(float *y, const float *gate, const float *up, long n)
{
    for (long i = 0; i < n; ++i) {
        float g = gate[i];
        float s = g / (1.0f + expf(-g));
        y[i] = s * up[i];
    }
}

/* ------------------------------------------------------------------------ */
/* One layer's attention stage.  [P1] §1 (the decoder layer picture) and §3.4
 * (store before attention): xn = RMSNorm(h) * gain; RoPE on q (nh heads of hd)
 * and on k (nk heads of hdkv), in place; KV store of the rotated k and of v at
 * pos[t]; attention over the regions with scale = 1/sqrt(hd) ([P1] §2.4).
 * The q/k/v projections need trained weights and are outside this stage, so
 * xn is a separate output and q, k, v are inputs. */
int orc_layer_attn_step(float *xn, const float *h, const float *gain, float eps, int n_embd,
                        float *q, float *k, const float *v, const int32_t *pos, int nt,
                        float *k_reg, float *v_reg, int cap, int nh, int nk, int hd, int hdkv,
                        float theta, float freq_scale, int style, float *out, int n_threads)
{
    if (hd < hdkv || nh <= 0 || nk <= 0 || nh % nk != 0)
        return ORC_ERR_GEOMETRY;
    orc_rms_norm(xn, h, gain, nt, n_embd, eps);
    int st = orc_rope(q, pos, nt, nh, hd, theta, freq_scale, style);
    if (st != ORC_OK)
        return st;
    st = orc_rope(k, pos, nt, nk, hdkv, theta, freq_scale, style);
    if (st != ORC_OK)
        return st;
    st = orc_kv_append(k_reg, v_reg, cap, nk * hdkv, k, v, pos, nt);
    if (st != ORC_OK)
        return st;
    float scale = 1.0f / sqrtf((float)hd);
    return orc_gqa_attn(out, q, k_reg, v_reg, cap, pos, nt, nh, nk, hd, hdkv, scale, n_threads);
}

/* The same stage over f16 regions ([P1] §2.5): the store converts the rotated
 * k and v to f16; the attention read converts the regions back (exactly) and
 * runs the fp32 attention above on those values. */
int orc_layer_attn_step_f16(float *xn, const float *h, const float *gain, float eps, int n_embd,
                            float *q, float *k, const float *v, const int32_t *pos, int nt,
                            uint16_t *k_reg, uint16_t *v_reg, int cap, int nh, int nk, int hd,
                            int hdkv, float theta, float freq_scale, int style, float *out,
                            int n_threads)
{
    if (hd < hdkv || nh <= 0 || nk <= 0 || nh % nk != 0)
        return ORC_ERR_GEOMETRY;
    orc_rms_norm(xn, h, gain, nt, n_embd, eps);
    int st = orc_rope(q, pos, nt, nh, hd, theta, freq_scale, style);
    if (st != ORC_OK)
        return st;
    st = orc_rope(k, pos, nt, nk, hdkv, theta, freq_scale, style);
    if (st != ORC_OK)
        return st;
    int W = nk * hdkv;
    st = orc_kv_append_f16(k_reg, v_reg, cap, W, k, v, pos, nt);
    if (st != ORC_OK)
        return st;
    float *kf = malloc(sizeof(float) * (size_t)cap * W);
    float *vf = malloc(sizeof(float) * (size_t)cap * W);
    if (!kf || !vf) {
        free(kf);
        free(vf);
        return ORC_ERR_ARG;
    }
    orc_f16_to_f32_array(kf, k_reg, (long)cap * W);
    orc_f16_to_f32_array(vf, v_reg, (long)cap * W);
    float scale = 1.0f / sqrtf((float)hd);
    st = orc_gqa_attn(out, q, kf, vf, cap, pos, nt, nh, nk, hd, hdkv, scale, n_threads);
    free(kf);
    free(vf);
    return st;
}
