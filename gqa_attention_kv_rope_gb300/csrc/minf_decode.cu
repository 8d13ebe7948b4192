// minf_decode.cu -- plans and launches the decode kernel of minf_decode.cuh: split counts,
// the workspace layout, tensor maps, and the fp32 instantiation of the kernel.
#include "minf_decode.cuh"

namespace minf {

namespace {

using namespace dec;

// Rows per pipeline stage for a region storage kind (as the kernel's Cfg has them).
inline int stage_rows(int hd_kv, int kind) {
    if (kind == kKvQ8) return hd_kv == 64 ? Cfg<64, Q8>::R : Cfg<128, Q8>::R;
    const int eb = kind == kKvF16 ? 2 : 4;
    return kStageBytes / (2 * hd_kv * eb);
}

struct WsLayout {
    size_t ml_off, acc_off, tk_off, total;
    int key;  // the layout tag a call of this layout leaves in the control block
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The control block (counters and layout tag, shared with the prefill layout), then the split
// partials: (m, l) pairs and accumulators, zero (not yet written) between calls, then one merge
// ticket per (sequence, q head) for the units of many heads, which merge by ticket.
WsLayout ws_layout(int n_seq, int nh, int hd_kv, int splits) {
    WsLayout w;
    const size_t parts = static_cast<size_t>(n_seq) * nh * splits;
    w.ml_off = kWsCtlBytes;
    w.acc_off = w.ml_off + align256(parts * 2 * sizeof(float));
    w.tk_off = w.acc_off + align256(parts * hd_kv * sizeof(float));
    w.total = w.tk_off + align256(static_cast<size_t>(n_seq) * nh * sizeof(int));
    w.key = ws_key(kWsKindDecode, w.acc_off, w.total, parts, static_cast<unsigned long long>(splits));
    return w;
}

// Query heads of a group handled by one unit: keep the q slice (GH*hd_kv/8 floats per lane)
// within 64 registers where the group allows it.
int heads_per_cta(int g, int hd_kv) {
    if (g * hd_kv / 8 <= 64) return g;
    if (g % 2 == 0 && (g / 2) * hd_kv / 8 <= 64) return g / 2;
    if (g % 4 == 0) return g / 4;
    return g;
}

// Splits per (sequence, kv group): fill the SMs once when the pairs alone cannot; otherwise
// (a batch) cut only long windows, into units of at most kMaxRows, since the persistent CTAs
// take units from a shared counter, longest first.
int choose_splits(long long pairs, int hd_kv, int max_cap, int kind) {
    const long long R = stage_rows(hd_kv, kind);
    long long s = pairs < kGridTarget ? kGridTarget / pairs
                                      : (static_cast<long long>(max_cap) + kMaxRows - 1) / kMaxRows;
    const long long s_rows = (static_cast<long long>(max_cap) + R - 1) / R;
    if (s > s_rows) s = s_rows;
    if (s > kMaxSplit) s = kMaxSplit;
    if (s < 1) s = 1;
    return static_cast<int>(s);
}

struct Plan {
    int gh, groups, S, min_rows, sorted;
    WsLayout w;
};

// kind: the region storage (binary16 and Q8_0 stages hold more rows than fp32 ones).  The
// workspace is laid out for fp32's split count, which is never below the others', so one
// workspace size serves every storage kind.
Plan plan_for(int n_seq, int nh, int nk, int hd_kv, int max_cap, int kind) {
    Plan p;
    const int g = nh / nk;
    p.gh = heads_per_cta(g, hd_kv);
    p.groups = g / p.gh;
    const long long pairs = static_cast<long long>(n_seq) * nk * p.groups;
    p.S = choose_splits(pairs, hd_kv, max_cap, kind);
    const bool batch = pairs >= kGridTarget;
    p.min_rows = batch ? kBatchMinRows : stage_rows(hd_kv, kind);
    p.sorted = batch && n_seq > 1 && n_seq <= kMaxSort;
    p.w = ws_layout(n_seq, nh, hd_kv, choose_splits(pairs, hd_kv, max_cap, kKvF32));
    return p;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

int launch_impl(const DecodeArgs &d, const DecodeStepExtra *x, cudaStream_t s) {
    if (d.n_seq == 0) return MINF_OK;
    const bool f16 = d.kv == kKvF16, q8 = d.kv == kKvQ8;
    const int eb = f16 ? 2 : (q8 ? 1 : 4);
    const Plan pl = plan_for(d.n_seq, d.nh, d.nk, d.hd_kv, d.cap, d.kv);
    if (!d.ws || d.ws_bytes < pl.w.total || !aligned16(d.ws)) return MINF_ERR_WORKSPACE;
    const long long units = static_cast<long long>(d.n_seq) * d.nk * pl.groups * pl.S;
    if (units > 0x7fffffffLL) return MINF_ERR_UNSUPPORTED;
    const long long rows = (d.row_off || d.table) ? d.arena_rows : d.cap;
    if (rows <= 0) return MINF_ERR_ARG;
    if (rows > 0x7fffffffLL - 4096) return MINF_ERR_UNSUPPORTED;
    const int R = stage_rows(d.hd_kv, d.kv);
    // paged: a stage is copied in pieces of one block (or one stage when blocks are larger)
    const int box = d.table ? (d.block_rows < R ? d.block_rows : R) : R;
    CUtensorMap tk, tv, tks, tvs;
    const uint64_t W = static_cast<uint64_t>(d.nk) * d.hd_kv;
    // Q8_0 rows are bytes: the quants of this kv head, and a 16-byte slice of the scales
    const uint64_t cols = q8 ? static_cast<uint64_t>(q8_row_bytes(static_cast<int>(W))) : W;
    const CUtensorMapDataType dt = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                       : (q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
    if (!make_tensor_map_2d(&tk, d.k_reg, dt, eb, cols, static_cast<uint64_t>(rows), d.hd_kv, box, false) ||
        !make_tensor_map_2d(&tv, d.v_reg, dt, eb, cols, static_cast<uint64_t>(rows), d.hd_kv, box, false))
        return MINF_ERR_CUDA;
    tks = tk;
    tvs = tv;
    if (q8 && (!make_tensor_map_2d(&tks, d.k_reg, dt, 1, cols, static_cast<uint64_t>(rows), 16, box, false) ||
               !make_tensor_map_2d(&tvs, d.v_reg, dt, 1, cols, static_cast<uint64_t>(rows), 16, box, false)))
        return MINF_ERR_CUDA;
    char *ws = static_cast<char *>(d.ws);
    KParams k = {};
    k.out = d.out;
    k.q = d.q;
    k.row_off = d.row_off;
    k.caps = d.caps;
    k.pos = d.pos;
    k.cap = d.cap;
    k.n_seq = d.n_seq;
    k.nh = d.nh;
    k.nk = d.nk;
    k.hd = d.hd;
    k.n_split = pl.S;
    k.groups = pl.groups;
    k.scale_log2 = d.scale * kLog2e;
    k.err = d.err;
    k.ws_ml = reinterpret_cast<float *>(ws + pl.w.ml_off);
    k.ws_acc = reinterpret_cast<float *>(ws + pl.w.acc_off);
    k.ws_ticket = reinterpret_cast<int *>(ws + pl.w.tk_off);
    k.ws_ctr = reinterpret_cast<int *>(ws) + kWsUnitCtr;
    k.ws_done = reinterpret_cast<int *>(ws) + kWsUnitDone;
    k.ws_tag = reinterpret_cast<int *>(ws) + kWsTag;
    k.ws_key = pl.w.key;
    k.early = 1;  // without programmatic dependent launch the waits are no-ops
    k.min_rows = pl.min_rows;
    k.sorted = pl.sorted;
    k.table = d.table;
    k.max_blocks = d.max_blocks;
    k.block_rows = d.block_rows;
    k.box_rows = box;
    k.pool_rows = rows;
    k.row_bytes = q8 ? static_cast<long long>(cols) : 0;
    k.k_reg = const_cast<void *>(d.k_reg);
    k.v_reg = const_cast<void *>(d.v_reg);
    bool pdl = false;
    if (x) {
        k.q_io = const_cast<float *>(d.q);
        k.k_io = x->k;
        k.v_new = x->v;
        k.xn = x->xn;
        k.h = x->h;
        k.gain = x->gain;
        k.eps = x->eps;
        k.n_embd = x->n_embd;
        k.style = x->style;
        rope_table(&k.tab, d.hd_kv, x->theta, x->freq_scale);
        pdl = x->pdl;
        k.early = x->early;
    }
    const int sms = sm_count();
    const int grid = static_cast<int>(units < sms ? units : sms);
    const cudaError_t e = f16  ? dispatch_decode_f16(d.hd_kv, x != nullptr, pl.gh, tk, tv, tks, tvs, k, grid, s, pdl)
                          : q8 ? dispatch_decode_q8(d.hd_kv, x != nullptr, pl.gh, tk, tv, tks, tvs, k, grid, s, pdl)
                               : dispatch<float>(d.hd_kv, x != nullptr, pl.gh, tk, tv, tks, tvs, k, grid, s, pdl);
    if (e == cudaErrorInvalidValue) return MINF_ERR_UNSUPPORTED;
    return e == cudaSuccess ? MINF_OK : MINF_ERR_CUDA;
}

}  // namespace

bool make_tensor_map_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint32_t elem_bytes, uint64_t cols,
                        uint64_t rows, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * elem_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool decode_supported(int nh, int nk, int hd, int hd_kv) {
    if (hd_kv != 64 && hd_kv != 128) return false;
    if (hd % 4 != 0 || hd > 256) return false;
    const int g = nh / nk;
    return g >= 1 && g <= 8;
}

bool fused_step_supported(int nh, int nk, int hd, int hd_kv, int n_embd) {
    if (!decode_supported(nh, nk, hd, hd_kv) || hd != hd_kv || n_embd % 4 != 0) return false;
    const int g = nh / nk;
    return heads_per_cta(g, hd_kv) == g;  // one unit per kv head owns its k row and q heads
}

size_t decode_workspace_bytes(int n_seq, int nh, int nk, int hd_kv, int max_cap) {
    if (n_seq <= 0 || nh <= 0 || nk <= 0 || hd_kv <= 0 || max_cap <= 0 || nh % nk) return 0;
    return plan_for(n_seq, nh, nk, hd_kv, max_cap, kKvF32).w.total;  // the layout serves every storage kind
}

int launch_decode(const DecodeArgs &d, cudaStream_t s) { return launch_impl(d, nullptr, s); }

int launch_decode_step(const DecodeArgs &d, const DecodeStepExtra &x, cudaStream_t s) {
    return launch_impl(d, &x, s);
}

}  // namespace minf
