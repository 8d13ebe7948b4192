// minf_noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory for a workspace: code that runs inside
// an allocator-less embedding (a plugin handed only its input and output buffers), callers
// that must not touch the device allocator on their hot path because it would synchronise
// or fragment a pool they do not own, or environments where cudaMalloc is forbidden after
// start-up.  This file gives them one entry point that needs no workspace argument: the split
// partials and merge tickets of the decode kernel live in a fixed array of device memory that
// belongs to the library itself.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds it
// until the process exits.  Host code cannot use the variable's name as a device address (on
// the host it only names a stand-in); the address is looked up with cudaGetSymbolAddress, with
// the device current, and then passed to the kernel like any caller-provided workspace.  The
// address belongs to the CUDA context that was current when it was looked up, so it is kept
// per context (a caller that switches contexts on one device gets each context's own copy).
#include <cudaTypedefs.h>

#include <mutex>

#include "minf_common.cuh"
#include "minf_kernels.h"

namespace minf {
namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB per device
constexpr int kMaxContexts = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
struct ScratchEntry {
    CUcontext ctx;
    void *ptr;
};
ScratchEntry g_scratch[kMaxContexts] = {};
int g_n_scratch = 0;

// The driver's cuCtxGetCurrent, through the runtime's entry-point query (no link to libcuda).
PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;  // guarded by g_scratch_mu
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }
    return fn;
}

// The device address of the scratch array in the current context (looked up on first use).
int scratch_for_current_context(void **out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    auto get = ctx_get_current();
    if (!get) return MINF_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return MINF_ERR_CUDA;
    void *p = nullptr;
    if (!ctx) {
        // no context is current yet: the runtime call below makes the device's primary context
        // current (as any runtime call does), and the address is that context's
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return MINF_ERR_CUDA;
        if (get(&ctx) != CUDA_SUCCESS || !ctx) return MINF_ERR_CUDA;
    }
    for (int i = 0; i < g_n_scratch; ++i)
        if (g_scratch[i].ctx == ctx) {
            *out = g_scratch[i].ptr;
            return MINF_OK;
        }
    if (g_n_scratch == kMaxContexts) return MINF_ERR_CUDA;
    if (!p && (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p)) return MINF_ERR_CUDA;
    g_scratch[g_n_scratch++] = {ctx, p};
    *out = p;
    return MINF_OK;
}

}  // namespace
}  // namespace minf

using namespace minf;

extern "C" int minf_gqa_attn_decode_static_ws(float *out, const float *q, const float *k_reg,
                                              const float *v_reg, const int64_t *seq_row_off,
                                              const int32_t *seq_cap, int max_cap,
                                              int64_t arena_rows, const int32_t *pos, int n_seq,
                                              int n_head, int n_kv_head, int hd, int hd_kv,
                                              float scale, int32_t *err, minf_stream_t stream) {
    if (n_head <= 0 || n_kv_head <= 0 || hd <= 0 || hd_kv <= 0) return MINF_ERR_ARG;
    if (hd < hd_kv || n_head % n_kv_head != 0) return MINF_ERR_GEOMETRY;
    if (!decode_supported(n_head, n_kv_head, hd, hd_kv)) return MINF_ERR_UNSUPPORTED;
    if (!out || !q || !k_reg || !v_reg || !pos || !err || !aligned16(out) || !aligned16(q) ||
        !aligned16(k_reg) || !aligned16(v_reg))
        return MINF_ERR_ARG;
    if (n_seq < 0 || max_cap <= 0 || (seq_row_off && arena_rows <= 0)) return MINF_ERR_ARG;
    if (n_seq == 0) return MINF_OK;
    const size_t need = decode_workspace_bytes(n_seq, n_head, n_kv_head, hd_kv, max_cap);
    if (need == 0 || need > kStaticScratchBytes) return MINF_ERR_WORKSPACE;  // beyond the fixed 8 MiB
    void *ws = nullptr;
    const int st = scratch_for_current_context(&ws);
    if (st != MINF_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The merge tickets must start at zero; a previous call (or one that stopped early) may
    // have left anything behind, so the part this call uses is cleared first.
    if (cudaMemsetAsync(ws, 0, need, s) != cudaSuccess) return MINF_ERR_CUDA;
    DecodeArgs d = {};
    d.out = out;
    d.q = q;
    d.k_reg = k_reg;
    d.v_reg = v_reg;
    d.kv = kKvF32;
    d.row_off = seq_row_off;
    d.caps = seq_cap;
    d.cap = max_cap;
    d.arena_rows = arena_rows;
    d.pos = pos;
    d.n_seq = n_seq;
    d.nh = n_head;
    d.nk = n_kv_head;
    d.hd = hd;
    d.hd_kv = hd_kv;
    d.scale = scale;
    d.err = err;
    d.ws = ws;
    d.ws_bytes = kStaticScratchBytes;
    return launch_decode(d, s);
}
