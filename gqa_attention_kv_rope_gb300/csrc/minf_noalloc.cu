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
// the host it only names a stand-in); the address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and then passed to the kernel like any
// caller-provided workspace.
#include <mutex>

#include "minf_common.cuh"
#include "minf_kernels.h"

namespace minf {
namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// The device address of this device's copy of the scratch array (looked up on first use).
int scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MINF_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return MINF_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
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
    const int st = scratch_for_current_device(&ws);
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
