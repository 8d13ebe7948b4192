// minf_decode_f16.cu -- the binary16-region instantiation of the decode kernel, compiled
// apart from the fp32 one so that the two build in parallel.
#include "minf_decode.cuh"

namespace minf {

cudaError_t dispatch_decode_f16(int hd_kv, bool fused, int gh, const CUtensorMap &tk, const CUtensorMap &tv,
                                const dec::KParams &k, int grid, cudaStream_t s, bool pdl) {
    return dec::dispatch<__half>(hd_kv, fused, gh, tk, tv, k, grid, s, pdl);
}

}  // namespace minf
