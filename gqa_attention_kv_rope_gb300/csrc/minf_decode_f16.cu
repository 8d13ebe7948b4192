// minf_decode_f16.cu -- the binary16-region instantiation of the decode kernel, compiled apart
// from the others so that they build in parallel.
#include "minf_decode.cuh"

namespace minf {

cudaError_t dispatch_decode_f16(int hd_kv, bool fused, int gh, const CUtensorMap &tk, const CUtensorMap &tv,
                                const CUtensorMap &tks, const CUtensorMap &tvs, const dec::KParams &k, int grid,
                                cudaStream_t s, bool pdl) {
    return dec::dispatch<__half>(hd_kv, fused, gh, tk, tv, tks, tvs, k, grid, s, pdl);
}

}  // namespace minf
