// minf_decode_q8.cu -- the Q8_0-region instantiation of the decode kernel, compiled apart from
// the others so that they build in parallel.
#include "minf_decode.cuh"

namespace minf {

cudaError_t dispatch_decode_q8(int hd_kv, bool fused, int gh, const CUtensorMap &tk, const CUtensorMap &tv,
                               const CUtensorMap &tks, const CUtensorMap &tvs, const dec::KParams &k, int grid,
                               cudaStream_t s, bool pdl) {
    return dec::dispatch<Q8>(hd_kv, fused, gh, tk, tv, tks, tvs, k, grid, s, pdl);
}

}  // namespace minf
