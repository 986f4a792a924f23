// decode_launch_fp8.cu -- the decode instantiations over an fp8 e4m3 cache
// (full attention), in a translation unit of their own so they compile in
// parallel with the rest.
#include "decode_launch.cuh"

namespace pa {

cudaError_t launch_decode_fp8_full(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                                   const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    return launch_decode_cfg<false, true>(head_dim, group, tk, tv, p, grid, stream);
}

}  // namespace pa
