// decode_launch_fp8_window.cu -- the sliding-window decode instantiations over
// an fp8 e4m3 cache, in a translation unit of their own.
#include "decode_launch.cuh"

namespace pa {

cudaError_t launch_decode_fp8_window(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                                     const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    return launch_decode_cfg<true, true>(head_dim, group, tk, tv, p, grid, stream);
}

}  // namespace pa
