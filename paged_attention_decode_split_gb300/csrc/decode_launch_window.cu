// decode_launch_window.cu -- the sliding-window decode instantiations, in a
// translation unit of their own so they compile in parallel with the rest.
#include "decode_launch.cuh"

namespace pa {

cudaError_t launch_decode_window(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    return launch_decode_cfg<true, false>(head_dim, group, tk, tv, p, grid, stream);
}

}  // namespace pa
