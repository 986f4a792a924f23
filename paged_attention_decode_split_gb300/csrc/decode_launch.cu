// decode_launch.cu -- launches the split-KV decode kernel (full attention
// here, sliding window and fp8 in their own translation units) and the
// partition-reduce kernel, a programmatic dependent of the split kernel of a
// decode or verify call.
#include "decode_launch.cuh"

namespace pa {

bool decode_supported(int head_dim, int group) {
    if (head_dim != 256 && head_dim != 128) return false;
    switch (group) {
        case 1: case 2: case 3: case 4: case 5: case 6: case 8: case 12: case 16: return true;
    }
    return false;
}

cudaError_t launch_decode(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    if (p.window > 0) return launch_decode_window(head_dim, group, tk, tv, p, grid, stream);
    return launch_decode_cfg<false, false>(head_dim, group, tk, tv, p, grid, stream);
}

cudaError_t launch_decode_fp8(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                              const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    if (p.window > 0) return launch_decode_fp8_window(head_dim, group, tk, tv, p, grid, stream);
    return launch_decode_fp8_full(head_dim, group, tk, tv, p, grid, stream);
}

cudaError_t launch_reduce(int head_dim, const ReduceParams &p, int rows, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.num_splits <= kReduceSmallMaxSplits) {
        const int pairs = rows * p.num_q_heads;
        cfg.gridDim = dim3((pairs + 7) / 8);
        cfg.blockDim = dim3(256);
        if (head_dim == 256) return cudaLaunchKernelEx(&cfg, pa_split_reduce_small_kernel<256>, p, pairs);
        if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_split_reduce_small_kernel<128>, p, pairs);
        return cudaErrorInvalidValue;
    }
    cfg.gridDim = dim3(p.num_q_heads, rows, head_dim / 32);
    cfg.blockDim = dim3(128);
    if (head_dim == 256) return cudaLaunchKernelEx(&cfg, pa_split_reduce_kernel<256>, p);
    if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_split_reduce_kernel<128>, p);
    return cudaErrorInvalidValue;
}

}  // namespace pa
