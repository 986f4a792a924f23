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

namespace {

// The few-split merge with NSL register slots (>= S) and PPW pairs per warp.
template <int D, int NSL, int PPW>
cudaError_t launch_reduce_small_t(cudaLaunchConfig_t cfg, const ReduceParams &p, int pairs, int slot) {
    auto kern = pa_split_reduce_small_kernel<D, NSL, PPW>;
    const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(kern), kReduceSmallSmem, slot);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((pairs + 8 * PPW - 1) / (8 * PPW));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = kReduceSmallSmem;
    return cudaLaunchKernelEx(&cfg, kern, p, pairs);
}

template <int D, int NSL>
cudaError_t launch_reduce_small_n(cudaLaunchConfig_t cfg, const ReduceParams &p, int pairs, int ppw, int slot) {
    if (ppw <= 1) return launch_reduce_small_t<D, NSL, 1>(cfg, p, pairs, slot);
    if constexpr (NSL * 3 > 16) {  // 8 slots: at most 2 pairs per warp in registers
        return launch_reduce_small_t<D, NSL, 2>(cfg, p, pairs, slot + 1);
    } else {
        if (ppw <= 2) return launch_reduce_small_t<D, NSL, 2>(cfg, p, pairs, slot + 1);
        if (ppw <= 3) return launch_reduce_small_t<D, NSL, 3>(cfg, p, pairs, slot + 2);
        return launch_reduce_small_t<D, NSL, 4>(cfg, p, pairs, slot + 3);
    }
}

}  // namespace

cudaError_t launch_reduce(int head_dim, const ReduceParams &p, int rows, int num_sms, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.num_splits <= kReduceSmallMaxSplits) {
        // pairs per warp: as few as keep the grid within one CTA per SM (up to 4)
        const int pairs = rows * p.num_q_heads;
        const int sms = num_sms > 0 ? num_sms : 1;
        const int ppw = (pairs + 8 * sms - 1) / (8 * sms);
        // kernel slots 110..133: four per (head_dim, split slots)
        if (head_dim == 256) {
            if (p.num_splits <= 2) return launch_reduce_small_n<256, 2>(cfg, p, pairs, ppw, 110);
            if (p.num_splits <= 4) return launch_reduce_small_n<256, 4>(cfg, p, pairs, ppw, 114);
            return launch_reduce_small_n<256, 8>(cfg, p, pairs, ppw, 118);
        }
        if (head_dim == 128) {
            if (p.num_splits <= 2) return launch_reduce_small_n<128, 2>(cfg, p, pairs, ppw, 122);
            if (p.num_splits <= 4) return launch_reduce_small_n<128, 4>(cfg, p, pairs, ppw, 126);
            return launch_reduce_small_n<128, 8>(cfg, p, pairs, ppw, 130);
        }
        return cudaErrorInvalidValue;
    }
    cfg.gridDim = dim3(p.num_q_heads, rows, head_dim / 32);
    cfg.blockDim = dim3(128);
    if (head_dim == 256) return cudaLaunchKernelEx(&cfg, pa_split_reduce_kernel<256>, p);
    if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_split_reduce_kernel<128>, p);
    return cudaErrorInvalidValue;
}

}  // namespace pa
