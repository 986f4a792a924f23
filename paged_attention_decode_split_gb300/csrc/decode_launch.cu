// decode_launch.cu -- instantiates the split-KV decode kernel for the
// (head_dim, GQA group) pairs of the models served here and launches it, and
// launches the partition-reduce kernel as a programmatic dependent of it.
#include "pa_internal.h"

namespace pa {

namespace {

template <int D, int G, int TS, int NST, int SPS>
cudaError_t launch_decode_t(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, dim3 grid,
                            cudaStream_t stream, int slot) {
    using C = DecodeCfg<D, G, TS, NST, SPS>;
    auto kern = pa_decode_split_kernel<D, G, TS, NST, SPS>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(kern), C::SMEM_BYTES, slot);
    if (e != cudaSuccess) return e;
    // Programmatic dependent launch: the kernel's set-up overlaps the previous
    // kernel in the stream (e.g. reshape_and_cache); it waits for that kernel
    // before touching global memory.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace

bool decode_supported(int head_dim, int group) {
    if (head_dim == 256) return group == 1 || group == 2 || group == 4 || group == 6;
    if (head_dim == 128) return group == 1 || group == 2 || group == 4 || group == 6 || group == 8;
    return false;
}

// Per (head_dim, group): warps per chunk (TS), chunk streams (NST), stages
// per stream (SPS).  D = 256: 6 streams x 2 stages x 16 KiB; groups of 4 and
// 6 heads split each chunk's tokens over 2 warps, giving 13 warps per CTA.
// D = 128: 12 streams x 2 x 8 KiB, or 6 streams x 4 with the tokens split
// over 2 warps.
cudaError_t launch_decode(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    if (head_dim == 256) {
        switch (group) {
            case 1: return launch_decode_t<256, 1, 1, 6, 2>(tk, tv, p, grid, stream, 0);
            case 2: return launch_decode_t<256, 2, 1, 6, 2>(tk, tv, p, grid, stream, 1);
            case 4: return launch_decode_t<256, 4, 2, 4, 3>(tk, tv, p, grid, stream, 2);
            case 6: return launch_decode_t<256, 6, 2, 4, 3>(tk, tv, p, grid, stream, 3);
        }
    } else if (head_dim == 128) {
        switch (group) {
            case 1: return launch_decode_t<128, 1, 1, 12, 2>(tk, tv, p, grid, stream, 4);
            case 2: return launch_decode_t<128, 2, 1, 12, 2>(tk, tv, p, grid, stream, 5);
            case 4: return launch_decode_t<128, 4, 2, 6, 4>(tk, tv, p, grid, stream, 6);
            case 6: return launch_decode_t<128, 6, 2, 4, 6>(tk, tv, p, grid, stream, 7);
            case 8: return launch_decode_t<128, 8, 2, 4, 6>(tk, tv, p, grid, stream, 8);
        }
    }
    return cudaErrorInvalidValue;
}

// rows = sequences x query rows per sequence.  Few splits: one warp per
// (row, head); many splits: a CTA per (head, row, 64-dim slice) whose threads
// split the splits.
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
    cfg.gridDim = dim3(p.num_q_heads, rows, head_dim / 64);
    cfg.blockDim = dim3(128);
    if (head_dim == 256) return cudaLaunchKernelEx(&cfg, pa_split_reduce_kernel<256>, p);
    if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_split_reduce_kernel<128>, p);
    return cudaErrorInvalidValue;
}

}  // namespace pa
