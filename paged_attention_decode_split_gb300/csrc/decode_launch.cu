// decode_launch.cu -- instantiates the split-KV decode kernel for the
// (head_dim, GQA group) pairs of the models served here and launches it, and
// launches the partition-reduce kernel as a programmatic dependent of it.
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kDecodeWarps = 7;  // consumer warps per CTA (+1 producer warp): 8 warps keep the 255-register budget

template <int D>
constexpr int decode_stages() {
    return D == 256 ? 12 : 16;  // 12 x 16 KiB or 16 x 8 KiB of K/V in flight per CTA
}

template <int D, int G>
cudaError_t launch_decode_t(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, dim3 grid,
                            cudaStream_t stream, int slot) {
    constexpr int NS = decode_stages<D>();
    using C = DecodeCfg<D, G, kDecodeWarps, NS>;
    auto kern = pa_decode_split_kernel<D, G, kDecodeWarps, NS>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(kern), C::SMEM_BYTES, slot);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

bool decode_supported(int head_dim, int group) {
    if (head_dim == 256) return group == 1 || group == 2 || group == 4 || group == 6;
    if (head_dim == 128) return group == 1 || group == 2 || group == 4 || group == 6 || group == 8;
    return false;
}

cudaError_t launch_decode(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    if (head_dim == 256) {
        switch (group) {
            case 1: return launch_decode_t<256, 1>(tk, tv, p, grid, stream, 0);
            case 2: return launch_decode_t<256, 2>(tk, tv, p, grid, stream, 1);
            case 4: return launch_decode_t<256, 4>(tk, tv, p, grid, stream, 2);
            case 6: return launch_decode_t<256, 6>(tk, tv, p, grid, stream, 3);
        }
    } else if (head_dim == 128) {
        switch (group) {
            case 1: return launch_decode_t<128, 1>(tk, tv, p, grid, stream, 4);
            case 2: return launch_decode_t<128, 2>(tk, tv, p, grid, stream, 5);
            case 4: return launch_decode_t<128, 4>(tk, tv, p, grid, stream, 6);
            case 6: return launch_decode_t<128, 6>(tk, tv, p, grid, stream, 7);
            case 8: return launch_decode_t<128, 8>(tk, tv, p, grid, stream, 8);
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce(int head_dim, const ReduceParams &p, dim3 grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (head_dim == 256) return cudaLaunchKernelEx(&cfg, pa_split_reduce_kernel<256>, p);
    if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_split_reduce_kernel<128>, p);
    return cudaErrorInvalidValue;
}

}  // namespace pa
