// verify_launch.cu -- instantiates the multi-row verify kernel per head_dim
// and number of 16-row slices, and launches it.
#include "pa_internal.h"
#include "verify_tc.cuh"

namespace pa {

namespace {

template <int D, int NWC>
cudaError_t launch_verify_t(const CUtensorMap &tk, const CUtensorMap &tv, const VerifyParams &p, dim3 grid,
                            cudaStream_t stream, int slot) {
    constexpr int NS = 8;
    using C = VerifyCfg<D, NWC, NS>;
    auto kern = pa_verify_mma_kernel<D, NWC, NS>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(kern), C::SMEM_BYTES, slot);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

template <int D, int NS>
cudaError_t launch_verify_tc(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tk64,
                             const CUtensorMap &tv64, const VerifyParams &p, dim3 grid, cudaStream_t stream,
                             int slot) {
    using C = VerifyTcCfg<D, NS>;
    auto kern = pa_verify_tc_kernel<D, NS>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(kern), C::SMEM_BYTES, slot);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tk, tv, tk64, tv64, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_verify_d(int slices, const CUtensorMap &tk, const CUtensorMap &tv, const VerifyParams &p,
                            dim3 grid, cudaStream_t stream, int slot0) {
    switch (slices) {
        case 1: return launch_verify_t<D, 1>(tk, tv, p, grid, stream, slot0 + 0);
        case 2: return launch_verify_t<D, 2>(tk, tv, p, grid, stream, slot0 + 1);
        case 3: return launch_verify_t<D, 3>(tk, tv, p, grid, stream, slot0 + 2);
        case 4: return launch_verify_t<D, 4>(tk, tv, p, grid, stream, slot0 + 3);
        case 5: return launch_verify_t<D, 5>(tk, tv, p, grid, stream, slot0 + 4);
        case 6: return launch_verify_t<D, 6>(tk, tv, p, grid, stream, slot0 + 5);
        case 7: return launch_verify_t<D, 7>(tk, tv, p, grid, stream, slot0 + 6);
        case 8: return launch_verify_t<D, 8>(tk, tv, p, grid, stream, slot0 + 7);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

bool verify_supported(int head_dim, int rows) {
    return (head_dim == 256 || head_dim == 128) && rows >= 1 && rows <= 128;
}

cudaError_t launch_verify(int head_dim, int rows, const CUtensorMap &tk, const CUtensorMap &tv,
                          const CUtensorMap &tk64, const CUtensorMap &tv64, const VerifyParams &p, dim3 grid,
                          cudaStream_t stream) {
    (void)rows;  // every row count up to 128 runs as one M = 128 block
    if (head_dim == 256) return launch_verify_tc<256, 2>(tk, tv, tk64, tv64, p, grid, stream, 32);
    if (head_dim == 128) return launch_verify_tc<128, 4>(tk, tv, tk64, tv64, p, grid, stream, 33);
    return cudaErrorInvalidValue;
}

}  // namespace pa
