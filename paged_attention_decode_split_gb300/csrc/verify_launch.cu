// verify_launch.cu -- instantiates the tensor-core verify kernel per head_dim
// and launches it.
#include "pa_internal.h"

namespace pa {

namespace {

template <int D, int NK, int NV>
cudaError_t launch_verify_tc(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tk64,
                             const CUtensorMap &tv64, const VerifyParams &p, dim3 grid, cudaStream_t stream,
                             int slot) {
    using C = VerifyTcCfg<D, NK, NV>;
    auto kern = pa_verify_tc_kernel<D, NK, NV>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(kern), C::SMEM_BYTES, slot);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tk, tv, tk64, tv64, p);
    return cudaGetLastError();
}

}  // namespace

bool verify_supported(int head_dim, int rows) {
    return (head_dim == 256 || head_dim == 128) && rows >= 1 && rows <= 128;
}

cudaError_t launch_verify(int head_dim, int rows, const CUtensorMap &tk, const CUtensorMap &tv,
                          const CUtensorMap &tk64, const CUtensorMap &tv64, const VerifyParams &p, dim3 grid,
                          cudaStream_t stream) {
    (void)rows;  // every row count up to 128 runs as one M = 128 block
    if (head_dim == 256) return launch_verify_tc<256, 4, 3>(tk, tv, tk64, tv64, p, grid, stream, 32);
    if (head_dim == 128) return launch_verify_tc<128, 6, 6>(tk, tv, tk64, tv64, p, grid, stream, 33);
    return cudaErrorInvalidValue;
}

}  // namespace pa
