// verify_launch.cu -- instantiates the tensor-core verify kernel per head_dim
// and launches it.
#include "pa_internal.h"

namespace pa {

namespace {

template <int D, int NK, int NV, int NSG, int NSB, int TK = 64>
cudaError_t launch_verify_tc(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tk64,
                             const CUtensorMap &tv64, const VerifyParams &p, dim3 grid, cudaStream_t stream,
                             int slot) {
    using C = VerifyTcCfg<D, NK, NV, NSG, NSB, TK>;
    auto kern = pa_verify_tc_kernel<D, NK, NV, NSG, NSB, TK>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(kern), C::SMEM_BYTES, slot);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: the set-up overlaps the work before it
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
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, tk64, tv64, p);
}

}  // namespace

// Rows beyond 128 run as several 128-row blocks (grid y = Hkv x blocks), up
// to q_len 4096 x G 8 = 32768 rows.
bool verify_supported(int head_dim, int rows) {
    return (head_dim == 256 || head_dim == 128) && rows >= 1 && rows <= 32768;
}

bool verify_wide_score_tiles(int head_dim, int rows) { return (head_dim == 256 || head_dim == 128) && rows > 128; }

// Each CTA runs one M = 128 block of rows.  With several blocks per KV head
// the blocks read their tiles mostly from L2 and the score product's
// instruction rate bounds the tile: 128-key score tiles (D = 256: Q in shared
// memory, one K slot of 128 keys and three V slots of 64; D = 128: Q in tensor
// memory, three K slots and six V slots).  A single block streams from HBM and
// keeps the 64-key tiles and deeper rings.
cudaError_t launch_verify(int head_dim, int rows, const CUtensorMap &tk, const CUtensorMap &tv,
                          const CUtensorMap &tk64, const CUtensorMap &tv64, const CUtensorMap &tk128,
                          const VerifyParams &p, dim3 grid, cudaStream_t stream) {
    const bool wide = verify_wide_score_tiles(head_dim, rows);  // (K's whole-tile boxes are then 128 tokens)
    if (head_dim == 256)
        return wide ? launch_verify_tc<256, 1, 3, 0, 2, 128>(tk, tv, tk128, tv64, p, grid, stream, 104)
                    : launch_verify_tc<256, 4, 3, 0, 2>(tk, tv, tk64, tv64, p, grid, stream, 100);
    if (head_dim == 128)
        return wide ? launch_verify_tc<128, 3, 6, 0, 2, 128>(tk, tv, tk128, tv64, p, grid, stream, 105)
                    : launch_verify_tc<128, 6, 6, 0, 2>(tk, tv, tk64, tv64, p, grid, stream, 101);
    return cudaErrorInvalidValue;
}

// fp8 cache: the f16 rings shrink to make room for the e4m3 staging rings
// (D = 256: 2 K + 3 V slots of 32 KiB and 2 + 2 staging slots of 16 KiB).
cudaError_t launch_verify_fp8(int head_dim, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tk64,
                              const CUtensorMap &tv64, const VerifyParams &p, dim3 grid, cudaStream_t stream) {
    if (head_dim == 256) return launch_verify_tc<256, 2, 3, 2, 2>(tk, tv, tk64, tv64, p, grid, stream, 102);
    if (head_dim == 128) return launch_verify_tc<128, 4, 4, 4, 2>(tk, tv, tk64, tv64, p, grid, stream, 103);
    return cudaErrorInvalidValue;
}

}  // namespace pa
