// decode_launch.cuh -- the decode kernel instantiations per (head_dim, GQA
// group), shared by the translation units of the full-attention, sliding-
// window and fp8 variants (compiled in parallel).
#pragma once

#include "pa_internal.h"

namespace pa {

template <int D, int G, int NST, int SPS, int DS, bool WIN, bool F8, bool LP>
cudaError_t launch_decode_mma_t(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, dim3 grid,
                                cudaStream_t stream, int slot) {
    constexpr int NT = G > 8 ? 2 : 1;
    using C = MmaCfg<D, NT, NST, SPS, DS, F8>;
    auto kern = pa_decode_mma_kernel<D, G, NT, NST, SPS, DS, WIN, F8, LP>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(kern), C::SMEM_BYTES, slot);
    if (e != cudaSuccess) return e;
    // Programmatic dependent launch: the kernel's set-up overlaps the previous
    // kernel in the stream (e.g. reshape_and_cache); it waits for that kernel
    // before touching global memory (early_kv: before touching q, the new row,
    // the workspace or the output).
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

// Per (head_dim, cache type): chunk streams (NST), stages per stream (SPS),
// warps per chunk (DS, splitting the d range of P.V), a producer lane per
// stream (LP).  Every layout keeps about 192 KiB of stages per SM in flight.
//  * bf16, D = 256: 16 KiB stages; 2 streams x 6 stages, 2 warps per chunk
//    (32K call 23.2 us, against 24.1 with 4 x 3 and 23.4 with 3 x 4; 12 and
//    16 heads: 3 streams x 4 stages, so that 7 warps leave each warp the
//    registers of 16 heads' Q fragments and accumulators).
//  * bf16, D = 128 and fp8, D = 256: 8 KiB stages; 8 streams x 3 stages, a
//    producer lane per stream (one issuing lane caps a CTA at about one
//    stage per 0.3 us, which stages under 16 KiB feel).
//  * fp8, D = 128: 4 KiB stages; 12 streams x 4 stages, a lane per stream.
//  * 12 and 16 heads over fp8 take fewer warps (3 streams x 8 stages with 2
//    warps per chunk at D = 256, 6 x 8 with one at D = 128) for the same
//    register reason.
template <bool WIN, bool F8>
cudaError_t launch_decode_cfg(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                              const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    // shared-memory limit bookkeeping: one slot per kernel
    constexpr int slot0 = (WIN ? 20 : 0) + (F8 ? 40 : 0);
#define PA_DECODE_CASES(D, NST, SPS, DS, LP, NST2, SPS2, DS2, S0)                                             \
    switch (group) {                                                                                          \
        case 1: return launch_decode_mma_t<D, 1, NST, SPS, DS, WIN, F8, LP>(tk, tv, p, grid, stream, S0 + 0);  \
        case 2: return launch_decode_mma_t<D, 2, NST, SPS, DS, WIN, F8, LP>(tk, tv, p, grid, stream, S0 + 1);  \
        case 3: return launch_decode_mma_t<D, 3, NST, SPS, DS, WIN, F8, LP>(tk, tv, p, grid, stream, S0 + 2);  \
        case 4: return launch_decode_mma_t<D, 4, NST, SPS, DS, WIN, F8, LP>(tk, tv, p, grid, stream, S0 + 3);  \
        case 5: return launch_decode_mma_t<D, 5, NST, SPS, DS, WIN, F8, LP>(tk, tv, p, grid, stream, S0 + 4);  \
        case 6: return launch_decode_mma_t<D, 6, NST, SPS, DS, WIN, F8, LP>(tk, tv, p, grid, stream, S0 + 5);  \
        case 8: return launch_decode_mma_t<D, 8, NST, SPS, DS, WIN, F8, LP>(tk, tv, p, grid, stream, S0 + 6);  \
        case 12:                                                                                              \
            return launch_decode_mma_t<D, 12, NST2, SPS2, DS2, WIN, F8, LP>(tk, tv, p, grid, stream, S0 + 7); \
        case 16:                                                                                              \
            return launch_decode_mma_t<D, 16, NST2, SPS2, DS2, WIN, F8, LP>(tk, tv, p, grid, stream, S0 + 8); \
    }                                                                                                         \
    return cudaErrorInvalidValue;
    if constexpr (F8) {
        if (head_dim == 256) {
            PA_DECODE_CASES(256, 8, 3, 1, true, 3, 8, 2, slot0)
        } else if (head_dim == 128) {
            PA_DECODE_CASES(128, 12, 4, 1, true, 6, 8, 1, slot0 + 10)
        }
    } else {
        if (head_dim == 256) {
            PA_DECODE_CASES(256, 2, 6, 2, false, 3, 4, 2, slot0)
        } else if (head_dim == 128) {
            PA_DECODE_CASES(128, 8, 3, 1, true, 8, 3, 1, slot0 + 10)
        }
    }
#undef PA_DECODE_CASES
    return cudaErrorInvalidValue;
}

// the sliding-window instantiations (decode_launch_window.cu) and the fp8
// ones (decode_launch_fp8.cu, decode_launch_fp8_window.cu)
cudaError_t launch_decode_window(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const DecodeParams &p, dim3 grid, cudaStream_t stream);
cudaError_t launch_decode_fp8_full(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                                   const DecodeParams &p, dim3 grid, cudaStream_t stream);
cudaError_t launch_decode_fp8_window(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                                     const DecodeParams &p, dim3 grid, cudaStream_t stream);

}  // namespace pa
