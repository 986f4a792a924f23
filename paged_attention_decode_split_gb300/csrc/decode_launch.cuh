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
    // L2 prefetch ahead of the dependency wait: 6 chunks for the 8 KiB bf16
    // stages of D = 128 (32K dense control: 23.4 -> 22.5 us); none elsewhere
    // (hybrid bf16 within noise, fp8 slower, and more chunks slower for all)
    constexpr int PF = (D == 128 && !F8) ? 6 : 0;
    using C = MmaCfg<D, NT, NST, SPS, DS, F8>;
    auto kern = pa_decode_mma_kernel<D, G, NT, NST, SPS, DS, WIN, F8, LP, PF>;
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
// Chosen by measurement (32K context, one layer call in a 16-layer graph):
//  * bf16, D = 256: 16 KiB stages; 2 streams x 6 stages, 2 warps per chunk,
//    one producer lane (23.2 us against 24.1 with 4 x 3, 23.4 with 3 x 4 and
//    25.2 with a lane per stream).  12 and 16 heads take the same layout
//    (12 heads: 24.4 us against 25.1 with 3 x 4); fewer streams with more
//    stages each kept more copies in flight per stream.
//  * bf16, D = 128: 8 KiB stages; 4 streams x 6 stages, 2 warps per chunk, a
//    producer lane per stream (one issuing lane caps a CTA at about one stage
//    per 0.3 us, which stages under 16 KiB feel): 23.7 us against 24.7 with
//    8 x 3 and one warp per chunk; 12 and 16 heads: 8 x 3, one warp.
//  * fp8, D = 256: 8 KiB stages; 4 streams x 6 stages, one warp per chunk, a
//    lane per stream (17.0 us against 17.2 with 8 x 3, 20.0 with 2 x 12;
//    with the unmasked P.V of full chunks 15.25 us against 15.85 with 3 x 8,
//    16.25 with 6 x 4, 17.4 with 8 x 3).  12 and 16 heads take the same layout
//    (22.1 / 22.5 us against 23.2 / 23.1 with 3 x 8 x 2 and 27.1 / 28.5 with
//    4 x 6 x 2), although their accumulators and Q fragments spill 20 / 76
//    bytes at 255 registers.
//  * fp8, D = 128: 4 KiB stages; 12 streams x 4 stages, a lane per stream;
//    12 and 16 heads: 6 x 8, one warp per chunk (registers, as above).
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
            PA_DECODE_CASES(256, 4, 6, 1, true, 4, 6, 1, slot0)
        } else if (head_dim == 128) {
            PA_DECODE_CASES(128, 12, 4, 1, true, 6, 8, 1, slot0 + 10)
        }
    } else {
        if (head_dim == 256) {
            PA_DECODE_CASES(256, 2, 6, 2, false, 2, 6, 2, slot0)
        } else if (head_dim == 128) {
            PA_DECODE_CASES(128, 4, 6, 2, true, 8, 3, 1, slot0 + 10)
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
