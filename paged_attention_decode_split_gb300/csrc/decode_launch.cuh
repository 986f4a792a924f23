// decode_launch.cuh -- the decode kernel instantiations per (head_dim, GQA
// group), shared by the full-attention and the sliding-window translation
// units (compiled in parallel).
#pragma once

#include "pa_internal.h"

namespace pa {

template <int D, int G, int TS, int NST, int SPS, int HG, bool WIN, bool F8>
cudaError_t launch_decode_t(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, dim3 grid,
                            cudaStream_t stream, int slot) {
    using C = DecodeCfg<D, G, TS, NST, SPS, HG, F8 ? 1 : 2>;
    auto kern = pa_decode_split_kernel<D, G, TS, NST, SPS, HG, WIN, F8>;
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

// Per (head_dim, group): token halves (TS), chunk streams (NST), stages per
// stream (SPS), head groups (HG).  D = 256: groups of 4 and 6 heads run 4
// streams x 3 stages x 16 KiB with each chunk's tokens split over 2 warps (9
// warps, 168 registers); groups of 1 and 2 run 6 streams x 2 stages, one
// warp per chunk; 12 heads split into 3 head groups of 4, each warp taking a
// whole chunk (4 streams x 3 stages, 13 warps: measured 54.6 us against 60 us
// for 2 groups of 6 with split tokens at 32K).  D = 128: 12 streams x 2 x 8
// KiB for small groups, else the tokens split over 2 warps.  Groups of 3 and 5
// heads run like 4 and 6; 8 and 16 heads split into head groups of 4 (D = 256)
// or 8 (D = 128, 16 heads).  An fp8 cache halves the stage, and
// each stream owns twice the stages: the same bytes in flight per SM.
template <bool WIN, bool F8>
cudaError_t launch_decode_cfg(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                              const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    // shared-memory limit bookkeeping: one slot per kernel
    constexpr int slot0 = (WIN ? 20 : 0) + (F8 ? 40 : 0);
    if constexpr (F8) {
        if (head_dim == 256) {
            switch (group) {
                case 1: return launch_decode_t<256, 1, 1, 6, 4, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 0);
                case 2: return launch_decode_t<256, 2, 1, 6, 4, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 1);
                case 4: return launch_decode_t<256, 4, 2, 4, 6, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 2);
                case 6: return launch_decode_t<256, 6, 2, 4, 6, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 3);
                case 12: return launch_decode_t<256, 12, 1, 4, 6, 3, WIN, F8>(tk, tv, p, grid, stream, slot0 + 9);
                case 3: return launch_decode_t<256, 3, 2, 4, 6, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 11);
                case 5: return launch_decode_t<256, 5, 2, 4, 6, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 12);
                case 8: return launch_decode_t<256, 8, 1, 4, 6, 2, WIN, F8>(tk, tv, p, grid, stream, slot0 + 13);
                case 16: return launch_decode_t<256, 16, 1, 3, 8, 4, WIN, F8>(tk, tv, p, grid, stream, slot0 + 14);
            }
        } else if (head_dim == 128) {
            switch (group) {
                case 1: return launch_decode_t<128, 1, 1, 12, 4, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 4);
                case 2: return launch_decode_t<128, 2, 1, 12, 4, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 5);
                case 4: return launch_decode_t<128, 4, 2, 6, 8, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 6);
                case 6: return launch_decode_t<128, 6, 2, 4, 12, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 7);
                case 8: return launch_decode_t<128, 8, 2, 4, 12, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 8);
                case 12: return launch_decode_t<128, 12, 2, 2, 24, 2, WIN, F8>(tk, tv, p, grid, stream, slot0 + 10);
                case 3: return launch_decode_t<128, 3, 2, 6, 8, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 15);
                case 5: return launch_decode_t<128, 5, 2, 4, 12, 1, WIN, F8>(tk, tv, p, grid, stream, slot0 + 16);
                case 16: return launch_decode_t<128, 16, 1, 4, 12, 2, WIN, F8>(tk, tv, p, grid, stream, slot0 + 17);
            }
        }
        return cudaErrorInvalidValue;
    }
    if (head_dim == 256) {
        switch (group) {
            case 1: return launch_decode_t<256, 1, 1, 6, 2, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 0);
            case 2: return launch_decode_t<256, 2, 1, 6, 2, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 1);
            case 4: return launch_decode_t<256, 4, 2, 4, 3, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 2);
            case 6: return launch_decode_t<256, 6, 2, 4, 3, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 3);
            case 12: return launch_decode_t<256, 12, 1, 4, 3, 3, WIN, false>(tk, tv, p, grid, stream, slot0 + 9);
            case 3: return launch_decode_t<256, 3, 2, 4, 3, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 11);
            case 5: return launch_decode_t<256, 5, 2, 4, 3, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 12);
            case 8: return launch_decode_t<256, 8, 1, 4, 3, 2, WIN, false>(tk, tv, p, grid, stream, slot0 + 13);
            case 16: return launch_decode_t<256, 16, 1, 3, 4, 4, WIN, false>(tk, tv, p, grid, stream, slot0 + 14);
        }
    } else if (head_dim == 128) {
        switch (group) {
            case 1: return launch_decode_t<128, 1, 1, 12, 2, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 4);
            case 2: return launch_decode_t<128, 2, 1, 12, 2, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 5);
            case 4: return launch_decode_t<128, 4, 2, 6, 4, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 6);
            case 6: return launch_decode_t<128, 6, 2, 4, 6, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 7);
            case 8: return launch_decode_t<128, 8, 2, 4, 6, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 8);
            case 12: return launch_decode_t<128, 12, 2, 2, 12, 2, WIN, false>(tk, tv, p, grid, stream, slot0 + 10);
            case 3: return launch_decode_t<128, 3, 2, 6, 4, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 15);
            case 5: return launch_decode_t<128, 5, 2, 4, 6, 1, WIN, false>(tk, tv, p, grid, stream, slot0 + 16);
            case 16: return launch_decode_t<128, 16, 1, 4, 6, 2, WIN, false>(tk, tv, p, grid, stream, slot0 + 17);
        }
    }
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
