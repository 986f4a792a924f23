// decode_launch.cuh -- the decode kernel instantiations per (head_dim, GQA
// group), shared by the full-attention and the sliding-window translation
// units (compiled in parallel).
#pragma once

#include <atomic>

#include "pa_internal.h"

namespace pa {

template <int D, int G, int TS, int NST, int SPS, int HG, bool WIN, bool F8, bool LP, bool RB = false>
cudaError_t launch_decode_t(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, dim3 grid,
                            cudaStream_t stream, int slot) {
    using C = DecodeCfg<D, G, TS, NST, SPS, HG, F8 ? 1 : 2, RB ? 4 : 1>;
    auto kern = pa_decode_split_kernel<D, G, TS, NST, SPS, HG, WIN, F8, LP, RB>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(kern), C::SMEM_BYTES, slot);
    if (e != cudaSuccess) return e;
    if constexpr (RB) {
        // The warpgroups' register budgets add up to REG_LAUNCH per thread;
        // a kernel launched with fewer registers would wait forever in
        // setmaxnreg.inc, so it is not launched.
        static std::atomic<int> launch_regs{0};  // per instantiation; the same on every sm_103a device
        int regs = launch_regs.load(std::memory_order_relaxed);
        if (regs == 0) {
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void *>(kern));
            if (e != cudaSuccess) return e;
            regs = fa.numRegs;
            launch_regs.store(regs, std::memory_order_relaxed);
        }
        if (regs * C::THREADS < 128 * C::REG_PRODUCER + C::NWC * 32 * C::REG_CONSUMER)
            return cudaErrorInvalidConfiguration;
    }
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
// stream (SPS), head groups (HG), a producer lane per stream (LP).
//  * D = 256: groups of 3 to 6 heads run 4 streams x 3 stages x 16 KiB with
//    each chunk's tokens split over 2 warps (9 warps, 168 registers; for 4
//    and 6 heads the producer sits in a warpgroup of its own that hands its
//    registers to the 8 consumers, 232 each: no spills, the 16-layer step at
//    32K measured 0.528 ms against 0.537 ms, and a 4-head call 28.7 us
//    against 29.2 us; for 3 and 5 heads the same change measured within
//    noise or slower, so they keep the even split); groups of 1 and 2 run
//    6 streams x 2 stages, one warp per chunk.  8, 12 and 16 heads also take
//    the producer warpgroup, whose registers let a warp hold more heads:
//    8 heads in one warp with split tokens (40.65 -> 40.36 us at 32K), 12
//    and 16 heads in 2 head groups of 6 and 8, each warp taking a whole chunk
//    (54.7 -> 52.8 us and 69.7 -> 68.6 us against 3 and 4 groups of 4 at
//    the even split).  One producer lane serves all streams.
//  * D = 128 (8 KiB stages): every stream has its own producer lane.  Up to 4
//    heads: 12 streams x 2 stages (1 and 2 heads) or 6 x 4 with split tokens;
//    5 and 6 heads: 6 x 4 with split tokens; 8, 12 and 16 heads: head groups
//    of 4 (8 x 3, 6 x 4 and 4 x 6 streams x stages).  Measured at 32K over
//    8 KV heads against one producer lane and the earlier layouts: 4 heads 41.9 -> 28.3 us, 8 heads 48.6 -> 46.3 us, 12 heads
//    68.9 -> 65.3 us.
//  * An fp8 cache halves the stage and each stream owns twice the stages:
//    the same bytes in flight per SM.  At D = 256, groups of up to 4 heads
//    take a producer lane per stream (1 head: 21.3 -> 17.5 us at 32K); wider
//    groups, whose widening arithmetic bounds them, measured 0-1 % faster
//    with one lane.  The 6-head fp8 kernel also takes the producer
//    warpgroup (33.9 -> 32.6 us at 32K).
template <bool WIN, bool F8>
cudaError_t launch_decode_cfg(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                              const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    // shared-memory limit bookkeeping: one slot per kernel
    constexpr int slot0 = (WIN ? 20 : 0) + (F8 ? 40 : 0);
    if constexpr (F8) {
        if (head_dim == 256) {
            switch (group) {
                case 1: return launch_decode_t<256, 1, 1, 6, 4, 1, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 0);
                case 2: return launch_decode_t<256, 2, 1, 6, 4, 1, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 1);
                case 4: return launch_decode_t<256, 4, 2, 4, 6, 1, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 2);
                case 6: return launch_decode_t<256, 6, 2, 4, 6, 1, WIN, F8, false, true>(tk, tv, p, grid, stream, slot0 + 3);
                case 12: return launch_decode_t<256, 12, 1, 4, 6, 3, WIN, F8, false>(tk, tv, p, grid, stream, slot0 + 9);
                case 3: return launch_decode_t<256, 3, 2, 4, 6, 1, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 11);
                case 5: return launch_decode_t<256, 5, 2, 4, 6, 1, WIN, F8, false>(tk, tv, p, grid, stream, slot0 + 12);
                case 8: return launch_decode_t<256, 8, 1, 4, 6, 2, WIN, F8, false>(tk, tv, p, grid, stream, slot0 + 13);
                case 16: return launch_decode_t<256, 16, 1, 3, 8, 4, WIN, F8, false>(tk, tv, p, grid, stream, slot0 + 14);
            }
        } else if (head_dim == 128) {
            switch (group) {
                case 1: return launch_decode_t<128, 1, 1, 12, 4, 1, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 4);
                case 2: return launch_decode_t<128, 2, 1, 12, 4, 1, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 5);
                case 4: return launch_decode_t<128, 4, 2, 6, 8, 1, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 6);
                case 6: return launch_decode_t<128, 6, 2, 6, 8, 1, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 7);
                case 8: return launch_decode_t<128, 8, 1, 8, 6, 2, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 8);
                case 12: return launch_decode_t<128, 12, 1, 6, 8, 3, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 10);
                case 3: return launch_decode_t<128, 3, 2, 6, 8, 1, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 15);
                case 5: return launch_decode_t<128, 5, 2, 6, 8, 1, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 16);
                case 16: return launch_decode_t<128, 16, 1, 4, 12, 4, WIN, F8, true>(tk, tv, p, grid, stream, slot0 + 17);
            }
        }
        return cudaErrorInvalidValue;
    }
    if (head_dim == 256) {
        switch (group) {
            case 1: return launch_decode_t<256, 1, 1, 6, 2, 1, WIN, false, false>(tk, tv, p, grid, stream, slot0 + 0);
            case 2: return launch_decode_t<256, 2, 1, 6, 2, 1, WIN, false, false>(tk, tv, p, grid, stream, slot0 + 1);
            case 4: return launch_decode_t<256, 4, 2, 4, 3, 1, WIN, false, false, true>(tk, tv, p, grid, stream, slot0 + 2);
            case 6: return launch_decode_t<256, 6, 2, 4, 3, 1, WIN, false, false, true>(tk, tv, p, grid, stream, slot0 + 3);
            case 12: return launch_decode_t<256, 12, 1, 4, 3, 2, WIN, false, false, true>(tk, tv, p, grid, stream, slot0 + 9);
            case 3: return launch_decode_t<256, 3, 2, 4, 3, 1, WIN, false, false>(tk, tv, p, grid, stream, slot0 + 11);
            case 5: return launch_decode_t<256, 5, 2, 4, 3, 1, WIN, false, false>(tk, tv, p, grid, stream, slot0 + 12);
            case 8: return launch_decode_t<256, 8, 2, 4, 3, 1, WIN, false, false, true>(tk, tv, p, grid, stream, slot0 + 13);
            case 16: return launch_decode_t<256, 16, 1, 4, 3, 2, WIN, false, false, true>(tk, tv, p, grid, stream, slot0 + 14);
        }
    } else if (head_dim == 128) {
        switch (group) {
            case 1: return launch_decode_t<128, 1, 1, 12, 2, 1, WIN, false, true>(tk, tv, p, grid, stream, slot0 + 4);
            case 2: return launch_decode_t<128, 2, 1, 12, 2, 1, WIN, false, true>(tk, tv, p, grid, stream, slot0 + 5);
            case 4: return launch_decode_t<128, 4, 2, 6, 4, 1, WIN, false, true>(tk, tv, p, grid, stream, slot0 + 6);
            case 6: return launch_decode_t<128, 6, 2, 6, 4, 1, WIN, false, true>(tk, tv, p, grid, stream, slot0 + 7);
            case 8: return launch_decode_t<128, 8, 1, 8, 3, 2, WIN, false, true>(tk, tv, p, grid, stream, slot0 + 8);
            case 12: return launch_decode_t<128, 12, 1, 6, 4, 3, WIN, false, true>(tk, tv, p, grid, stream, slot0 + 10);
            case 3: return launch_decode_t<128, 3, 2, 6, 4, 1, WIN, false, true>(tk, tv, p, grid, stream, slot0 + 15);
            case 5: return launch_decode_t<128, 5, 2, 6, 4, 1, WIN, false, true>(tk, tv, p, grid, stream, slot0 + 16);
            case 16: return launch_decode_t<128, 16, 1, 4, 6, 4, WIN, false, true>(tk, tv, p, grid, stream, slot0 + 17);
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
