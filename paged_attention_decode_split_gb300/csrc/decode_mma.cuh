// decode_mma.cuh -- split-KV paged-attention decode with both products on the
// tensor cores (warp-level mma.sync m16n8k16, fp32 accumulation).
//
// What it computes is the decode of decode_split.cuh ("DCU page832 attention",
// Sec.5 and Sec.7; the split-KV fix of "Hybrid SSM decode rate on dual Radeon
// under vLLM"): for one (sequence, KV head) split of whole 16-token chunks,
// the online softmax of the G query heads of the group over the split's keys,
// written as the split's normalised output with its max logit and exponential
// sum (or as the final output when the plan has one split); the partition
// reduce of decode_split.cuh merges the splits.
//
// Why tensor cores here: on the CUDA cores the G-head dot products, the bf16
// widening and the cross-lane sums cost about 1,900 warp instructions per
// 16-token chunk, which bounds the kernel below the HBM rate.  As two small
// MMAs per chunk the same work is about 110 instructions.
//
// Layout on sm_103a:
//  * A 16-token chunk of one KV head arrives by one 5-D TMA copy per tensor
//    with the 128-byte swizzle: [ROW_BYTES / 128 column blocks][16 tokens]
//    [128 B], 16-byte unit u of token t stored at unit u ^ (t % 8).  The eight
//    16-byte rows that ldmatrix reads for one 8x8 matrix then always fall in
//    eight different bank groups.
//  * Scores, transposed: S^T [16 tokens x 8 heads] = K [16 x D] . Q^T [D x 8]:
//    keys on M, the group's heads (padded to 8, or 16 as two n-tiles) on N,
//    one m16n8k16 per 16 dims.  K comes from shared memory through ldmatrix;
//    Q^T stays in registers as B fragments for the whole split.  A lane ends
//    up with the scores of tokens r and r + 8 (r = lane / 4) for heads 2c and
//    2c + 1 (c = lane % 4).
//  * Online softmax on those fragments: the scale, the lazy max test (a warp
//    vote; a head's reference max is raised only when the chunk max exceeds
//    it by more than 2^8) and the exponential sums stay in the lane; only a
//    raise reduces across lanes.
//  * P.V, also transposed: O^T [D x 8] += V^T [D x 16] . P^T [16 x 8], d on M.
//    V^T comes from shared memory through ldmatrix.trans; P^T is the score
//    fragment itself, transposed in registers (movmatrix), carried as a bf16
//    head plus a bf16 residual (two MMAs) so P keeps about 16 significant
//    bits.  A lane's accumulator fragment holds the same two heads as its
//    score fragment, so a rescale touches only the lane's own registers.
//  * DS warps may share a chunk: each forms the whole score fragment (the
//    softmax needs every token of every head) and takes 1/DS of the d range
//    in P.V.
//  * fp8 e4m3 cache: ldmatrix moves the codes as 16-bit pairs, cvt widens
//    them to f16 (exact: every e4m3 value is an f16 value) and the MMAs run in
//    f16.  For K, a lane's four codes of one row are four consecutive dims,
//    so the k index of the score MMA walks the dims in a permuted order that
//    the Q fragments follow.  For V, the transposed load gives a lane two
//    codes of each of two tokens; one byte permute makes a (token, token)
//    pair per dim, and the output rows of a tile are the dims in the order
//    2r, 2r + 1.  q enters as f16 scaled by a power of two per head so that
//    its largest element lies in [2^14, 2^15); the inverse power joins the
//    softmax scale, so every finite bf16 q keeps its bits up to the f16
//    subnormal range 2^-38 below its largest element.
#pragma once

#include <type_traits>

#include "decode_split.cuh"

namespace pa {

namespace mm {

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// 8x8 b16 matrix transposed across the warp (same fragment layout in and out).
__device__ __forceinline__ uint32_t movt(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// D += A B for one m16n8k16 tile; A row-major 16x16, B column-major 16x8.
template <bool F16>
__device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
    if constexpr (F16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four e4m3 codes (bytes 0..3 of w) -> f16 pairs (bytes 0, 1) and (bytes 2, 3).
__device__ __forceinline__ void e4m3x4_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(a), "r"(sel));
    return d;
}

}  // namespace mm

// D: head_dim.  NT: n-tiles of 8 heads (1 for G <= 8, 2 for G <= 16).  NST
// chunk streams, each owning SPS stages; DS warps per stream split the d
// range of P.V.  F8: fp8 e4m3 cache.
template <int D, int NT, int NST, int SPS, int DS, bool F8>
struct MmaCfg {
    static constexpr int KVB = F8 ? 1 : 2;
    static constexpr int ROW_BYTES = D * KVB;
    static constexpr int BLOCK_BYTES = kChunk * 128;  // one 128-byte column block of a chunk
    static constexpr int CHUNK_BYTES = ROW_BYTES / 128 * BLOCK_BYTES;
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;  // K chunk, then V chunk
    static constexpr int NS = NST * SPS;
    static constexpr int NWC = NST * DS;                 // consumer warps
    static constexpr int THREADS = (NWC + 1) * 32;       // + the producer warp
    static constexpr int KS = D / 16;                    // k16 steps of the score product
    static constexpr int MTW = D / 16 / DS;              // m16 tiles of d per warp in P.V
    static constexpr int HS = D + 4;                     // merge row stride in floats (bank spread)
    static constexpr int GMAX = 8 * NT;
    static constexpr int STAGES_BYTES = NS * STAGE_BYTES;
    static constexpr int OFF_BAR = STAGES_BYTES;
    static constexpr int OFF_FLAGS = OFF_BAR + 2 * NS * 8;
    static constexpr int OFF_ML = OFF_FLAGS + 16;             // [NST][GMAX] (m, l)
    static constexpr int OFF_W = OFF_ML + NST * GMAX * 8;     // [NST][GMAX] merge weights
    static constexpr int OFF_PT = OFF_W + NST * GMAX * 4;
    static constexpr int SMEM_BYTES = OFF_PT + kPageTab * 4 + 1024;  // + slack to align the base to 1 KiB
    static_assert(D == 128 || D == 256, "head_dim 128 or 256");
    static_assert(NT == 1 || NT == 2, "up to 16 heads per KV head");
    static_assert((D / 16) % DS == 0 && (!F8 || MTW % 2 == 0), "whole (pairs of) m16 tiles per warp");
    static_assert(NST * GMAX * HS * 4 <= STAGES_BYTES, "the CTA merge reuses the stage buffers");
    static_assert(NST <= 32, "one producer lane per stream at most");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// The fused append (pa_paged_attention_decode_append): the CTA whose split
// holds token L - 1 of its sequence writes that token's K and V rows of its
// KV head into the cache slot the block table gives for it, exactly as
// reshape_and_cache would (bf16 copied; fp8 quantised like
// reshape_and_cache_fp8), then makes the write visible to the copy engine
// before the chunk that holds it is copied.  Called by the producer warp.
template <int D, bool F8>
__device__ __forceinline__ void append_new_row(const DecodeParams &p, int b, int kvh, int L, int c_begin, int n_my,
                                               const int32_t *page_tab, int lp_first) {
    const int t = L - 1;
    if (t < 0 || t / kChunk < c_begin || t / kChunk >= c_begin + n_my) return;  // not this split's token
    const int lane = threadIdx.x & 31;
    const int lp = t / p.block_size;
    const int page = page_tab ? page_tab[lp - lp_first] : p.block_table[(size_t)b * p.max_pages_per_seq + lp];
    if (page >= 0 && (int64_t)page < p.num_pages) {  // (a bad page is flagged when its chunk is copied)
        const int hkv = gridDim.y;
        const size_t slot = (size_t)page * p.block_size + (t - lp * p.block_size);
        const size_t row = slot * hkv + kvh;  // [P, BS, Hkv, D]
        const uint4 *ks = reinterpret_cast<const uint4 *>(p.k_new + ((size_t)b * hkv + kvh) * D);
        const uint4 *vs = reinterpret_cast<const uint4 *>(p.v_new + ((size_t)b * hkv + kvh) * D);
        for (int j = lane; j < D / 8; j += 32) {  // 8 elements per lane and step
            const uint4 kw = ks[j], vw = vs[j];
            if constexpr (F8) {
                reinterpret_cast<uint2 *>(p.k_cache + row * D)[j] = e4m3x8_div(kw, p.k_scale[kvh]);
                reinterpret_cast<uint2 *>(p.v_cache + row * D)[j] = e4m3x8_div(vw, p.v_scale[kvh]);
            } else {
                reinterpret_cast<uint4 *>(p.k_cache + row * D * 2)[j] = kw;
                reinterpret_cast<uint4 *>(p.v_cache + row * D * 2)[j] = vw;
            }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");  // generic-proxy writes before the TMA reads
    }
    __syncwarp();
}

// PF: chunks of old context a CTA prefetches into L2, beyond its stages, ahead
// of the dependency wait (PA_FLAG_EARLY_KV_READ).
template <int D, int G, int NT, int NST, int SPS, int DS, bool WIN, bool F8, bool LP, int PF = 0>
__global__ void __launch_bounds__((NST * DS + 1) * 32, 1)
    pa_decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const DecodeParams p) {
    using C = MmaCfg<D, NT, NST, SPS, DS, F8>;
    constexpr int NS = C::NS, NWC = C::NWC, KS = C::KS, MTW = C::MTW, HS = C::HS, GMAX = C::GMAX;
    static_assert(G <= GMAX && G > GMAX - 8, "n-tiles match the group");
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + NS;
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::OFF_FLAGS);  // [0] abort, [1] bad page
    float2 *merge_ml = reinterpret_cast<float2 *>(smem + C::OFF_ML);
    float *merge_w = reinterpret_cast<float *>(smem + C::OFF_W);
    int32_t *page_tab = reinterpret_cast<int32_t *>(smem + C::OFF_PT);

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq0 = kvh * G;

    // Programmatic dependent launch: as in the CUDA-core decode kernel, every
    // global access waits for the work before this call unless early_kv lets
    // the block table, seq_lens and the K/V chunks wholly before the new row
    // go first.
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], DS);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    if (warp == NWC && lane == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (!p.early_kv) pdl_wait_primary();

    int L = p.seq_lens[b];
    int c_begin = split * p.chunks_per_split;
    if constexpr (WIN) {
        if (L > p.window && L <= p.max_seq_len) c_begin += (L - p.window) / kChunk;
    }
    const int32_t *bt = p.block_table + (size_t)b * p.max_pages_per_seq;
    const int lp_first = (c_begin * kChunk) / p.block_size;
    const int lp_last = min(((c_begin + p.chunks_per_split) * kChunk - 1) / p.block_size, p.max_pages_per_seq - 1);
    const int n_pt = lp_last - lp_first + 1;
    const bool staged = n_pt <= kPageTab;
    if (staged)
        for (int j = threadIdx.x; j < n_pt; j += C::THREADS) page_tab[j] = bt[lp_first + j];
    if (L < 0 || L > p.max_seq_len) {
        if (threadIdx.x == 0 && split == 0 && kvh == 0) set_status(p.status, PA_DEV_BAD_SEQLEN);
        L = 0;
    }
    const int n_chunks = (L + kChunk - 1) / kChunk;
    const int n_my = min(n_chunks - c_begin, p.chunks_per_split);
    if (n_my <= 0) {
        // no key of this sequence in this split: the record says so (m = -inf,
        // l = 0); an unsplit call owns its output rows and zeroes them
        if (p.early_kv) pdl_wait_primary();
        if (p.num_splits == 1) {
            for (int idx = threadIdx.x; idx < G * D; idx += C::THREADS)
                store_out(p.out, ((size_t)b * p.num_q_heads + hq0) * D + idx, 0.f, p.out_bf16);
        } else if (threadIdx.x < G) {
            p.part_ml[((size_t)b * p.num_q_heads + hq0 + threadIdx.x) * p.num_splits + split] =
                make_float2(-INFINITY, 0.f);
        }
        return;
    }
    __syncthreads();  // barrier initialisation and the page table are visible to every thread

    const int stream = warp / DS, ds = warp % DS;
    const int r = lane >> 2, c = lane & 3;
    float m_run[NT][2], l_run[NT][2];
    float oacc[MTW][NT][4];

    if (warp == NWC) {
        // ---------------- producer: PL lanes issue the copies ----------------
        // Lane c0 < PL serves streams c0, c0 + PL, ...  A lane polls its
        // streams' next stages without blocking and issues as soon as one is
        // free; within a stream, chunks and stage phases go strictly in order.
        constexpr int PL = LP ? NST : 1, SPL = NST / PL;
        static_assert(NST % PL == 0, "streams spread evenly over the producer lanes");
        const unsigned mask = PL == 32 ? 0xffffffffu : (1u << PL) - 1u;
        auto any = [&](bool v) {  // over the producer lanes
            if constexpr (PL == 1)
                return v;
            else
                return __any_sync(mask, v);
        };
        const uint64_t policy = l2_policy_evict_first();
        auto issue = [&](int cs, int k) {  // chunk cs + k * NST into stream cs's stage k % SPS
            const int i = cs + k * NST, s = cs * SPS + k % SPS;
            const int t0 = (c_begin + i) * kChunk;
            const int lp = t0 / p.block_size;
            const int page = staged ? page_tab[lp - lp_first] : bt[lp];
            if (page < 0 || (int64_t)page >= p.num_pages) {
                flags[1] = 1;  // the copy below reads zeros (box outside the tensor)
                set_status(p.status, PA_DEV_BAD_PAGE);
            }
            const int off = t0 - lp * p.block_size;
            uint8_t *st = smem + s * C::STAGE_BYTES;
            mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
            tma_load_5d(st, &tm_k, &full[s], 0, off, 0, kvh, page, policy);
            tma_load_5d(st + C::CHUNK_BYTES, &tm_v, &full[s], 0, off, 0, kvh, page, policy);
        };
        int next[SPL];
        int remaining = PL == 1 ? n_my : 0;
#pragma unroll
        for (int j = 0; j < SPL; ++j) {
            next[j] = 0;
            if constexpr (PL > 1) remaining += max(0, (n_my - lane - j * PL + NST - 1) / NST);  // chunks c, c + NST, ...
        }
        if (p.early_kv) {
            // First use of every stage: the chunks i < n_pre (those that end
            // before the new row, token L - 1) go out before the dependency
            // wait; chunk i is stream i % NST's (i / NST)-th, and n_pre <= NS,
            // so none of them waits for a free stage.
            const int n_old = (L - 1) / kChunk - c_begin;  // chunks that end before the new row
            const int n_pre = max(0, min(min(NS, n_my), n_old));
            if (lane < PL) {
#pragma unroll 1
                for (int i = lane; i < n_pre; i += PL) issue(i % NST, i / NST);
            }
            // The next chunks of old context go to L2 ahead of the wait as
            // well, so the copies keep streaming while the work before this
            // call finishes; the consumers then find them in L2.
            const int n_l2 = max(0, min(min(n_pre + PF, n_my), n_old));
            for (int i = n_pre + lane; i < n_l2; i += 32) {
                const int t0 = (c_begin + i) * kChunk;
                const int lp = t0 / p.block_size;
                const int page = staged ? page_tab[lp - lp_first] : bt[lp];
                if (page >= 0 && (int64_t)page < p.num_pages) {  // (a bad page is flagged when the chunk is copied)
                    const int off = t0 - lp * p.block_size;
                    tma_prefetch_l2_5d(&tm_k, 0, off, 0, kvh, page);
                    tma_prefetch_l2_5d(&tm_v, 0, off, 0, kvh, page);
                }
            }
#pragma unroll
            for (int j = 0; j < SPL; ++j) {
                const int cs = lane + j * PL;
                next[j] = max(0, (n_pre - cs + NST - 1) / NST);
                remaining -= next[j];
            }
            pdl_wait_primary();
        }
        // Fused append: the new token's rows go into its cache slot before the
        // chunk that holds them is copied (the whole warp; after the wait, as
        // the rows may come from the work before this call).
        if (p.k_new != nullptr) append_new_row<D, F8>(p, b, kvh, L, c_begin, n_my, staged ? page_tab : nullptr, lp_first);
        if (lane < PL) {
            uint32_t idle = 0;
            bool gave_up = false;
            while (any(remaining > 0)) {
                bool progress = false;
#pragma unroll
                for (int j = 0; j < SPL; ++j) {
                    const int cs = lane + j * PL, k = next[j], i = cs + k * NST;
                    if (i >= n_my) continue;
                    const int s = cs * SPS + k % SPS, ph = k / SPS;
                    if (ph > 0 && !mbar_test_wait(&empty[s], (ph - 1) & 1)) continue;
                    issue(cs, k);
                    next[j] = k + 1;
                    --remaining;
                    progress = true;
                }
                if (any(progress)) {
                    idle = 0;
                } else if (++idle > kWaitPollLimit || any(flags[0] != 0)) {
                    gave_up = true;
                    break;
                }
            }
            if (gave_up || flags[0]) {
                // giving up: let the copies in flight land before the CTA ends
                if (lane == 0) flags[0] = 1;
#pragma unroll
                for (int j = 0; j < SPL; ++j) {
                    const int cs = lane + j * PL;
                    for (int k = max(0, next[j] - SPS); k < next[j]; ++k) {
                        uint64_t *bar = &full[cs * SPS + k % SPS];
                        for (uint32_t n = 0; n < kWaitPollLimit && !mbar_try_wait(bar, (k / SPS) & 1); ++n) {
                        }
                    }
                }
                if (lane == 0) set_status(p.status, PA_DEV_TIMEOUT);
            }
        }
        // The producer leaves: its copies have all landed (the consumers wait
        // for every chunk, or it waited for its own copies before giving up).
        // A bad page index reaches the consumers through the full barrier of
        // that chunk, which orders the flag write before their wait returns.
        return;
    }

    // ---------------- consumers ----------------
    // Q^T as B fragments: n-tile nt, k-step ks -> {b0b1, b2b3} for head
    // 8 nt + r.  bf16: dims 16 ks + 2c (+1) and 16 ks + 8 + 2c (+1).  fp8 (the
    // permuted k order): dims 16 ks + 4c (+1) and 16 ks + 4c + 2 (+3), in f16.
    uint32_t qf[NT][KS][2];
    float qsc[NT][2];  // multiplier of the raw scores of heads 8 nt + 2c + j (log2 units)
    if (p.early_kv) pdl_wait_primary();  // q may come from the work before this call
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int h = nt * 8 + r;
        const bool live = h < G;
        const __nv_bfloat16 *qrow = p.q + ((size_t)b * p.num_q_heads + hq0 + (live ? h : 0)) * D;
        float qmul = 1.f;
        if constexpr (F8) {
            // the largest |q| of the head, over the 4 lanes holding it, sets
            // the power of two the head enters f16 with (f16_prescale)
            uint32_t amax = 0;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint2 w = live ? *reinterpret_cast<const uint2 *>(qrow + 16 * ks + 4 * c) : make_uint2(0u, 0u);
                amax = max(amax, max(bf16x2_absmax(w.x), bf16x2_absmax(w.y)));
            }
            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            qmul = f16_prescale(amax);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint2 w = live ? *reinterpret_cast<const uint2 *>(qrow + 16 * ks + 4 * c) : make_uint2(0u, 0u);
                qf[nt][ks][0] = bf16x2_to_f16x2_scaled(w.x, qmul);
                qf[nt][ks][1] = bf16x2_to_f16x2_scaled(w.y, qmul);
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                qf[nt][ks][0] = live ? *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 2 * c) : 0u;
                qf[nt][ks][1] = live ? *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 8 + 2 * c) : 0u;
            }
        }
        // lane 4 h' holds head h''s factor; this lane's score columns are heads 2c, 2c + 1
        const float base = F8 ? p.scale_log2 * p.k_scale[kvh] : p.scale_log2;
        const float inv = F8 ? 1.f / qmul : 1.f;  // a power of two: exact
        const float mine = base * inv;
        qsc[nt][0] = __shfl_sync(0xffffffffu, mine, 8 * c);
        qsc[nt][1] = __shfl_sync(0xffffffffu, mine, 8 * c + 4);
        m_run[nt][0] = m_run[nt][1] = -INFINITY;
        l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) oacc[mt][nt][i] = 0.f;
    }

    // ldmatrix row addresses (byte offsets inside a chunk), for the 16-byte
    // unit pair starting at an even unit 2j of a column block: lanes 8m..8m+7
    // give the rows of matrix m.
    //  pattern A (K, and fp8 V): m = 0: tokens 0-7 / unit 2j, 1: tokens 8-15 /
    //    2j, 2: tokens 0-7 / 2j + 1, 3: tokens 8-15 / 2j + 1
    //  pattern B (bf16 V^T): m = 0: tokens 0-7 / 2j, 1: tokens 0-7 / 2j + 1,
    //    2: tokens 8-15 / 2j, 3: tokens 8-15 / 2j + 1
    uint32_t offA[4], offB[4];
    {
        const int x = lane & 7;
        const int tA = x + 8 * ((lane >> 3) & 1), uA = lane >> 4;
        const int tB = x + 8 * (lane >> 4), uB = (lane >> 3) & 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            offA[j] = tA * 128 + (((2 * j + uA) ^ x) << 4);
            offB[j] = tB * 128 + (((2 * j + uB) ^ x) << 4);
        }
    }
    const uint32_t smem_base = smem_addr(smem);

    for (int i = stream, k = 0; i < n_my; i += NST, ++k) {
        const int s = stream * SPS + k % SPS;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (k / SPS) & 1, &flags[0]))) {
            flags[0] = 1;
            break;
        }
        const uint32_t kb = smem_base + s * C::STAGE_BYTES, vb = kb + C::CHUNK_BYTES;
        const int t_chunk = (c_begin + i) * kChunk;
        const int nv = min(kChunk, L - t_chunk);                     // valid rows [lead, nv)
        const int lead = WIN ? max(0, L - p.window - t_chunk) : 0;
        const bool partial = nv < kChunk || lead > 0;                // warp-uniform

        // ---- S^T = K Q^T, two accumulators per n-tile (even / odd k-steps) ----
        float sa[NT][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int q = 0; q < 4; ++q) sa[nt][u][q] = 0.f;
        if constexpr (!F8) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {  // units 2 ks, 2 ks + 1
                uint32_t a[4];
                mm::ldsm_x4(a, kb + (ks >> 2) * C::BLOCK_BYTES + offA[ks & 3]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mm::mma<false>(sa[nt][ks & 1], a[0], a[1], a[2], a[3], qf[nt][ks][0], qf[nt][ks][1]);
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < KS; ks += 2) {  // unit ks is k-step ks; one load covers two
                uint32_t w[4];
                mm::ldsm_x4(w, kb + (ks >> 3) * C::BLOCK_BYTES + offA[(ks & 7) >> 1]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    uint32_t a0, a2, a4, a6;
                    mm::e4m3x4_f16(w[2 * u], a0, a4);      // row r
                    mm::e4m3x4_f16(w[2 * u + 1], a2, a6);  // row r + 8
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mm::mma<true>(sa[nt][u], a0, a2, a4, a6, qf[nt][ks + u][0], qf[nt][ks + u][1]);
                }
            }
        }

        // ---- online softmax on the fragments (log2 units) ----
        float x[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) x[nt][q] = (sa[nt][0][q] + sa[nt][1][q]) * qsc[nt][q & 1];
        if (partial) {
            const bool v0 = r >= lead && r < nv, v1 = r + 8 >= lead && r + 8 < nv;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (!v0) x[nt][0] = x[nt][1] = -INFINITY;
                if (!v1) x[nt][2] = x[nt][3] = -INFINITY;
            }
        }
        bool up = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) up |= x[nt][q] > m_run[nt][q & 1] + kLazyLog2;
        if (__any_sync(0xffffffffu, up)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float cm = fmaxf(x[nt][j], x[nt][j + 2]);
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
                    if (cm > m_run[nt][j] + kLazyLog2) {
                        const float alpha = fast_exp2(m_run[nt][j] - cm);  // 0 on the first chunk
                        m_run[nt][j] = cm;
                        l_run[nt][j] *= alpha;
#pragma unroll
                        for (int mt = 0; mt < MTW; ++mt) {
                            oacc[mt][nt][j] *= alpha;
                            oacc[mt][nt][j + 2] *= alpha;
                        }
                    }
                }
        }
        // P^T fragments: head + residual, each transposed in registers
        uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float pr[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) pr[q] = fast_exp2(x[nt][q] - m_run[nt][q & 1]);  // 0 for masked rows
            l_run[nt][0] += pr[0] + pr[2];
            l_run[nt][1] += pr[1] + pr[3];
            uint32_t h01, h23, r01, r23;
            if constexpr (F8) {
                split_f16(pr[0], pr[1], h01, r01);
                split_f16(pr[2], pr[3], h23, r23);
            } else {
                split_bf16(pr[0], pr[1], h01, r01);
                split_bf16(pr[2], pr[3], h23, r23);
            }
            bh[nt][0] = mm::movt(h01);
            bh[nt][1] = mm::movt(h23);
            bl[nt][0] = mm::movt(r01);
            bl[nt][1] = mm::movt(r23);
        }

        // ---- O^T += V^T P^T over this warp's m16 tiles of d ----
        // A lane's V^T fragment holds tokens 2c, 2c + 1 (regs 0, 1) and 8 + 2c,
        // 9 + 2c (regs 2, 3); rows past the sequence end may hold anything
        // (NaN included) and are zeroed in a partial chunk.
        // Over an fp8 cache, full chunks (all but a sequence's last and a
        // window's first) skip the masking: two copies of the product, chosen
        // once per chunk (fp8 32K call 16.55 -> 15.24 us; bf16 measured 1 %
        // slower that way and keeps the single masked loop).
        auto pv = [&](auto masked) {
            constexpr bool MASK = decltype(masked)::value;
            uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
            if (MASK && partial) {
                mlo = (2 * c < nv ? 0x0000ffffu : 0u) | (2 * c + 1 < nv ? 0xffff0000u : 0u);
                mhi = (2 * c + 8 < nv ? 0x0000ffffu : 0u) | (2 * c + 9 < nv ? 0xffff0000u : 0u);
            }
            if constexpr (!F8) {
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) {
                    const int gt = ds * MTW + mt;  // global m16 tile: dims 16 gt .. 16 gt + 15 = units 2 gt, 2 gt + 1
                    uint32_t a[4];
                    mm::ldsm_x4_t(a, vb + (gt >> 2) * C::BLOCK_BYTES + offB[gt & 3]);
                    if constexpr (MASK) {
                        a[0] &= mlo;
                        a[1] &= mlo;
                        a[2] &= mhi;
                        a[3] &= mhi;
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mm::mma<false>(oacc[mt][nt], a[0], a[1], a[2], a[3], bh[nt][0], bh[nt][1]);
                        mm::mma<false>(oacc[mt][nt], a[0], a[1], a[2], a[3], bl[nt][0], bl[nt][1]);
                    }
                }
            } else {
#pragma unroll
                for (int mt = 0; mt < MTW; mt += 2) {
                    const int gt = ds * MTW + mt;  // unit gt = m16 tile gt (dims 16 gt ..), and gt + 1
                    uint32_t w[4];
                    mm::ldsm_x4_t(w, vb + (gt >> 3) * C::BLOCK_BYTES + offA[(gt & 7) >> 1]);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        uint32_t a0, a2, a4, a6;
                        mm::e4m3x4_f16(mm::prmt(w[2 * u], 0x3120u), a0, a2);      // tokens 2c, 2c+1: dims 2r, 2r+1
                        mm::e4m3x4_f16(mm::prmt(w[2 * u + 1], 0x3120u), a4, a6);  // tokens 8+2c, 9+2c
                        if constexpr (MASK) {
                            a0 &= mlo;
                            a2 &= mlo;
                            a4 &= mhi;
                            a6 &= mhi;
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mm::mma<true>(oacc[mt + u][nt], a0, a2, a4, a6, bh[nt][0], bh[nt][1]);
                            mm::mma<true>(oacc[mt + u][nt], a0, a2, a4, a6, bl[nt][0], bl[nt][1]);
                        }
                    }
                }
            }
        };
        if (!F8 || partial)
            pv(std::true_type{});
        else
            pv(std::false_type{});
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    // exponential sums: a lane holds tokens r and r + 8; sum over r
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float l = l_run[nt][j];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            l_run[nt][j] = l;
        }

    // ---- CTA merge of the streams' states (log-sum-exp weights) ----
    named_bar_sync(1, NWC * 32);  // every chunk is consumed: the stages become the merge area
    const bool aborted = flags[0] != 0;
    const bool poisoned = aborted || flags[1] != 0;
    float *macc = reinterpret_cast<float *>(smem);  // [NST][G][HS], unnormalised sums
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt) {
        const int gt = ds * MTW + mt;
        const int d0 = F8 ? 16 * gt + 2 * r : 16 * gt + r;  // accumulator row r
        const int d1 = F8 ? d0 + 1 : d0 + 8;                // accumulator row r + 8
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int h = nt * 8 + 2 * c + j;
                if (h < G) {
                    float *row = macc + (stream * G + h) * HS;
                    row[d0] = oacc[mt][nt][j];
                    row[d1] = oacc[mt][nt][j + 2];
                }
            }
    }
    if (ds == 0 && r == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int h = nt * 8 + 2 * c + j;
                if (h < G) merge_ml[stream * GMAX + h] = make_float2(m_run[nt][j], l_run[nt][j]);
            }
    }
    named_bar_sync(1, NWC * 32);
    if (threadIdx.x < G) {
        const int h = threadIdx.x;
        float M = -INFINITY;
        for (int st = 0; st < NST; ++st) M = fmaxf(M, merge_ml[st * GMAX + h].x);
        float lsum = 0.f;
        for (int st = 0; st < NST; ++st) {
            const float2 ml = merge_ml[st * GMAX + h];
            const float e = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;  // 0 for a stream without chunks
            merge_w[st * GMAX + h] = e;
            lsum = fmaf(ml.y, e, lsum);
        }
        const bool zero = poisoned || !(lsum > 0.f);
        const float norm = zero ? 0.f : (F8 ? p.v_scale[kvh] / lsum : 1.f / lsum);
        for (int st = 0; st < NST; ++st) merge_w[st * GMAX + h] *= norm;
        if (p.num_splits > 1)
            p.part_ml[((size_t)b * p.num_q_heads + hq0 + h) * p.num_splits + split] =
                make_float2(M, poisoned ? -1.f : lsum);
    }
    named_bar_sync(1, NWC * 32);
    for (int idx = threadIdx.x; idx < G * D / 4; idx += NWC * 32) {
        const int h = (4 * idx) / D, d = 4 * idx - h * D;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int st = 0; st < NST; ++st) {
            const float wg = merge_w[st * GMAX + h];
            const float4 v = *reinterpret_cast<const float4 *>(macc + (st * G + h) * HS + d);
            o.x = fmaf(v.x, wg, o.x);
            o.y = fmaf(v.y, wg, o.y);
            o.z = fmaf(v.z, wg, o.z);
            o.w = fmaf(v.w, wg, o.w);
        }
        const size_t row = (size_t)b * p.num_q_heads + hq0 + h;
        if (p.num_splits == 1) {
            store_out(p.out, row * D + d, o.x, p.out_bf16);
            store_out(p.out, row * D + d + 1, o.y, p.out_bf16);
            store_out(p.out, row * D + d + 2, o.z, p.out_bf16);
            store_out(p.out, row * D + d + 3, o.w, p.out_bf16);
        } else {
            *reinterpret_cast<float4 *>(p.part_o + (row * p.num_splits + split) * D + d) = o;
        }
    }
}

}  // namespace pa
