// decode_split.cuh -- split-KV paged-attention decode on the CUDA cores.
//
// What it computes ("DCU page832 attention", Sec.5 and Sec.7; "Hybrid SSM
// decode rate on dual Radeon under vLLM", the split-KV fix): for one query row
// per sequence, out = softmax(scale * q K^T) V over the sequence's cached
// tokens, K/V rows found through the block table.  The context of every
// (sequence, KV head) is cut into splits of whole 16-token chunks; each split
// is one CTA, so batch 1 with 4 KV heads still spreads over every SM.  A CTA
// writes its split's normalised output with its max logit and exponential sum;
// pa_split_reduce_kernel merges the splits (log-sum-exp weights).
//
// Design on sm_103a:
//  * Unit of transfer: a 16-token chunk of one KV head, [16, D] bf16 of K and
//    the same of V, fetched by one 4-D TMA copy each from the
//    [pages, BS, Hkv, D] cache.  16 divides 784 = 49 x 16, 832 and 16, so a
//    chunk never straddles a page and the 16-token tail of a 784-token page
//    (784 = 12 x 64 + 16) is just the 49th chunk of the page: no masks inside
//    a page, and the split's block-table entries are staged in shared memory
//    once (the page-contiguous walk of Sec.7 reads the table once per page).  Only the last chunk of a sequence
//    can be partial; its rows past the end are masked (scores) and skipped (PV).
//  * NST chunk streams take chunks round-robin, each owning SPS of the NS
//    stages; one lane of the producer warp (or one lane per stream) issues
//    the copies and refills a stage as soon as its stream frees it.  A chunk is shared by TS warps that split
//    its 16 tokens (8 each when TS = 2); every warp keeps its own online
//    softmax state over the tokens it sees, and the CTA merges the states.
//  * Every warp handles all G query heads of the group, so each K/V element
//    is read from shared memory and widened to fp32 once per CTA and used by
//    the G heads (GQA reuse).  A lane owns E = D/32 consecutive elements of
//    d: q (pre-scaled to log2 units) and the output accumulators of the G
//    heads stay in registers.  Arithmetic runs on packed fp32 pairs (FFMA2).
//  * Scores: per micro-batch of 8 tokens a lane forms 8 x G partial dot
//    products over its d slice, and a transposing butterfly sums them across
//    the 32 lanes.  Lane l computes token (slot XOR ((l >> 2) & 7)) in slot, so
//    at every halving step each lane keeps its low slots and sends its high
//    ones (no selects); afterwards lane l holds all scores of token
//    (l >> 2) & 7 of the micro-batch.
//  * Softmax is lazy: a head's reference max is raised (and its O and l
//    rescaled) only when the chunk max exceeds it by more than 2^8, so most
//    chunks skip the rescale.  Probabilities go through a per-warp shared
//    buffer as (p, p) pairs that every lane broadcast-reads for P.V.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kChunk = 16;    // tokens per TMA copy and per pipeline stage
constexpr int kPageTab = 512;  // block-table entries a CTA stages in shared memory
constexpr float kLazyLog2 = 8.f;  // a head's reference max is raised only when it grows by more than 2^8

struct DecodeParams {
    const __nv_bfloat16 *q;  // [B, Hq, D]
    const int32_t *block_table;
    const int32_t *seq_lens;
    void *out;            // [B, Hq, D], written when num_splits == 1
    float *part_o;        // [B, Hq, S, D]
    float2 *part_ml;      // [B, Hq, S]: (max logit in log2 units, exp sum; -1 = poisoned)
    int32_t *status;
    int64_t num_pages;
    int num_q_heads;
    int max_pages_per_seq;
    int max_seq_len;
    int block_size;
    int chunks_per_split;
    int num_splits;
    float scale_log2;     // scale * log2(e)
    int out_bf16;
    int early_kv;         // stream the context before the new row ahead of the dependency wait
    int window;           // 0: full attention; W > 0: only the last W keys
    const float *k_scale; // fp8 cache: [Hkv] dequantisation scales of K and V
    const float *v_scale;
};

// D: head_dim.  G: query heads per KV head.  TS x HG warps share one chunk,
// each taking 16 / TS of its tokens and G / HG of the heads (HG > 1 only
// for groups too wide for one warp's registers).  NST: chunk streams
// (consumer warps = TS * HG * NST).  SPS: stages owned by each stream (NS =
// NST * SPS in all).  KVB: bytes per cached element (2 bf16, 1 fp8 e4m3).
// PW: warps beside the consumers (1: the producer warp; 4: a producer
// warpgroup whose registers go to the consumers, see RB below).
//
// Stage ownership matters for correctness: an mbarrier wait tests the parity
// of a phase, so a waiter must never run two phases ahead of the barrier.
// Each stream therefore owns SPS stages and cycles through them in order; it
// has consumed every earlier phase of a stage before it waits on the next,
// and the producer waits on every phase of a stage's empty barrier in order.
template <int D, int G, int TS, int NST, int SPS, int HG, int KVB = 2, int PW = 1>
struct DecodeCfg {
    static constexpr int NS = NST * SPS;
    static constexpr int E = D / 32;
    static constexpr int MB = 2 / TS;                    // micro-batches of 8 tokens per warp and chunk
    static constexpr int GW = G / HG;                    // heads per warp
    static constexpr int WPC = TS * HG;                  // warps per chunk
    static constexpr int NWC = WPC * NST;                // consumer warps
    static constexpr int NWH = TS * NST;                 // warps holding a given head
    static constexpr int ROW_BYTES = D * KVB;
    static constexpr int CHUNK_BYTES = kChunk * ROW_BYTES;
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;  // K chunk, then V chunk
    static constexpr int GP2 = (GW + 1) & ~1;            // (p, p) pairs per P row (16-byte rows)
    static constexpr int STAGES_BYTES = NS * STAGE_BYTES;
    static constexpr int MERGE_BYTES = NWC * GW * D * 4;
    static constexpr int OFF_P = STAGES_BYTES;
    static constexpr int OFF_ML = OFF_P + NWC * 8 * MB * GP2 * 8;
    static constexpr int OFF_BAR = OFF_ML + NWC * GW * 12;  // (m, l) pairs, then the merge weights
    static constexpr int OFF_FLAGS = OFF_BAR + 2 * NS * 8;
    static constexpr int OFF_PT = OFF_FLAGS + 16;
    static constexpr int SMEM_BYTES = OFF_PT + kPageTab * 4 + 1024;  // + slack to align the base to 1 KiB
    static constexpr int THREADS = (NWC + PW) * 32;
    // register budgets with a producer warpgroup (PW = 4): the launch gives
    // every thread REG_LAUNCH registers; the producer warpgroup keeps
    // REG_PRODUCER and the consumer warpgroups take the rest
    static constexpr int REG_LAUNCH = (65536 / THREADS) & ~7;
    static constexpr int REG_PRODUCER = 40;
    static constexpr int REG_CONSUMER = ((REG_LAUNCH * THREADS - 128 * REG_PRODUCER) / (NWC * 32)) & ~7;
    static_assert(PW == 1 || (PW == 4 && NWC % 4 == 0 && REG_CONSUMER <= 256), "whole warpgroups");
    static_assert(D % 32 == 0 && (E == 8 || E == 4), "head_dim 256 or 128");
    static_assert(TS == 1 || TS == 2, "a chunk is consumed by one warp or split in token halves");
    static_assert(G % HG == 0, "heads split evenly over the head groups");
    static_assert(MERGE_BYTES <= STAGES_BYTES, "the CTA merge reuses the stage buffers");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// E consecutive bf16 of a row -> E/2 float pairs (element 2j in .x, 2j+1 in .y).
template <int E>
__device__ __forceinline__ void load_bf16_pairs(const uint8_t *src, float2 (&f)[E / 2]) {
    if constexpr (E == 8) {
        const uint4 w = *reinterpret_cast<const uint4 *>(src);
        f[0] = make_float2(bf16lo(w.x), bf16hi(w.x));
        f[1] = make_float2(bf16lo(w.y), bf16hi(w.y));
        f[2] = make_float2(bf16lo(w.z), bf16hi(w.z));
        f[3] = make_float2(bf16lo(w.w), bf16hi(w.w));
    } else {
        const uint2 w = *reinterpret_cast<const uint2 *>(src);
        f[0] = make_float2(bf16lo(w.x), bf16hi(w.x));
        f[1] = make_float2(bf16lo(w.y), bf16hi(w.y));
    }
}

// E consecutive e4m3 codes of a row -> E/2 float pairs (exact: every e4m3
// value is an f16 value, and every f16 value an fp32 one).
__device__ __forceinline__ void e4m3x4_to_float(uint32_t w, float2 &a, float2 &b) {
    uint32_t h0, h1;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h0), "=r"(h1)
        : "r"(w));
    a = __half22float2(*reinterpret_cast<const __half2 *>(&h0));
    b = __half22float2(*reinterpret_cast<const __half2 *>(&h1));
}

template <int E>
__device__ __forceinline__ void load_e4m3_pairs(const uint8_t *src, float2 (&f)[E / 2]) {
    if constexpr (E == 8) {
        const uint2 w = *reinterpret_cast<const uint2 *>(src);
        e4m3x4_to_float(w.x, f[0], f[1]);
        e4m3x4_to_float(w.y, f[2], f[3]);
    } else {
        e4m3x4_to_float(*reinterpret_cast<const uint32_t *>(src), f[0], f[1]);
    }
}

template <int E, bool F8>
__device__ __forceinline__ void load_kv_pairs(const uint8_t *src, float2 (&f)[E / 2]) {
    if constexpr (F8)
        load_e4m3_pairs<E>(src, f);
    else
        load_bf16_pairs<E>(src, f);
}

__device__ __forceinline__ void store_out(void *out, size_t idx, float v, int out_bf16) {
    if (out_bf16)
        reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float *>(out)[idx] = v;
}

// WIN: the sliding-window variant (a separate instantiation, so the full-
// attention kernel carries none of its bookkeeping).  F8: the cache holds fp8
// e4m3 codes with one scale per KV head for K and for V; the K scale is folded
// into q and the V scale into the merge weights, so the inner loops only
// widen codes instead of bf16 values.  LP: one producer lane per chunk stream
// (else one lane serves all streams).  RB: the producer is the first warp of
// a warpgroup of its own that lowers its register budget (setmaxnreg) so the
// consumer warpgroups run with more registers than an even split of the
// register file allows; its three other warps have no work.
template <int D, int G, int TS, int NST, int SPS, int HG, bool WIN, bool F8 = false, bool LP = false,
          bool RB = false>
__global__ void __launch_bounds__((TS * HG * NST + (RB ? 4 : 1)) * 32, 1)
    pa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const DecodeParams p) {
    using C = DecodeCfg<D, G, TS, NST, SPS, HG, F8 ? 1 : 2, RB ? 4 : 1>;
    constexpr int E = C::E, MB = C::MB, NWC = C::NWC, NS = C::NS, GW = C::GW, WPC = C::WPC, NWH = C::NWH;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    float2 *pbuf_all = reinterpret_cast<float2 *>(smem + C::OFF_P);
    float2 *merge_ml = reinterpret_cast<float2 *>(smem + C::OFF_ML);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + NS;
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::OFF_FLAGS);  // [0] abort, [1] bad page
    int32_t *page_tab = reinterpret_cast<int32_t *>(smem + C::OFF_PT);

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq0 = kvh * G;

    // Programmatic dependent launch: the reduce grid may be scheduled now, and
    // this grid's set-up overlaps the work before it in the stream (which may
    // be writing the cache).  By default every global access waits for that
    // work.  With early_kv, the block table, seq_lens and the K/V chunks that
    // lie wholly before the new row are read first; q, the new row, the
    // workspace and the output wait.  Every thread passes the wait before it
    // exits, so this grid completes only after the work before it.
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], WPC);
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

    // The pages this split may touch are staged in shared memory once, so the
    // producer resolves every chunk's page without a dependent global load.
    // Their range depends only on the split (entries past the sequence's end
    // are staged but never used), so these loads are in flight together with
    // the seq_lens load instead of after it.
    int L = p.seq_lens[b];
    // With a sliding window the splits cover chunks from the window's first
    // key s0 on (that start depends on the sequence length); without one
    // they start at 0 and the page-table loads need not wait for seq_lens.
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
        // Nothing of this sequence falls in this split: its record says "no
        // keys" (m = -inf, l = 0) so the reduce can read every split without
        // knowing the sequence length; an unsplit call owns its output rows
        // and zeroes them.
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

    // consumer warps: chunk stream, token half, head group
    const int stream = warp / WPC, wh = (warp % WPC) % TS, hg = (warp % WPC) / TS;
    float m_run[GW], l_run[GW];
    float2 acc[GW][E / 2];
    // With RB each role's register budget is set inside its own branch, and
    // neither branch rejoins the other before its budget ends: the compiler
    // allocates registers per region, and code reachable under both budgets
    // gets the smaller one.
    if (warp >= NWC) {
        if constexpr (RB) {
            setmaxnreg_dec<C::REG_PRODUCER>();
            if (warp > NWC) return;  // the producer warpgroup's idle warps
        }
        // ---------------- producer: PL lanes issue the copies ----------------
        // Lane c0 < PL serves streams c0, c0 + PL, ... (PL = NST: a lane per
        // stream; PL = 1: one lane for all).  A lane polls its streams' next
        // stages without blocking and issues as soon as one is free, so a
        // slow stream never holds back the others; within a stream, chunks
        // and stage phases are issued strictly in order.  One issuing lane
        // caps a CTA at roughly one stage per 0.3 us, which 8 KiB stages feel
        // (D = 128, fp8 caches); with 16 KiB stages and wide groups the one
        // lane, which staggers the streams, measured faster.
        constexpr int PL = LP ? NST : 1, SPL = NST / PL;
        static_assert(PL <= 32, "one producer warp");
        if (lane < PL) {
            const unsigned mask = PL == 32 ? 0xffffffffu : (1u << PL) - 1u;
            auto any = [&](bool v) {  // over the producer lanes
                if constexpr (PL == 1)
                    return v;
                else
                    return __any_sync(mask, v);
            };
            const uint64_t policy = l2_policy_evict_first();
            auto issue = [&](int c, int k) {  // chunk c + k * NST into stream c's stage k % SPS
                const int i = c + k * NST, s = c * SPS + k % SPS;
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
                tma_load_4d(st, &tm_k, &full[s], 0, kvh, off, page, policy);
                tma_load_4d(st + C::CHUNK_BYTES, &tm_v, &full[s], 0, kvh, off, page, policy);
            };
            int next[SPL];
            int remaining = PL == 1 ? n_my : 0;
#pragma unroll
            for (int j = 0; j < SPL; ++j) {
                next[j] = 0;
                if constexpr (PL > 1) remaining += max(0, (n_my - lane - j * PL + NST - 1) / NST);  // chunks c, c + NST, ...
            }
            if (p.early_kv) {
                // First use of every stage: the chunks i < n_pre (those that
                // end before the new row, token L - 1) go out before the
                // dependency wait; chunk i is stream i % NST's (i / NST)-th,
                // and n_pre <= NS, so none of them waits for a free stage.
                const int n_pre = max(0, min(min(NS, n_my), (L - 1) / kChunk - c_begin));
#pragma unroll 1
                for (int i = lane; i < n_pre; i += PL) issue(i % NST, i / NST);
#pragma unroll
                for (int j = 0; j < SPL; ++j) {
                    const int c = lane + j * PL;
                    next[j] = max(0, (n_pre - c + NST - 1) / NST);
                    remaining -= next[j];
                }
                pdl_wait_primary();
            }
            uint32_t idle = 0;
            bool gave_up = false;
            while (any(remaining > 0)) {
                bool progress = false;
#pragma unroll
                for (int j = 0; j < SPL; ++j) {
                    const int c = lane + j * PL, k = next[j], i = c + k * NST;
                    if (i >= n_my) continue;
                    const int s = c * SPS + k % SPS, ph = k / SPS;
                    if (ph > 0 && !mbar_test_wait(&empty[s], (ph - 1) & 1)) continue;
                    issue(c, k);
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
                // Giving up: let the copies already in flight land before the
                // CTA ends (each stream's last SPS chunks, one per stage).
                if (lane == 0) flags[0] = 1;
#pragma unroll
                for (int j = 0; j < SPL; ++j) {
                    const int c = lane + j * PL;
                    for (int k = max(0, next[j] - SPS); k < next[j]; ++k) {
                        uint64_t *bar = &full[c * SPS + k % SPS];
                        for (uint32_t n = 0; n < kWaitPollLimit && !mbar_try_wait(bar, (k / SPS) & 1); ++n) {
                        }
                    }
                }
                if (lane == 0) set_status(p.status, PA_DEV_TIMEOUT);
            }
        }
        // With RB the producer leaves here: its copies have all landed (the
        // consumers wait for every chunk, or it waited for its own copies
        // before giving up), and the merge below synchronises the consumers
        // only.  A bad page index it met reaches the consumers through the
        // full barrier of that chunk, which orders its flag write before
        // their wait returns.
        if constexpr (RB) return;
    } else {
        if constexpr (RB) setmaxnreg_inc<C::REG_CONSUMER>();
        // ---------------- consumers ----------------
        // Arithmetic runs on fp32 pairs (packed FFMA2): dot products pair
        // adjacent dims (even/odd partial sums), the P.V update pairs adjacent
        // output dims with the probability duplicated in both halves.
        const int cg = (lane >> 2) & 7;
        float2 *pbuf = pbuf_all + warp * (8 * MB * C::GP2);
        float2 q2[GW][E / 2];
        if (p.early_kv) pdl_wait_primary();  // q may come from the work before this call
        {
            const uint8_t *qrow =
                reinterpret_cast<const uint8_t *>(p.q + ((size_t)b * p.num_q_heads + hq0 + hg * GW) * D) + lane * E * 2;
            const float qs = F8 ? p.scale_log2 * p.k_scale[kvh] : p.scale_log2;
            const float2 sc2 = make_float2(qs, qs);
#pragma unroll
            for (int g = 0; g < GW; ++g) {
                load_bf16_pairs<E>(qrow + g * D * 2, q2[g]);
#pragma unroll
                for (int j = 0; j < E / 2; ++j) q2[g][j] = __fmul2_rn(q2[g][j], sc2);
            }
        }
#pragma unroll
        for (int g = 0; g < GW; ++g) {
            m_run[g] = -INFINITY;
            l_run[g] = 0.f;
#pragma unroll
            for (int j = 0; j < E / 2; ++j) acc[g][j] = make_float2(0.f, 0.f);
        }

        for (int i = stream, k = 0; i < n_my; i += NST, ++k) {
            const int s = stream * SPS + k % SPS;
            // the loop body holds full-warp shuffles: every lane leaves together
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (k / SPS) & 1, &flags[0]))) {
                flags[0] = 1;
                break;
            }
            const uint8_t *kst = smem + s * C::STAGE_BYTES + wh * 8 * C::ROW_BYTES + lane * E * (F8 ? 1 : 2);
            const uint8_t *vst = kst + C::CHUNK_BYTES;
            // valid rows [lead, nv) of this warp's part of the chunk: nv may be
            // <= lead in the last chunk, lead > 0 only where the window starts
            const int nv = min(8 * MB, L - (c_begin + i) * kChunk - wh * 8);
            const int lead = WIN ? max(0, L - p.window - (c_begin + i) * kChunk - wh * 8) : 0;

            float sc[MB][GW];
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
                // Slots j and j + 4 are formed together and the first butterfly
                // step (lane XOR 16) folds the high one into the low one at once.
                float part[4][GW];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float hi[GW];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int slot = j + 4 * h;
                        float2 k2[E / 2];
                        load_kv_pairs<E, F8>(kst + (mb * 8 + (slot ^ cg)) * C::ROW_BYTES, k2);
#pragma unroll
                        for (int g = 0; g < GW; ++g) {
                            float2 a = __fmul2_rn(q2[g][0], k2[0]);
#pragma unroll
                            for (int jj = 1; jj < E / 2; ++jj) a = __ffma2_rn(q2[g][jj], k2[jj], a);
                            if (h == 0)
                                part[j][g] = a.x + a.y;
                            else
                                hi[g] = a.x + a.y;
                        }
                    }
                    // with an even number of heads, pairs of heads are added as packed
                    // fp32 pairs (one instruction per two heads)
                    if constexpr (GW % 2 == 0) {
#pragma unroll
                        for (int g = 0; g < GW; g += 2) {
                            const float2 x = __fadd2_rn(make_float2(part[j][g], part[j][g + 1]),
                                                        make_float2(__shfl_xor_sync(0xffffffffu, hi[g], 16),
                                                                    __shfl_xor_sync(0xffffffffu, hi[g + 1], 16)));
                            part[j][g] = x.x;
                            part[j][g + 1] = x.y;
                        }
                    } else {
#pragma unroll
                        for (int g = 0; g < GW; ++g) part[j][g] += __shfl_xor_sync(0xffffffffu, hi[g], 16);
                    }
                }
                // Rest of the transposing butterfly: 4 slots x GW -> 1 slot x GW.
                if constexpr (GW % 2 == 0) {
                    auto add2 = [&](float &a, float &b, float x, float y) {
                        const float2 r = __fadd2_rn(make_float2(a, b), make_float2(x, y));
                        a = r.x;
                        b = r.y;
                    };
#pragma unroll
                    for (int g = 0; g < GW; g += 2) {
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            add2(part[j][g], part[j][g + 1], __shfl_xor_sync(0xffffffffu, part[j + 2][g], 8),
                                 __shfl_xor_sync(0xffffffffu, part[j + 2][g + 1], 8));
                        add2(part[0][g], part[0][g + 1], __shfl_xor_sync(0xffffffffu, part[1][g], 4),
                             __shfl_xor_sync(0xffffffffu, part[1][g + 1], 4));
                        add2(part[0][g], part[0][g + 1], __shfl_xor_sync(0xffffffffu, part[0][g], 2),
                             __shfl_xor_sync(0xffffffffu, part[0][g + 1], 2));
                        add2(part[0][g], part[0][g + 1], __shfl_xor_sync(0xffffffffu, part[0][g], 1),
                             __shfl_xor_sync(0xffffffffu, part[0][g + 1], 1));
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < GW; ++g) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) part[j][g] += __shfl_xor_sync(0xffffffffu, part[j + 2][g], 8);
                        part[0][g] += __shfl_xor_sync(0xffffffffu, part[1][g], 4);
                        part[0][g] += __shfl_xor_sync(0xffffffffu, part[0][g], 2);
                        part[0][g] += __shfl_xor_sync(0xffffffffu, part[0][g], 1);
                    }
                }
                const bool valid = (mb * 8 + cg) < nv && (mb * 8 + cg) >= lead;
#pragma unroll
                for (int g = 0; g < GW; ++g) sc[mb][g] = valid ? part[0][g] : -INFINITY;
            }

            if (nv > lead) {  // warp-uniform
                // Lazy online softmax (log2 domain): the chunk max of a head is
                // finite because this part has >= 1 valid row.
                float mx[GW];
                bool raise_any = false;
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    float v = sc[0][g];
#pragma unroll
                    for (int mb = 1; mb < MB; ++mb) v = fmaxf(v, sc[mb][g]);
                    mx[g] = warp_max(v);
                    raise_any |= mx[g] > m_run[g] + kLazyLog2;
                }
                if (raise_any) {
#pragma unroll
                    for (int g = 0; g < GW; ++g) {
                        if (mx[g] > m_run[g] + kLazyLog2) {
                            const float alpha = fast_exp2(m_run[g] - mx[g]);  // 0 on the first chunk
                            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                            for (int j = 0; j < E / 2; ++j) acc[g][j] = __fmul2_rn(acc[g][j], a2);
                            l_run[g] *= alpha;
                            m_run[g] = mx[g];
                        }
                    }
                }
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    float ps = 0.f;
#pragma unroll
                    for (int mb = 0; mb < MB; ++mb) {
                        const float pv = fast_exp2(sc[mb][g] - m_run[g]);  // 0 for rows past the end
                        ps += pv;
                        sc[mb][g] = pv;
                    }
                    l_run[g] += ps;
                }
                if ((lane & 3) == 0) {
#pragma unroll
                    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
                        for (int g = 0; g < GW; ++g) pbuf[(mb * 8 + cg) * C::GP2 + g] = make_float2(sc[mb][g], sc[mb][g]);
                }
                __syncwarp();

                auto pv_row = [&](int t) {
                    float2 v2[E / 2];
                    load_kv_pairs<E, F8>(vst + t * C::ROW_BYTES, v2);
                    float2 pp[C::GP2];
#pragma unroll
                    for (int j = 0; j < C::GP2; j += 2) {
                        const float4 x = *reinterpret_cast<const float4 *>(pbuf + t * C::GP2 + j);
                        pp[j] = make_float2(x.x, x.y);
                        pp[j + 1] = make_float2(x.z, x.w);
                    }
#pragma unroll
                    for (int g = 0; g < GW; ++g)
#pragma unroll
                        for (int j = 0; j < E / 2; ++j) acc[g][j] = __ffma2_rn(pp[g], v2[j], acc[g][j]);
                };
                // rows before the window start have p = 0 and hold finite
                // cached values, so they run through P.V like the others
                if (nv == 8 * MB) {
                    // measured: two rows per step beat four and eight for the
                    // register-rebalanced layout (32.07 against 32.27 us at 32K)
#pragma unroll(RB ? 2 : 4)
                    for (int t = 0; t < 8 * MB; ++t) pv_row(t);
                } else {
#pragma unroll 1
                    for (int t = 0; t < nv; ++t) pv_row(t);
                }
                __syncwarp();
            }
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // l_run counts each token once per 4 lanes (bits 0-1 replicate) and is
        // split across lane bits 2-4.
#pragma unroll
        for (int g = 0; g < GW; ++g) {
            float l = l_run[g];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            l_run[g] = l;
        }
    }

    auto cta_sync = [&]() {
        if constexpr (RB)
            named_bar_sync(1, NWC * 32);
        else
            __syncthreads();
    };
    constexpr int MT = RB ? NWC * 32 : C::THREADS;  // threads taking part in the merge
    cta_sync();  // every chunk is consumed: the stage buffers become the merge area
    const bool aborted = flags[0] != 0;
    // Merge the warp states of this split (same log-sum-exp rule as the split
    // reduce) and write the split result: the warps store their states
    // ([warp][GW][D], [warp][GW]), warp 0 forms the weights 2^(m_w - M) /
    // sum_w l_w 2^(m_w - M) over the NWH warps holding each head with
    // shuffles, and every output is a weighted sum over those warps read with
    // 16-byte shared loads.
    float *merge_acc = reinterpret_cast<float *>(smem);  // [NWC][GW][D]
    float *wgt = reinterpret_cast<float *>(merge_ml + NWC * GW);  // [NWC][GW] after (m, l)
    const bool poisoned = aborted || flags[1] != 0;
    // the k-th warp holding head h (k < NWH): stream k / TS, token half k % TS
    auto holder = [&](int h, int k) { return (k / TS) * WPC + (h / GW) * TS + (k % TS); };
    if (warp < NWC) {
#pragma unroll
        for (int g = 0; g < GW; ++g) {
            float *dst = merge_acc + (warp * GW + g) * D + lane * E;
#pragma unroll
            for (int j = 0; j < E / 2; j += 2)
                *reinterpret_cast<float4 *>(dst + 2 * j) =
                    make_float4(acc[g][j].x, acc[g][j].y, acc[g][j + 1].x, acc[g][j + 1].y);
            if (lane == 0) merge_ml[warp * GW + g] = make_float2(m_run[g], l_run[g]);
        }
    }
    cta_sync();
    if (warp == 0) {
        // lane groups of NWP >= NWH lanes, one group per head; surplus lanes hold empty states
        constexpr int NWP = NWH <= 8 ? 8 : (NWH <= 16 ? 16 : 32);
        static_assert(NWH <= 32, "the warp states of a head fit one warp");
        constexpr int HPP = 32 / NWP;  // heads per pass
#pragma unroll
        for (int h0 = 0; h0 < G; h0 += HPP) {
            const int k = lane % NWP, h = h0 + lane / NWP;
            const bool mine = k < NWH && h < G;
            const int slot = mine ? holder(h, k) * GW + h % GW : 0;
            const float2 ml = mine ? merge_ml[slot] : make_float2(-INFINITY, 0.f);
            float M = ml.x;
#pragma unroll
            for (int o = 1; o < NWP; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float e = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;  // 0 for a warp without rows
            float lsum = ml.y * e;
#pragma unroll
            for (int o = 1; o < NWP; o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
            const bool zero = poisoned || !(lsum > 0.f);
            if (mine) {
                wgt[slot] = zero ? 0.f : (F8 ? e / lsum * p.v_scale[kvh] : e / lsum);
                if (k == 0 && p.num_splits > 1)
                    p.part_ml[((size_t)b * p.num_q_heads + hq0 + h) * p.num_splits + split] =
                        make_float2(M, poisoned ? -1.f : lsum);
            }
        }
    }
    cta_sync();
    for (int idx = threadIdx.x; idx < G * D / 4; idx += MT) {
        const int h = (4 * idx) / D, d = 4 * idx - h * D;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
        for (int k = 0; k < NWH; ++k) {
            const int slot = holder(h, k) * GW + h % GW;
            const float4 x = *reinterpret_cast<const float4 *>(merge_acc + slot * D + d);
            const float wg = wgt[slot];
            o.x = fmaf(x.x, wg, o.x);
            o.y = fmaf(x.y, wg, o.y);
            o.z = fmaf(x.z, wg, o.z);
            o.w = fmaf(x.w, wg, o.w);
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

// ---------------------------------------------------------------------------
// Partition reduce: out[row, h, :] = sum_i w_i o_i / sum_i w_i with
// w_i = l_i 2^(m_i - max_j m_j) over the non-empty splits of the row's sequence
// (the "reduce afterwards" step of the split-KV fix).  A poisoned split
// (l = -1: bad page or an abandoned wait) zeroes the row.  Rows are
// (sequence, new row) pairs: q_len = 1 for decode, > 1 for verify.
struct ReduceParams {
    const float *part_o;
    const float2 *part_ml;
    void *out;
    int num_q_heads;
    int num_splits;
    int out_bf16;
};


// Grid (Hq, rows, D / 32), 128 threads: each CTA merges a 32-wide slice of
// one (row, head) output.  Its threads split the splits 16 ways; every thread
// issues the loads of all its splits' statistics and partial outputs at once,
// folds them with a running log-sum-exp, and a single exchange merges the 16
// per-group states.  (32-wide slices measured 0.56 us faster per 32K call than
// 64-wide ones and 0.17 us faster than 16-wide ones: more CTAs, fewer loads
// per thread.)
template <int D>
__global__ void __launch_bounds__(128) pa_split_reduce_kernel(const ReduceParams p) {
    constexpr int QD = 8;   // float4 columns of the 32-wide slice
    constexpr int SG = 16;  // split groups
    constexpr int UNROLL = 4;
    __shared__ float4 red_o[SG][QD];
    __shared__ float2 red_ml[SG];
    __shared__ int red_bad;
    pdl_launch_dependents();  // a following attention call may start its set-up
    if (threadIdx.x == 0) red_bad = 0;
    pdl_wait_primary();       // partials of the split kernel are complete and visible

    const int hq = blockIdx.x, row = blockIdx.y, slice = blockIdx.z;
    // Every split wrote its record (an empty one as m = -inf, l = 0), so all
    // of them are read and the sequence length is not needed here.
    const int S_b = p.num_splits;
    const size_t r = (size_t)row * p.num_q_heads + hq;
    const float2 *ml = p.part_ml + r * p.num_splits;
    const int qd = threadIdx.x % QD, sg = threadIdx.x / QD;
    const float *po = p.part_o + r * p.num_splits * D + slice * 32 + qd * 4;

    float M = -INFINITY, W = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    bool bad = false;
    for (int i0 = sg; i0 < S_b; i0 += SG * UNROLL) {
        float2 v[UNROLL];
        float4 o[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {  // all loads first, none behind a branch
            const int i = min(i0 + u * SG, S_b - 1);
            v[u] = ml[i];
            o[u] = *reinterpret_cast<const float4 *>(po + (size_t)i * D);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (i0 + u * SG >= S_b) v[u] = make_float2(-INFINITY, 0.f);  // a repeated load: ignore it
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            bad |= v[u].y < 0.f;
            if (!(v[u].y > 0.f)) continue;  // empty split (or poisoned, flagged above)
            const float Mn = fmaxf(M, v[u].x);
            const float c = fast_exp2(M - Mn), e = fast_exp2(v[u].x - Mn) * v[u].y;
            W = fmaf(W, c, e);
            a.x = fmaf(a.x, c, e * o[u].x); a.y = fmaf(a.y, c, e * o[u].y);
            a.z = fmaf(a.z, c, e * o[u].z); a.w = fmaf(a.w, c, e * o[u].w);
            M = Mn;
        }
    }
    if (bad) red_bad = 1;
    red_o[sg][qd] = a;
    if (qd == 0) red_ml[sg] = make_float2(M, W);
    __syncthreads();
    if (sg == 0) {
        float Mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < SG; ++j) Mt = fmaxf(Mt, red_ml[j].x);
        float Wt = 0.f;
        float4 at = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < SG; ++j) {
            const float2 mw = red_ml[j];
            if (!(mw.y > 0.f)) continue;
            const float c = fast_exp2(mw.x - Mt);
            const float4 o = red_o[j][qd];
            Wt = fmaf(mw.y, c, Wt);
            at.x = fmaf(o.x, c, at.x); at.y = fmaf(o.y, c, at.y); at.z = fmaf(o.z, c, at.z); at.w = fmaf(o.w, c, at.w);
        }
        const bool zero = red_bad != 0 || !(Wt > 0.f);
        const float inv = zero ? 0.f : 1.f / Wt;
        const size_t base = r * D + slice * 32 + qd * 4;
        store_out(p.out, base + 0, at.x * inv, p.out_bf16);
        store_out(p.out, base + 1, at.y * inv, p.out_bf16);
        store_out(p.out, base + 2, at.z * inv, p.out_bf16);
        store_out(p.out, base + 3, at.w * inv, p.out_bf16);
    }
}

// The same merge for few splits (S <= 8, e.g. verify, batched decode): one
// warp per (row, head), a lane owning D/32 consecutive dims.  All S records
// and partial vectors of a lane are loaded at once, so the kernel makes one
// dependent round trip, and no CTA waits on a shared-memory exchange.
constexpr int kReduceSmallMaxSplits = 8;

template <int D>
__global__ void __launch_bounds__(256) pa_split_reduce_small_kernel(const ReduceParams p, int pairs) {
    constexpr int E = D / 32;  // dims per lane
    pdl_launch_dependents();   // a following attention call may start its set-up
    pdl_wait_primary();        // partials of the split kernel are complete and visible
    const int pair = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (pair >= pairs) return;
    const int S = p.num_splits;
    const float2 *ml = p.part_ml + (size_t)pair * S;
    const float *po = p.part_o + (size_t)pair * S * D + lane * E;
    float2 v[kReduceSmallMaxSplits];
    float4 o[kReduceSmallMaxSplits][E / 4];
#pragma unroll
    for (int u = 0; u < kReduceSmallMaxSplits; ++u) {  // all loads first, none behind a branch
        const int i = min(u, S - 1);
        v[u] = ml[i];
#pragma unroll
        for (int e = 0; e < E / 4; ++e) o[u][e] = *reinterpret_cast<const float4 *>(po + (size_t)i * D + 4 * e);
    }
    float M = -INFINITY, W = 0.f;
    float4 a[E / 4];
#pragma unroll
    for (int e = 0; e < E / 4; ++e) a[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    bool bad = false;
#pragma unroll
    for (int u = 0; u < kReduceSmallMaxSplits; ++u) {
        if (u >= S) break;
        bad |= v[u].y < 0.f;
        if (!(v[u].y > 0.f)) continue;  // empty split (or poisoned, flagged above)
        const float Mn = fmaxf(M, v[u].x);
        const float c = fast_exp2(M - Mn), w = fast_exp2(v[u].x - Mn) * v[u].y;
        W = fmaf(W, c, w);
#pragma unroll
        for (int e = 0; e < E / 4; ++e) {
            a[e].x = fmaf(a[e].x, c, w * o[u][e].x);
            a[e].y = fmaf(a[e].y, c, w * o[u][e].y);
            a[e].z = fmaf(a[e].z, c, w * o[u][e].z);
            a[e].w = fmaf(a[e].w, c, w * o[u][e].w);
        }
        M = Mn;
    }
    const float inv = (bad || !(W > 0.f)) ? 0.f : 1.f / W;
    const size_t base = (size_t)pair * D + lane * E;
#pragma unroll
    for (int e = 0; e < E / 4; ++e) {
        store_out(p.out, base + 4 * e + 0, a[e].x * inv, p.out_bf16);
        store_out(p.out, base + 4 * e + 1, a[e].y * inv, p.out_bf16);
        store_out(p.out, base + 4 * e + 2, a[e].z * inv, p.out_bf16);
        store_out(p.out, base + 4 * e + 3, a[e].w * inv, p.out_bf16);
    }
}

}  // namespace pa
