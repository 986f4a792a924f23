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
//    a page, and the block table is read once per page in chunk order
//    (the page-contiguous walk of Sec.7).  Only the last chunk of a sequence
//    can be partial; its rows past the end are masked (scores) and skipped (PV).
//  * One producer warp issues the copies into an NS-stage mbarrier ring; NW
//    consumer warps take chunks round-robin, each with its own online softmax.
//  * Each K/V row is read from shared memory once and used by all G query
//    heads of the group (GQA reuse).  A lane owns E = D/32 consecutive
//    elements of d: q (pre-scaled to log2 units) and the output accumulator
//    for its G heads stay in registers.
//  * Scores: per micro-batch of 8 tokens a lane forms 8 x G partial dot
//    products over its d slice, and a transposing butterfly sums them across
//    the 32 lanes.  Lane l computes token (slot XOR ((l >> 2) & 7)) in slot, so
//    at every halving step each lane keeps its low slots and sends its high
//    ones (no selects); afterwards lane l holds all G scores of token
//    (l >> 2) & 7 of the micro-batch.
//  * Probabilities go through a per-warp shared buffer so every lane can
//    broadcast-read p for each token of the PV accumulation.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kChunk = 16;  // tokens per TMA copy and per pipeline stage

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
};

template <int D, int G, int NW, int NS>
struct DecodeCfg {
    static constexpr int E = D / 32;
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int CHUNK_BYTES = kChunk * ROW_BYTES;
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;  // K chunk, then V chunk
    static constexpr int GP = (G + 3) & ~3;              // floats per P row (16-byte rows)
    static constexpr int STAGES_BYTES = NS * STAGE_BYTES;
    static constexpr int MERGE_BYTES = NW * G * D * 4;
    static constexpr int OFF_P = STAGES_BYTES;
    static constexpr int OFF_ML = OFF_P + NW * kChunk * GP * 4;
    static constexpr int OFF_BAR = OFF_ML + NW * G * 8;
    static constexpr int OFF_FLAGS = OFF_BAR + 2 * NS * 8;
    static constexpr int SMEM_BYTES = OFF_FLAGS + 16 + 1024;  // + slack to align the base to 1 KiB
    static constexpr int THREADS = (NW + 1) * 32;
    static_assert(D % 32 == 0 && (E == 8 || E == 4), "head_dim 256 or 128");
    static_assert(MERGE_BYTES <= STAGES_BYTES, "the CTA merge reuses the stage buffers");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// E consecutive bf16 of a row -> floats.
template <int E>
__device__ __forceinline__ void load_bf16_row(const uint8_t *src, float (&f)[E]) {
    if constexpr (E == 8) {
        const uint4 w = *reinterpret_cast<const uint4 *>(src);
        f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
        f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
    } else {
        const uint2 w = *reinterpret_cast<const uint2 *>(src);
        f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    }
}

__device__ __forceinline__ void store_out(void *out, size_t idx, float v, int out_bf16) {
    if (out_bf16)
        reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float *>(out)[idx] = v;
}

template <int D, int G, int NW, int NS>
__global__ void __launch_bounds__((NW + 1) * 32, 1)
    pa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const DecodeParams p) {
    using C = DecodeCfg<D, G, NW, NS>;
    constexpr int E = C::E;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    float *pbuf_all = reinterpret_cast<float *>(smem + C::OFF_P);
    float2 *merge_ml = reinterpret_cast<float2 *>(smem + C::OFF_ML);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + NS;
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::OFF_FLAGS);  // [0] abort, [1] bad page

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq0 = kvh * G;

    pdl_launch_dependents();

    int L = p.seq_lens[b];
    if (L < 0 || L > p.max_seq_len) {
        if (threadIdx.x == 0 && split == 0 && kvh == 0) set_status(p.status, PA_DEV_BAD_SEQLEN);
        L = 0;
    }
    const int n_chunks = (L + kChunk - 1) / kChunk;
    const int c_begin = split * p.chunks_per_split;
    const int n_my = min(n_chunks - c_begin, p.chunks_per_split);
    if (n_my <= 0) {
        // Nothing of this sequence falls in this split.  The merge reads only
        // non-empty splits; an unsplit call owns its output rows and zeroes them.
        if (p.num_splits == 1)
            for (int idx = threadIdx.x; idx < G * D; idx += C::THREADS)
                store_out(p.out, ((size_t)b * p.num_q_heads + hq0) * D + idx, 0.f, p.out_bf16);
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();

    float m_run[G], l_run[G], acc[G][E];
    if (warp == NW) {
        // ---------------- producer: one lane issues every copy ----------------
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            const uint64_t policy = l2_policy_evict_first();
            const int32_t *bt = p.block_table + (size_t)b * p.max_pages_per_seq;
            int cur_lp = -1, page = 0, issued = 0;
            for (int i = 0; i < n_my; ++i) {
                const int s = i % NS;
                if (i >= NS && !mbar_wait(&empty[s], ((i / NS) - 1) & 1, &flags[0])) {
                    flags[0] = 1;
                    break;
                }
                const int t0 = (c_begin + i) * kChunk;
                const int lp = t0 / p.block_size;
                if (lp != cur_lp) {  // one table read per page
                    cur_lp = lp;
                    page = bt[lp];
                    if (page < 0 || (int64_t)page >= p.num_pages) {
                        flags[1] = 1;  // the copy below reads zeros (box outside the tensor)
                        set_status(p.status, PA_DEV_BAD_PAGE);
                    }
                }
                const int off = t0 - lp * p.block_size;
                uint8_t *st = smem + s * C::STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
                tma_load_4d(st, &tm_k, &full[s], 0, kvh, off, page, policy);
                tma_load_4d(st + C::CHUNK_BYTES, &tm_v, &full[s], 0, kvh, off, page, policy);
                issued = i + 1;
            }
            if (flags[0]) {
                // Giving up: let the copies already in flight land before the CTA ends.
                for (int i = max(0, issued - NS); i < issued; ++i) {
                    uint64_t *bar = &full[i % NS];
                    for (uint32_t n = 0; n < kWaitPollLimit && !mbar_try_wait(bar, (i / NS) & 1); ++n) {
                    }
                }
                set_status(p.status, PA_DEV_TIMEOUT);
            }
        }
    } else {
        // ---------------- consumers ----------------
        const int cg = (lane >> 2) & 7;
        float *pbuf = pbuf_all + warp * (kChunk * C::GP);
        float qf[G][E];
        {
            const uint8_t *qrow = reinterpret_cast<const uint8_t *>(p.q + ((size_t)b * p.num_q_heads + hq0) * D) +
                                  lane * E * 2;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                load_bf16_row<E>(qrow + g * D * 2, qf[g]);
#pragma unroll
                for (int e = 0; e < E; ++e) qf[g][e] *= p.scale_log2;
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m_run[g] = -INFINITY;
            l_run[g] = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[g][e] = 0.f;
        }

        for (int i = warp; i < n_my; i += NW) {
            const int s = i % NS;
            if (!mbar_wait(&full[s], (i / NS) & 1, &flags[0])) {
                flags[0] = 1;
                break;
            }
            const uint8_t *kst = smem + s * C::STAGE_BYTES;
            const uint8_t *vst = kst + C::CHUNK_BYTES;
            const int nv = min(kChunk, L - (c_begin + i) * kChunk);  // valid rows, >= 1

            float sc[2][G];
#pragma unroll
            for (int mb = 0; mb < 2; ++mb) {
                float part[8][G];
#pragma unroll
                for (int slot = 0; slot < 8; ++slot) {
                    float kf[E];
                    load_bf16_row<E>(kst + (mb * 8 + (slot ^ cg)) * C::ROW_BYTES + lane * E * 2, kf);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float a = qf[g][0] * kf[0];
#pragma unroll
                        for (int e = 1; e < E; ++e) a = fmaf(qf[g][e], kf[e], a);
                        part[slot][g] = a;
                    }
                }
                // Transposing butterfly: 8 slots x G -> 1 slot x G, summed over all lanes.
#pragma unroll
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) part[j][g] += __shfl_xor_sync(0xffffffffu, part[j + 4][g], 16);
#pragma unroll
                    for (int j = 0; j < 2; ++j) part[j][g] += __shfl_xor_sync(0xffffffffu, part[j + 2][g], 8);
                    part[0][g] += __shfl_xor_sync(0xffffffffu, part[1][g], 4);
                    part[0][g] += __shfl_xor_sync(0xffffffffu, part[0][g], 2);
                    part[0][g] += __shfl_xor_sync(0xffffffffu, part[0][g], 1);
                }
                const bool valid = (mb * 8 + cg) < nv;
#pragma unroll
                for (int g = 0; g < G; ++g) sc[mb][g] = valid ? part[0][g] : -INFINITY;
            }

            // Online softmax update (log2 domain); every chunk has >= 1 valid row,
            // so the chunk max is finite.
            float alpha[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float mx = fmaxf(sc[0][g], sc[1][g]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m_run[g], mx);
                alpha[g] = fast_exp2(m_run[g] - m_new);
                const float p0 = fast_exp2(sc[0][g] - m_new);
                const float p1 = fast_exp2(sc[1][g] - m_new);
                l_run[g] = fmaf(l_run[g], alpha[g], p0 + p1);
                m_run[g] = m_new;
                sc[0][g] = p0;
                sc[1][g] = p1;
            }
            if ((lane & 3) == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    pbuf[cg * C::GP + g] = sc[0][g];
                    pbuf[(8 + cg) * C::GP + g] = sc[1][g];
                }
            }
            __syncwarp();
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < E; ++e) acc[g][e] *= alpha[g];

            auto pv_row = [&](int t) {
                float vf[E];
                load_bf16_row<E>(vst + t * C::ROW_BYTES + lane * E * 2, vf);
                float pr[C::GP];
#pragma unroll
                for (int j = 0; j < C::GP; j += 4) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(pbuf + t * C::GP + j);
                    pr[j] = v4.x; pr[j + 1] = v4.y; pr[j + 2] = v4.z; pr[j + 3] = v4.w;
                }
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[g][e] = fmaf(pr[g], vf[e], acc[g][e]);
            };
            if (nv == kChunk) {
#pragma unroll
                for (int t = 0; t < kChunk; ++t) pv_row(t);
            } else {
                for (int t = 0; t < nv; ++t) pv_row(t);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // l_run is replicated across lane bits 0-1 and split across bits 2-4.
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float l = l_run[g];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            l_run[g] = l;
        }
    }

    __syncthreads();  // every chunk is consumed: the stage buffers become the merge area
    const bool aborted = flags[0] != 0;
    float *merge_acc = reinterpret_cast<float *>(smem);  // [NW][G][D]
    if (warp < NW) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float *dst = merge_acc + (warp * G + g) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; e += 4) *reinterpret_cast<float4 *>(dst + e) = make_float4(acc[g][e], acc[g][e + 1], acc[g][e + 2], acc[g][e + 3]);
            if (lane == 0) merge_ml[warp * G + g] = make_float2(m_run[g], l_run[g]);
        }
    }
    __syncthreads();

    // Merge the NW warp states of this split (same log-sum-exp rule as the
    // split reduce) and write the split result.
    const bool poisoned = aborted || flags[1] != 0;
    for (int idx = threadIdx.x; idx < G * D; idx += C::THREADS) {
        const int g = idx / D, d = idx - (idx / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, merge_ml[w * G + g].x);
        float lsum = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float2 ml = merge_ml[w * G + g];
            const float wgt = fast_exp2(ml.x - M);  // 0 for a warp without chunks (m = -inf)
            lsum = fmaf(ml.y, wgt, lsum);
            o = fmaf(merge_acc[(w * G + g) * D + d], wgt, o);
        }
        const float res = (poisoned || !(lsum > 0.f)) ? 0.f : o / lsum;
        const size_t row = (size_t)b * p.num_q_heads + hq0 + g;
        if (p.num_splits == 1) {
            store_out(p.out, row * D + d, res, p.out_bf16);
        } else {
            p.part_o[(row * p.num_splits + split) * D + d] = res;
            if (d == 0) p.part_ml[row * p.num_splits + split] = make_float2(M, poisoned ? -1.f : lsum);
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
    const int32_t *seq_lens;
    void *out;
    int num_q_heads;
    int q_len;
    int max_seq_len;
    int chunks_per_split;
    int num_splits;
    int out_bf16;
};

template <int D>
__global__ void __launch_bounds__(256) pa_split_reduce_kernel(const ReduceParams p) {
    constexpr int QD = D / 4;       // float4 columns
    constexpr int SG = 256 / QD;    // split groups
    __shared__ float4 red[SG][QD];
    pdl_wait_primary();  // partials of the split kernel are complete and visible

    const int hq = blockIdx.x, row = blockIdx.y;
    const int b = row / p.q_len;
    int L = p.seq_lens[b];
    if (L < 0 || L > p.max_seq_len || L < p.q_len) L = 0;  // same rule as the split kernels
    const int n_chunks = (L + kChunk - 1) / kChunk;
    const int S_b = min(p.num_splits, (n_chunks + p.chunks_per_split - 1) / p.chunks_per_split);
    const size_t r = (size_t)row * p.num_q_heads + hq;
    const float2 *ml = p.part_ml + r * p.num_splits;

    float M = -INFINITY;
    bool bad = false;
    for (int i = 0; i < S_b; ++i) {
        const float2 v = ml[i];
        bad |= v.y < 0.f;
        if (v.y > 0.f) M = fmaxf(M, v.x);
    }
    float wsum = 0.f;
    for (int i = 0; i < S_b; ++i) {
        const float2 v = ml[i];
        if (v.y > 0.f) wsum = fmaf(v.y, fast_exp2(v.x - M), wsum);
    }
    const int qd = threadIdx.x % QD, sg = threadIdx.x / QD;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = sg; i < S_b; i += SG) {
        const float2 v = ml[i];
        if (!(v.y > 0.f)) continue;
        const float w = v.y * fast_exp2(v.x - M);
        const float4 o = *reinterpret_cast<const float4 *>(p.part_o + (r * p.num_splits + i) * D + qd * 4);
        a.x = fmaf(w, o.x, a.x); a.y = fmaf(w, o.y, a.y); a.z = fmaf(w, o.z, a.z); a.w = fmaf(w, o.w, a.w);
    }
    red[sg][qd] = a;
    __syncthreads();
    if (sg == 0) {
        for (int j = 1; j < SG; ++j) {
            const float4 o = red[j][qd];
            a.x += o.x; a.y += o.y; a.z += o.z; a.w += o.w;
        }
        const bool zero = bad || !(wsum > 0.f);
        const float inv = zero ? 0.f : 1.f / wsum;
        const size_t base = r * D + qd * 4;
        store_out(p.out, base + 0, a.x * inv, p.out_bf16);
        store_out(p.out, base + 1, a.y * inv, p.out_bf16);
        store_out(p.out, base + 2, a.z * inv, p.out_bf16);
        store_out(p.out, base + 3, a.w * inv, p.out_bf16);
    }
}

}  // namespace pa
