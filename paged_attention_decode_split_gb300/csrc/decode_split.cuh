// decode_split.cuh -- what the split-KV attention kernels share: the decode
// launch parameters, the 16-token chunk that is the unit of every split, and
// the partition reduce that merges the splits.
//
// The split method ("Hybrid SSM decode rate on dual Radeon under vLLM", the
// split-KV fix): the context of every (sequence, KV head) is cut into splits
// of whole 16-token chunks, each split is one CTA, so batch 1 with 4 KV heads
// still spreads over every SM; a CTA writes its split's normalised output with
// its max logit and exponential sum, and the splits are merged with
// log-sum-exp weights afterwards.  16 divides 784 = 49 x 16, 832 and 16, so a
// chunk never straddles a page and the 16-token tail of a 784-token page
// (784 = 12 x 64 + 16) is just the 49th chunk of the page ("DCU page832
// attention", Sec.2 and Sec.7).  The decode kernel is decode_mma.cuh.
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
    // Fused append (decode_append): the new token's rows [B, Hkv, D] bf16, written
    // into the cache slot of token L_b - 1 before the chunk holding it is copied;
    // nullptr for a plain decode.  k_cache / v_cache are the caches' base addresses.
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    uint8_t *k_cache;
    uint8_t *v_cache;
};

__device__ __forceinline__ void store_out(void *out, size_t idx, float v, int out_bf16) {
    if (out_bf16)
        reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float *>(out)[idx] = v;
}

// Four consecutive outputs from element idx (a multiple of 4): one 16-byte
// (fp32) or 8-byte (bf16) store.
__device__ __forceinline__ void store_out4(void *out, size_t idx, float4 v, int out_bf16) {
    if (out_bf16)
        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(out) + idx) =
            make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
    else
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + idx) = v;
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
    pdl_launch_dependents();  // a following attention call may start its set-up
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
    red_o[sg][qd] = a;
    if (qd == 0) red_ml[sg] = make_float2(M, W);
    const bool any_bad = __syncthreads_or(bad) != 0;  // a poisoned split anywhere zeroes the row
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
        const bool zero = any_bad || !(Wt > 0.f);
        const float inv = zero ? 0.f : 1.f / Wt;
        const size_t base = r * D + slice * 32 + qd * 4;
        store_out(p.out, base + 0, at.x * inv, p.out_bf16);
        store_out(p.out, base + 1, at.y * inv, p.out_bf16);
        store_out(p.out, base + 2, at.z * inv, p.out_bf16);
        store_out(p.out, base + 3, at.w * inv, p.out_bf16);
    }
}

// The same merge for few splits (S <= 8: verify, batched decode).  A warp
// merges PPW (row, head) pairs, a lane owning the 4-dim columns lane,
// lane + 32, ... of each (so a warp's load of one column set is 512
// contiguous bytes, and its stores are 16-byte vectors);
// every load of a warp is issued at once, so the kernel makes one dependent
// round trip and needs no shared-memory exchange.  Its CTAs reserve more than
// half of an SM's shared memory (kReduceSmallSmem, unused), so an SM holds at
// most one of them and none beside a split CTA: they land on SMs as the split
// CTAs leave, one per SM, and the grid is sized to about one CTA per SM.
// Packed several to an SM, small CTAs of this kind queued on that SM's share
// of L2 bandwidth while other SMs idled (the verify workload's 12.6 MB of
// partials: 5.9 us with 4 CTAs on each of 96 SMs).
constexpr int kReduceSmallMaxSplits = 8;
constexpr int kReduceSmallSmem = 120 * 1024;

template <int D, int NSL, int PPW>
__global__ void __launch_bounds__(256, 1) pa_split_reduce_small_kernel(const ReduceParams p, int pairs) {
    static_assert(NSL <= kReduceSmallMaxSplits && NSL * PPW <= 16, "slots held in registers");
    constexpr int E = D / 32;  // dims per lane
    pdl_launch_dependents();   // a following attention call may start its set-up
    pdl_wait_primary();        // partials of the split kernel are complete and visible
    const int pair0 = (blockIdx.x * 8 + (threadIdx.x >> 5)) * PPW, lane = threadIdx.x & 31;
    if (pair0 >= pairs) return;
    const int S = p.num_splits;
    float2 v[PPW][NSL];
    float4 o[PPW][NSL][E / 4];
#pragma unroll
    for (int j = 0; j < PPW; ++j) {  // all loads first, none behind a branch
        const int pair = min(pair0 + j, pairs - 1);
        const float2 *ml = p.part_ml + (size_t)pair * S;
        const float *po = p.part_o + (size_t)pair * S * D + 4 * lane;
#pragma unroll
        for (int u = 0; u < NSL; ++u) {
            const int i = min(u, S - 1);
            v[j][u] = ml[i];
#pragma unroll
            for (int e = 0; e < E / 4; ++e) o[j][u][e] = *reinterpret_cast<const float4 *>(po + (size_t)i * D + 128 * e);
        }
    }
#pragma unroll
    for (int j = 0; j < PPW; ++j) {
        if (pair0 + j >= pairs) break;
        float M = -INFINITY, W = 0.f;
        float4 a[E / 4];
#pragma unroll
        for (int e = 0; e < E / 4; ++e) a[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        bool bad = false;
#pragma unroll
        for (int u = 0; u < NSL; ++u) {
            if (u >= S) break;
            bad |= v[j][u].y < 0.f;
            if (!(v[j][u].y > 0.f)) continue;  // empty split (or poisoned, flagged above)
            const float Mn = fmaxf(M, v[j][u].x);
            const float c = fast_exp2(M - Mn), w = fast_exp2(v[j][u].x - Mn) * v[j][u].y;
            W = fmaf(W, c, w);
#pragma unroll
            for (int e = 0; e < E / 4; ++e) {
                a[e].x = fmaf(a[e].x, c, w * o[j][u][e].x);
                a[e].y = fmaf(a[e].y, c, w * o[j][u][e].y);
                a[e].z = fmaf(a[e].z, c, w * o[j][u][e].z);
                a[e].w = fmaf(a[e].w, c, w * o[j][u][e].w);
            }
            M = Mn;
        }
        const float inv = (bad || !(W > 0.f)) ? 0.f : 1.f / W;
        const size_t base = (size_t)(pair0 + j) * D + 4 * lane;
#pragma unroll
        for (int e = 0; e < E / 4; ++e)
            store_out4(p.out, base + 128 * e, make_float4(a[e].x * inv, a[e].y * inv, a[e].z * inv, a[e].w * inv),
                       p.out_bf16);
    }
}

}  // namespace pa
