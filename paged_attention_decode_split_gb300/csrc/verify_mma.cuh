// verify_mma.cuh -- multi-row (speculative verify) paged attention with the
// GQA rows of one KV head sharing every K/V tile on the tensor cores.
//
// What it computes ("Qwen3.8 on MI350P", Lektion 3: verify rows share K/V
// tiles, a causal mask applies per row, partial softmax statistics merge;
// "DCU page832 attention", Sec.5/7 for the paged walk): for the q_len new rows
// of a sequence, row r attends to keys 0 .. L - q_len + r.  All G * q_len query
// rows of one KV head form one M <= 128 block (row index rho = r * G + g), so a
// K/V chunk is read once per CTA for all of them.  The context is split
// across CTAs exactly like decode; the same partition reduce merges splits.
//
// This is the mma.sync (m16n8k16, bf16 in, fp32 accumulate) version: one
// consumer warp per 16-row slice, S = Q K^T and O += P V per 16-token chunk,
// with P carried as a bf16 head plus a bf16 residual in the second product.  K and V
// chunks arrive by TMA with the 128-byte swizzle so ldmatrix reads are free
// of bank conflicts.
#pragma once

#include "decode_split.cuh"

namespace pa {

struct VerifyParams {
    const __nv_bfloat16 *q;  // [B * q_len, Hq, D]
    const int32_t *block_table;
    const int32_t *seq_lens;
    void *out;
    float *part_o;
    float2 *part_ml;
    int32_t *status;
    int64_t num_pages;
    int num_q_heads;
    int q_len;
    int group;  // G
    int max_pages_per_seq;
    int max_seq_len;
    int block_size;
    int chunks_per_split;
    int num_splits;
    float scale_log2;
    int out_bf16;
};

template <int D, int NWC, int NS>
struct VerifyCfg {
    static constexpr int RP = NWC * 16;               // padded rows (<= 128)
    static constexpr int DB = D / 64;                 // 128-byte column blocks
    static constexpr int CHUNK_BYTES = kChunk * D * 2;
    static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;
    static constexpr int Q_BYTES = RP * D * 2;
    static constexpr int OFF_Q = NS * STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_Q + Q_BYTES;
    static constexpr int OFF_FLAGS = OFF_BAR + 2 * NS * 8;
    static constexpr int SMEM_BYTES = OFF_FLAGS + 16 + 1024;
    static constexpr int THREADS = (NWC + 1) * 32;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// Byte offset of 16-byte column chunk c of row t in a [D/64][rows][128 B]
// tile written with the 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz_off(int t, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// x = head + residual with both parts in bf16 (packed pairs for elements a, b).
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t &head, uint32_t &resid) {
    head = pack_bf16(a, b);
    const float ha = __uint_as_float(head << 16), hb = __uint_as_float(head & 0xffff0000u);
    resid = pack_bf16(a - ha, b - hb);
}

template <int D, int NWC, int NS>
__global__ void __launch_bounds__((NWC + 1) * 32, 1)
    pa_verify_mma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const VerifyParams p) {
    using C = VerifyCfg<D, NWC, NS>;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint8_t *qs = smem + C::OFF_Q;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + NS;
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::OFF_FLAGS);

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group, R = p.q_len * G;

    pdl_launch_dependents();

    int L = p.seq_lens[b];
    bool bad_len = L < 0 || L > p.max_seq_len || L < p.q_len;
    if (bad_len) {
        if (threadIdx.x == 0 && split == 0 && kvh == 0) set_status(p.status, PA_DEV_BAD_SEQLEN);
        L = 0;
    }
    const int n_chunks = (L + kChunk - 1) / kChunk;
    const int c_begin = split * p.chunks_per_split;
    const int n_my = min(n_chunks - c_begin, p.chunks_per_split);
    if (n_my <= 0) {
        if (p.num_splits == 1) {
            for (int idx = threadIdx.x; idx < R * D; idx += C::THREADS) {
                const int rho = idx / D, d = idx - rho * D;
                const size_t row = (size_t)b * p.q_len + rho / G;
                store_out(p.out, (row * p.num_q_heads + kvh * G + rho % G) * D + d, 0.f, p.out_bf16);
            }
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NWC);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    // Q block -> shared (swizzled [D/64][RP][128 B]); padding rows are zero.
    for (int idx = threadIdx.x; idx < C::RP * (D / 8); idx += C::THREADS) {
        const int rho = idx / (D / 8), c = idx - rho * (D / 8);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (rho < R) {
            const size_t row = (size_t)b * p.q_len + rho / G;
            v = *reinterpret_cast<const uint4 *>(p.q + (row * p.num_q_heads + kvh * G + rho % G) * D + c * 8);
        }
        *reinterpret_cast<uint4 *>(qs + swz_off(rho, c, C::RP)) = v;
    }
    __syncthreads();

    if (warp == NWC) {
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
                if (lp != cur_lp) {
                    cur_lp = lp;
                    page = bt[lp];
                    if (page < 0 || (int64_t)page >= p.num_pages) {
                        flags[1] = 1;
                        set_status(p.status, PA_DEV_BAD_PAGE);
                    }
                }
                const int off = t0 - lp * p.block_size;
                uint8_t *st = smem + s * C::STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
#pragma unroll
                for (int db = 0; db < C::DB; ++db) {
                    tma_load_4d(st + db * kChunk * 128, &tm_k, &full[s], db * 64, kvh, off, page, policy);
                    tma_load_4d(st + C::CHUNK_BYTES + db * kChunk * 128, &tm_v, &full[s], db * 64, kvh, off, page,
                                policy);
                }
                issued = i + 1;
            }
            if (flags[0]) {
                for (int i = max(0, issued - NS); i < issued; ++i) {
                    uint64_t *bar = &full[i % NS];
                    for (uint32_t n = 0; n < kWaitPollLimit && !mbar_try_wait(bar, (i / NS) & 1); ++n) {
                    }
                }
                set_status(p.status, PA_DEV_TIMEOUT);
            }
        }
        __syncthreads();
        return;
    }

    // ---------------- consumer warp: rows 16*warp .. 16*warp+15 ----------------
    const int gq = lane >> 2, tq = lane & 3;
    const int rho_lo = warp * 16 + gq, rho_hi = rho_lo + 8;
    // last visible key of each of the two rows this thread holds (-1: none / padding)
    const int lim_lo = rho_lo < R ? L - p.q_len + rho_lo / G : -1;
    const int lim_hi = rho_hi < R ? L - p.q_len + rho_hi / G : -1;
    const uint32_t qbase = smem_addr(qs);

    float o[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

    for (int i = 0; i < n_my; ++i) {
        const int s = i % NS;
        if (!mbar_wait(&full[s], (i / NS) & 1, &flags[0])) {
            flags[0] = 1;
            break;
        }
        const uint32_t kb = smem_addr(smem + s * C::STAGE_BYTES);
        const uint32_t vb = kb + C::CHUNK_BYTES;
        const int t0 = (c_begin + i) * kChunk;

        // S = Q K^T for 16 rows x 16 tokens (two n-tiles of 8 tokens)
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            {
                const int mi = lane >> 3;
                const int row = warp * 16 + (mi & 1) * 8 + (lane & 7);
                ldsm_x4(qbase + swz_off(row, kk * 2 + (mi >> 1), C::RP), a0, a1, a2, a3);
            }
            {
                const int mi = lane >> 3;
                const int tok = (mi >> 1) * 8 + (lane & 7);
                ldsm_x4(kb + swz_off(tok, kk * 2 + (mi & 1), kChunk), b0, b1, b2, b3);
            }
            mma_bf16(sacc[0], a0, a1, a2, a3, b0, b1);
            mma_bf16(sacc[1], a0, a1, a2, a3, b2, b3);
        }
        // scale to log2 units, causal mask per row, online softmax
        float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int t = t0 + nt * 8 + tq * 2 + c;
                const float slo = t <= lim_lo ? sacc[nt][c] * p.scale_log2 : -INFINITY;
                const float shi = t <= lim_hi ? sacc[nt][2 + c] * p.scale_log2 : -INFINITY;
                sacc[nt][c] = slo;
                sacc[nt][2 + c] = shi;
                mx_lo = fmaxf(mx_lo, slo);
                mx_hi = fmaxf(mx_hi, shi);
            }
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
        const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
        // a row with no visible key so far keeps m = -inf; use 0 as its shift
        const float sh_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
        const float sh_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
        const float al_lo = fast_exp2(m_lo - sh_lo), al_hi = fast_exp2(m_hi - sh_hi);
        m_lo = mn_lo;
        m_hi = mn_hi;
        float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                sacc[nt][c] = fast_exp2(sacc[nt][c] - sh_lo);
                sacc[nt][2 + c] = fast_exp2(sacc[nt][2 + c] - sh_hi);
                ps_lo += sacc[nt][c];
                ps_hi += sacc[nt][2 + c];
            }
        l_lo = fmaf(l_lo, al_lo, ps_lo);
        l_hi = fmaf(l_hi, al_hi, ps_hi);
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            o[j][0] *= al_lo;
            o[j][1] *= al_lo;
            o[j][2] *= al_hi;
            o[j][3] *= al_hi;
        }
        // P as the A operand: the two S n-tiles are exactly one k=16 slice.  P is
        // split into a bf16 head and a bf16 residual (two products), so the
        // probabilities keep about 16 significant bits instead of bf16's 8.
        uint32_t ph[4], pl[4];
        split_bf16(sacc[0][0], sacc[0][1], ph[0], pl[0]);
        split_bf16(sacc[0][2], sacc[0][3], ph[1], pl[1]);
        split_bf16(sacc[1][0], sacc[1][1], ph[2], pl[2]);
        split_bf16(sacc[1][2], sacc[1][3], ph[3], pl[3]);
        // rows of V past the end of the sequence may hold anything (NaN):
        // zero them in the B fragments of the last, partial chunk
        const int nv = min(kChunk, L - t0);
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
            uint32_t b0, b1, b2, b3;
            const int mi = lane >> 3;
            const int tok = (mi & 1) * 8 + (lane & 7);
            ldsm_x4_t(vb + swz_off(tok, jj * 2 + (mi >> 1), kChunk), b0, b1, b2, b3);
            if (nv < kChunk) {
                const int k0 = tq * 2;  // b0/b2 hold tokens k0, k0+1; b1/b3 tokens k0+8, k0+9
                const uint32_t m0 = (k0 < nv ? 0x0000ffffu : 0u) | (k0 + 1 < nv ? 0xffff0000u : 0u);
                const uint32_t m1 = (k0 + 8 < nv ? 0x0000ffffu : 0u) | (k0 + 9 < nv ? 0xffff0000u : 0u);
                b0 &= m0;
                b2 &= m0;
                b1 &= m1;
                b3 &= m1;
            }
            mma_bf16(o[2 * jj], ph[0], ph[1], ph[2], ph[3], b0, b1);
            mma_bf16(o[2 * jj + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
            mma_bf16(o[2 * jj], pl[0], pl[1], pl[2], pl[3], b0, b1);
            mma_bf16(o[2 * jj + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    __syncthreads();  // pairs with the producer warp's

    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    const bool poisoned = flags[0] != 0 || flags[1] != 0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int rho = half ? rho_hi : rho_lo;
        if (rho >= R) continue;
        const float l = half ? l_hi : l_lo, m = half ? m_hi : m_lo;
        const float inv = (poisoned || !(l > 0.f)) ? 0.f : 1.f / l;
        const size_t orow = ((size_t)b * p.q_len + rho / G) * p.num_q_heads + kvh * G + rho % G;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            const int d = j * 8 + tq * 2;
            const float v0 = o[j][half * 2] * inv, v1 = o[j][half * 2 + 1] * inv;
            if (p.num_splits == 1) {
                store_out(p.out, orow * D + d, v0, p.out_bf16);
                store_out(p.out, orow * D + d + 1, v1, p.out_bf16);
            } else {
                *reinterpret_cast<float2 *>(p.part_o + (orow * p.num_splits + split) * D + d) = make_float2(v0, v1);
            }
        }
        if (p.num_splits > 1 && tq == 0)
            p.part_ml[orow * p.num_splits + split] = make_float2(m, poisoned ? -1.f : l);
    }
}

}  // namespace pa
