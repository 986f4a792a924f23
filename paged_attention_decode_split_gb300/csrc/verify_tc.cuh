// verify_tc.cuh -- multi-row (speculative verify) paged attention on the
// sm_100-family tensor cores: tcgen05 MMAs with accumulators in tensor memory.
//
// What it computes ("Qwen3.8 on MI350P", Lektion 3: verify rows share K/V
// tiles, a causal mask applies per row, partial softmax statistics merge;
// "DCU page832 attention", Sec.5/7 for the paged walk): for the q_len new rows
// of a sequence, row r attends to keys 0 .. L - q_len + r.  All G * q_len query
// rows of one KV head form one M = 128 MMA block (row rho = r * G + g; rows
// past G * q_len are zero padding), so each K/V chunk is read from HBM once
// per CTA and consumed once by the tensor core for all rows.  The context is
// split across CTAs like decode; the same partition reduce merges the splits.
//
// Per 64-token tile i (four 16-token TMA chunks landing side by side):
//   S_i = Q K_i^T     M=128, N=64, K=D: D/16 MMAs with A = Q read from tensor
//                     memory, into one of two tensor-memory S buffers (tile
//                     i+1's scores are formed while the softmax warps work on
//                     tile i)
//   softmax           4 warps, one query row per thread (tensor-memory lane =
//                     row): scale, causal mask, running max and sum, P = 2^(s-m),
//                     written back over S_i in tensor memory
//   O += P_i V_i      M=128, N=D, K=16 per step (4 steps), A = P_i from tensor
//                     memory, carried as a bf16 head plus a bf16 residual (two
//                     MMAs) so it keeps ~16 significant bits
// The running max used for the exponentials is only raised when the row's
// max grows by more than 2^8 (then O and l are rescaled in place, after the
// previous tile's P.V product); otherwise P may exceed 1 by at most 2^8, which
// fp32 and the bf16 pair hold exactly enough, and the final division by l uses
// the same reference max.  Because O is touched only then, the softmax of tile
// i+1 overlaps the P.V product of tile i.
//
// Tensor memory (512 columns x 128 lanes): O fp32 in columns [0, D), NSB = 2
// S/P buffers of 64 columns from D on, and Q as bf16 pairs after them.
// Shared memory holds the K and V tiles in two rings (4 K and 3 V slots of
// 32 KiB for D = 256) and the split's block-table entries; a K slot is
// refilled once S_i is done:
//   K_i [D/64 blocks][64 tokens][128 B], 128-byte swizzle, K-major: one 5-D TMA
//       box of 64 tokens when the tile lies in one page, else 64-dim x 16-token
//       boxes per chunk
//   V_i same layout as K_i, read as the MN-major (N = d) B operand
// Warp roles: 0-3 softmax, 4 MMA issue (and tensor-memory allocation), 5 TMA
// (lane 0 decides, the whole warp issues a tile's boxes).
//
// fp8 e4m3 cache (NSG > 0): the copies land e4m3 tiles as [D/128 blocks][64
// tokens][128 B] with the 128-byte swizzle in a staging ring of NSG slots per
// tensor (so 8 lanes reading one 16-byte column of 8 consecutive tokens hit 8
// different bank groups), and four more warps
// widen them (warps 6-7: K, 8-9: V) into the same swizzled K/V rings as f16
// -- exact, since every e4m3 value is an f16 value -- zeroing rows past the
// tile's last key.  Q and P then enter the products as f16 (kind::f16 with
// f16 A and B), the K scale joins the softmax scale and the V scale the final
// normaliser.  A q row enters scaled by a power of two that brings its
// largest element into [2^14, 2^15), so any finite bf16 q fits f16; the
// inverse power joins the softmax scale.
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
    int early_kv;  // stream the context before the new rows ahead of the dependency wait
    int num_kv_heads;  // grid y = num_kv_heads x 128-row blocks
    int window;        // 0: full attention; W > 0: each row sees only its last W keys
    const float *k_scale;  // fp8 cache: [Hkv] dequantisation scales of K and V
    const float *v_scale;
};

// Byte offset of 16-byte column chunk c of row t in a [D/64][rows][128 B]
// tile written with the 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz_off(int t, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// Eight e4m3 codes (one 32-bit word each of four) -> eight f16 in 16 bytes.
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint32_t w0, uint32_t w1) {
    uint4 r;
    asm("{\n\t.reg .b16 a, b, c, d;\n\t"
        "mov.b32 {a, b}, %4;\n\tmov.b32 {c, d}, %5;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t"
        "cvt.rn.f16x2.e4m3x2 %2, c;\n\tcvt.rn.f16x2.e4m3x2 %3, d;\n\t}"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "r"(w0), "r"(w1));
    return r;
}

// Block-table entries a verify CTA stages in shared memory: with 16-token
// pages a 64-token tile spans 4 pages, and a page lookup per chunk from global
// memory would put a dependent load in front of every copy.
constexpr int kVerifyPageTab = 256;

namespace tc {

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]: A's M = 128 rows are the tensor-memory
// lanes, its K elements packed two per 32-bit column.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives on the mbarrier when every MMA issued so far by this thread is done.
__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets, descriptor version 1, layout (0: no swizzle, 2: 128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(layout & 7u) << 61;
    return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, A and B both bf16
// (ab_f16 = false) or both f16, A K-major, B K-major (b_mn = 0) or MN-major
// (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn, bool ab_f16 = false) {
    return (1u << 4) | (ab_f16 ? 0u : (1u << 7) | (1u << 10)) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}
// 16 consecutive fp32 columns, without waiting (tcgen05.wait::ld before use).
__device__ __forceinline__ void ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace tc

// NSB: S/P tensor-memory buffers (the Q K^T products run up to NSB tiles ahead
// of P V).  TK: keys per score tile, 64 or 128.  With 128 the score product
// S = Q K^T is M = 128 x N = 128: half as many MMA instructions per key as with
// N = 64, whose instruction rate bounds the tile when the tiles come from L2
// (many row blocks per KV head, chunked prefill), and P V runs over two 64-key
// V tiles per score tile.  At D = 256 two 128-column S/P buffers and O fill
// tensor memory, so Q moves to shared memory as the product's A operand (QSM)
// and the K ring holds one 128-key tile; at D = 128 Q stays in tensor memory.
template <int D, int NK, int NV, int NSG = 0, int NSB = 2, int TK = 64>
struct VerifyTcCfg {
    static constexpr bool F8 = NSG > 0;                // fp8 cache: e4m3 staging ring of NSG slots per tensor
    static constexpr bool QSM = TK == 128 && D == 256;  // Q in shared memory
    static constexpr int M = 128;                      // MMA rows (query rows, zero padded)
    static constexpr int TT = 64;                      // tokens per V tile (4 TMA chunks)
    static constexpr int CPT = TT / kChunk;            // chunks per V tile
    static constexpr int CPK = TK / kChunk;            // chunks per K (score) tile
    static constexpr int VPK = TK / TT;                // V tiles per score tile
    static constexpr int DB = D / 64;                  // 128-byte column blocks
    static constexpr int TILE_BYTES = TT * D * 2;      // V of one tile (bf16 or f16)
    static constexpr int KTILE_BYTES = TK * D * 2;     // K of one score tile
    static constexpr int KVB = F8 ? 1 : 2;             // bytes per cached element
    static constexpr int CHUNK_BYTES = kChunk * D * KVB;  // one TMA chunk as copied
    static constexpr int STG_BYTES = TT * D;           // one e4m3 tile, [D/128][64 tokens][128 B] swizzled
    static constexpr int OFF_V = NK * KTILE_BYTES;      // K ring, then V ring
    static constexpr int OFF_STG = OFF_V + NV * TILE_BYTES;  // K staging, then V staging
    static constexpr int OFF_Q = OFF_STG + 2 * NSG * STG_BYTES;  // QSM: Q as [D/64][M rows][128 B], swizzled
    static constexpr int Q_BYTES = QSM ? M * D * 2 : 0;
    static constexpr int OFF_BAR = OFF_Q + Q_BYTES;
    // k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_full[NSB], p_full[NSB], o_done[NSB], mma_fin,
    // then (fp8) kst_full[NSG], kst_empty[NSG], vst_full[NSG], vst_empty[NSG]
    static constexpr int OFF_TMEM = OFF_BAR + (2 * NK + 2 * NV + 3 * NSB + 1 + 4 * NSG) * 8;
    static constexpr int OFF_FLAGS = OFF_TMEM + 16;
    static constexpr int OFF_PT = OFF_FLAGS + 16;                    // the split's block-table entries
    static constexpr int SMEM_BYTES = OFF_PT + kVerifyPageTab * 4 + 1024;
    // tensor-memory columns: O (fp32, D), NSB S/P buffers (TK each), Q (bf16
    // pairs, D / 2; not with QSM).  P of a score tile is written over its S
    // buffer, per 64-key half: a bf16 head in 32 columns, then the residual in 32.
    static constexpr int TMEM_COLS = 512;
    static constexpr int O_COL = 0;
    static constexpr int S_COL = D;
    static constexpr int Q_COL = D + NSB * TK;
    static constexpr int Q_TCOLS = QSM ? 0 : D / 2;
    static constexpr int SBUF(int j) { return S_COL + j * TK; }
    static constexpr int CW = 2;                       // fp8: widening warps per tensor
    static constexpr int SROW = D * 4 + 16;            // epilogue: output rows staged in the K/V rings
    static_assert(M * SROW <= OFF_STG, "the staged output rows fit in the K/V rings");
    static constexpr int THREADS = (F8 ? 6 + 2 * CW : 6) * 32;
    static_assert(D == 256 || D == 128, "head_dim 256 or 128");
    static_assert(Q_COL + Q_TCOLS <= TMEM_COLS, "tensor-memory columns");
    static_assert(TK == 64 || (TK == 128 && !F8), "128-key score tiles: bf16 cache only");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// NSG > 0: fp8 cache (tm_k / tm_v: e4m3 boxes of 128 codes x 16 tokens,
// tm_k64 / tm_v64: 5-D boxes of a whole 64-token tile, both with the 128-byte
// swizzle).
// tm_k64: 5-D boxes of a whole K tile of TK keys (64, or 128 with TK = 128).
template <int D, int NK, int NV, int NSG, int NSB, int TK = 64>
__global__ void __launch_bounds__(VerifyTcCfg<D, NK, NV, NSG, NSB, TK>::THREADS, 1)
    pa_verify_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_k64, const __grid_constant__ CUtensorMap tm_v64,
                        const VerifyParams p) {
    using C = VerifyTcCfg<D, NK, NV, NSG, NSB, TK>;
    constexpr bool F8 = C::F8, QSM = C::QSM;
    constexpr int TT = C::TT, CPT = C::CPT, CPK = C::CPK, VPK = C::VPK;
    constexpr float kLazy = 8.f;  // raise the reference max only when it grows by more than 2^8
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    // K and V tiles have their own rings: a K slot is free again as soon as
    // S_i = Q K_i^T is done, long before O += P_i V_i releases the V slot.
    uint64_t *k_full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *k_empty = k_full + NK;
    uint64_t *v_full = k_empty + NK;
    uint64_t *v_empty = v_full + NV;
    uint64_t *s_full = v_empty + NV;   // [NSB]: S_i written (buffer i % NSB)
    uint64_t *p_full = s_full + NSB;   // [NSB]: P_i written by the softmax warps
    uint64_t *o_done = p_full + NSB;   // [NSB]: O += P_i V_i finished
    uint64_t *mma_fin = o_done + NSB;
    uint64_t *kst_full = mma_fin + 1;  // fp8: e4m3 tile landed in a staging slot
    uint64_t *kst_empty = kst_full + NSG;  // fp8: staging slot widened, free again
    uint64_t *vst_full = kst_empty + NSG;
    uint64_t *vst_empty = vst_full + NSG;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::OFF_FLAGS);  // [0] abort, [1] bad page
    int32_t *page_tab = reinterpret_cast<int32_t *>(smem + C::OFF_PT);

    const int split = blockIdx.x, b = blockIdx.z;
    const int kvh = blockIdx.y % p.num_kv_heads;
    // Row blocks launch last-first: later blocks see more keys (causal), so the
    // longest CTAs go out in the first wave and a partial last wave holds the
    // shortest ones.
    const int n_blocks = gridDim.y / p.num_kv_heads;
    const int row0 = (n_blocks - 1 - (int)(blockIdx.y / p.num_kv_heads)) * C::M;  // first row (rho = r G + g)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group, R = min(C::M, p.q_len * G - row0);  // rows of this block

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        // a K/V ring slot is filled by the copy engine (one expect-tx arrival),
        // or with an fp8 cache by the CW widening warps of its tensor
        for (int s = 0; s < NK; ++s) {
            mbar_init(&k_full[s], F8 ? C::CW : 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(&v_full[s], F8 ? C::CW : 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int j = 0; j < NSB; ++j) {
            mbar_init(&s_full[j], 1);
            mbar_init(&p_full[j], 128);
            mbar_init(&o_done[j], 1);
        }
        mbar_init(mma_fin, 1);
        for (int s = 0; s < NSG; ++s) {
            mbar_init(&kst_full[s], 1);
            mbar_init(&kst_empty[s], C::CW);
            mbar_init(&vst_full[s], 1);
            mbar_init(&vst_empty[s], C::CW);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    if (warp == 5 && lane == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_k64);
        prefetch_tensormap(&tm_v64);
    }
    // This row's q goes to L2 ahead of the dependency wait: L2 is where global
    // memory is kept coherent, so a row the work before this call is still
    // writing is read in its final state after the wait all the same.
    const int rho_q = row0 + (int)threadIdx.x;  // the softmax threads' rows (rows past R are zero padding)
    const __nv_bfloat16 *qrow =
        p.q + (((size_t)b * p.q_len + rho_q / G) * p.num_q_heads + kvh * G + rho_q % G) * D;
    if (warp < 4 && (int)threadIdx.x < R) {
#pragma unroll
        for (int o = 0; o < D * 2; o += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(qrow) + o));
    }
    // Every global access waits for the work before this call on the stream,
    // except with early_kv: then the block table, seq_lens and the tiles that
    // end before the new rows are read first (see the producer below).
    if (!p.early_kv) pdl_wait_primary();

    int L = p.seq_lens[b];
    const bool bad_len = L < 0 || L > p.max_seq_len || L < p.q_len;
    if (bad_len) {
        if (threadIdx.x == 0 && split == 0 && kvh == 0) set_status(p.status, PA_DEV_BAD_SEQLEN);
        L = 0;
    }
    const int n_chunks = (L + kChunk - 1) / kChunk;
    // with a sliding window the splits start at the chunk of the block's first
    // visible key (its first row's window start)
    const int k_first = p.window > 0 ? max(0, L - p.q_len + row0 / G - p.window + 1) : 0;
    const int c_begin = k_first / kChunk + split * p.chunks_per_split;
    // keys past the block's last row's causal limit are never read
    const int k_last = L - p.q_len + (row0 + R - 1) / G;
    const int n_my = min(min(n_chunks, k_last / kChunk + 1) - c_begin, p.chunks_per_split);
    if (n_my <= 0) {
        // No key of this sequence in this split: an empty record (m = -inf,
        // l = 0) for the reduce, or zero rows when the call is unsplit.
        if (p.early_kv) pdl_wait_primary();
        if (p.num_splits == 1) {
            for (int idx = threadIdx.x; idx < R * D; idx += C::THREADS) {
                const int rho = row0 + idx / D, d = idx % D;
                const size_t row = (size_t)b * p.q_len + rho / G;
                store_out(p.out, (row * p.num_q_heads + kvh * G + rho % G) * D + d, 0.f, p.out_bf16);
            }
        } else {
            for (int rho = row0 + threadIdx.x; rho < row0 + R; rho += C::THREADS) {
                const size_t row = (size_t)b * p.q_len + rho / G;
                p.part_ml[(row * p.num_q_heads + kvh * G + rho % G) * p.num_splits + split] =
                    make_float2(-INFINITY, 0.f);
            }
        }
        return;
    }
    const int n_tiles = (n_my + CPK - 1) / CPK;   // score tiles (K tiles)
    const int n_vtiles = (n_my + CPT - 1) / CPT;  // V tiles (VPK per score tile)

    // The split's block-table entries, staged in shared memory by all threads
    // (visible to the producer after the next __syncthreads); splits spanning
    // more pages read the table from global memory.
    const int32_t *bt = p.block_table + (size_t)b * p.max_pages_per_seq;
    const int lp_first = (c_begin * kChunk) / p.block_size;
    const int n_pt = ((c_begin + n_my) * kChunk - 1) / p.block_size - lp_first + 1;
    const bool staged = n_pt <= kVerifyPageTab;
    if (staged)
        for (int j = threadIdx.x; j < n_pt; j += C::THREADS) page_tab[j] = bt[lp_first + j];

    // TMA copies of one tile of K (CPK chunks) or of V (CPT chunks), issued by
    // the whole producer warp: lane 0 arms the barrier; a tile inside one page
    // is one 5-D box (lane 0), otherwise lane c * NB + b copies column block b
    // of chunk c, so a tile over 16-token pages (16 boxes per tensor for
    // D = 256) costs no more issue time than one box.
    int issued_k = 0, issued_v = 0;
    auto issue_tile = [&](int i, int tensor, uint64_t policy) {
        constexpr int NB = F8 ? D / 128 : C::DB;  // boxes per 16-token chunk (128-byte columns)
        constexpr int BW = F8 ? 128 : 64;         // elements per box row
        const int s = F8 ? i % (NSG > 0 ? NSG : 1) : (tensor == 0 ? i % NK : i % NV);
        uint64_t *bar = F8 ? (tensor == 0 ? &kst_full[s] : &vst_full[s]) : (tensor == 0 ? &k_full[s] : &v_full[s]);
        uint8_t *dst0 = F8 ? smem + C::OFF_STG + (tensor * NSG + s) * C::STG_BYTES
                           : smem + (tensor == 0 ? s * C::KTILE_BYTES : C::OFF_V + s * C::TILE_BYTES);
        const CUtensorMap *m4 = tensor == 0 ? &tm_k : &tm_v;
        const CUtensorMap *m5 = tensor == 0 ? &tm_k64 : &tm_v64;
        const int cpt = tensor == 0 ? CPK : CPT, tt = cpt * kChunk;  // chunks and tokens per tile
        const int nc = min(cpt, n_my - i * cpt);  // chunks in this tile
        if (lane == 0) mbar_arrive_expect_tx(bar, nc * C::CHUNK_BYTES);
        __syncwarp();
        auto page_of = [&](int lp) {
            const int page = staged ? page_tab[lp - lp_first] : bt[lp];
            if (page < 0 || (int64_t)page >= p.num_pages) {
                flags[1] = 1;  // the copy reads zeros (box outside the tensor)
                set_status(p.status, PA_DEV_BAD_PAGE);
            }
            return page;
        };
        const int t00 = (c_begin + i * cpt) * kChunk;
        const int lp0 = t00 / p.block_size, off0 = t00 - lp0 * p.block_size;
        if (nc == cpt && off0 + tt <= p.block_size) {
            // the whole tile lies in one page: one copy lands it as [blocks][tt tokens][128 B]
            if (lane == 0) tma_load_5d(dst0, m5, bar, 0, off0, 0, kvh, page_of(lp0), policy);
        } else if (lane < nc * NB) {
            const int c = lane / NB, db = lane % NB;
            const int t0 = t00 + c * kChunk, lp = t0 / p.block_size;
            tma_load_4d(dst0 + db * tt * 128 + c * kChunk * 128, m4, bar, db * BW, kvh, t0 - lp * p.block_size,
                        page_of(lp), policy);
        }
        __syncwarp();
    };
    static_assert(CPK * (F8 ? D / 128 : C::DB) <= 32, "a lane per box of a tile");
    // tiles that end before the new rows (early_kv reads only those before the wait)
    auto before_new_rows = [&](int i, int cpt) {
        return (c_begin + i * cpt + min(cpt, n_my - i * cpt)) * kChunk <= L - p.q_len;
    };
    if (p.early_kv) {
        __syncthreads();  // barrier initialisation and the page table are visible to the producer warp
        if (warp == 5) {
            // first use of each slot: tiles that end before the new rows
            const uint64_t policy = l2_policy_evict_first();
            constexpr int FK = F8 ? NSG : NK, FV = F8 ? NSG : NV;  // slots the copies land in
            while (issued_k < min(FK, n_tiles) && before_new_rows(issued_k, CPK)) issue_tile(issued_k++, 0, policy);
            while (issued_v < min(FV, n_vtiles) && before_new_rows(issued_v, CPT)) issue_tile(issued_v++, 1, policy);
        }
        pdl_wait_primary();
    }

    // Q rows: each softmax thread loads its row (D / 8 16-byte words, one
    // round of loads) right after the dependency wait, so the loads are in
    // flight while tensor memory is allocated.
    constexpr int NQ = D / 8;
    uint4 qv[NQ];
    if (warp < 4) {
        const bool qlive = (int)threadIdx.x < R;
#pragma unroll
        for (int v = 0; v < NQ; ++v)
            qv[v] = qlive ? *reinterpret_cast<const uint4 *>(qrow + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (warp == 4) {
        tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    // The tensor-memory address reaches the softmax and MMA warps (0-4).  With
    // early_kv the other warps synchronised ahead of the wait (barriers, page
    // table) and go on streaming; without it this is their synchronisation.
    if (p.early_kv) {
        if (warp < 5) named_bar_sync(2, 160);
    } else {
        __syncthreads();
    }
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;  // (read by warps 0-4 only on the early_kv path)
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's tensor-memory lanes

    // Q block -> tensor memory, the A operand of S = Q K^T: row rho in lane
    // rho, dims packed two per column (column c holds elements 2c and 2c + 1);
    // padding rows are zero.  The softmax warps store it while the producer
    // already streams K and V; only the MMA warp waits for it (named barrier
    // 1: warps 0-4).  Over an fp8 cache the products run in f16, and each row
    // enters scaled by q_pre, the power of two that brings its largest element
    // into [2^14, 2^15) (f16_prescale).
    float q_pre = 1.f;
    if (warp < 4) {
        if constexpr (F8) {  // the products run in f16: Q too
            uint32_t amax = 0;
#pragma unroll
            for (int v = 0; v < NQ; ++v)
                amax = max(max(amax, max(bf16x2_absmax(qv[v].x), bf16x2_absmax(qv[v].y))),
                           max(bf16x2_absmax(qv[v].z), bf16x2_absmax(qv[v].w)));
            q_pre = f16_prescale(amax);
#pragma unroll
            for (int v = 0; v < NQ; ++v)
                qv[v] = make_uint4(bf16x2_to_f16x2_scaled(qv[v].x, q_pre), bf16x2_to_f16x2_scaled(qv[v].y, q_pre),
                                   bf16x2_to_f16x2_scaled(qv[v].z, q_pre), bf16x2_to_f16x2_scaled(qv[v].w, q_pre));
        }
        if constexpr (QSM) {
            // row rho of the block at [D/64 column blocks][M rows][128 B], 16-byte unit u of a
            // row stored at unit u ^ (row % 8): the K-major operand layout with the 128-byte swizzle
            const int r = threadIdx.x;
#pragma unroll
            for (int v = 0; v < NQ; ++v)
                *reinterpret_cast<uint4 *>(smem + C::OFF_Q + (v / 8) * (C::M * 128) + r * 128 +
                                           (((v % 8) ^ (r % 8)) << 4)) = qv[v];
            tc::fence_async_smem();  // the rows are read by the tensor core
        } else {
#pragma unroll
            for (int c = 0; c < NQ / 8; ++c) {
                uint32_t r[32];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    r[4 * v] = qv[8 * c + v].x;
                    r[4 * v + 1] = qv[8 * c + v].y;
                    r[4 * v + 2] = qv[8 * c + v].z;
                    r[4 * v + 3] = qv[8 * c + v].w;
                }
                tc::st32(lane_base + C::Q_COL + 32 * c, r);
            }
            tc::wait_st();
        }
        tc::fence_before();
        asm volatile("bar.arrive 1, 160;" ::: "memory");
    } else if (warp == 4) {
        asm volatile("bar.sync 1, 160;" ::: "memory");
        tc::fence_after();
    }

    if (warp == 5) {
        // ---------------- producer: TMA copies of K and V, 4 chunks per tile ----------------
        // Two rings refilled independently: lane 0 probes the next slot of
        // each without blocking and the warp issues the tile; within a ring
        // tiles go in order.  Every decision is lane 0's, so the warp stays
        // converged.
        const uint64_t policy = l2_policy_evict_first();
        uint32_t idle = 0;
        // the slots the copies land in: the K/V rings, or the fp8 staging rings
        constexpr int FK = F8 ? NSG : NK, FV = F8 ? NSG : NV;
        uint64_t *ke = F8 ? kst_empty : k_empty;
        uint64_t *ve = F8 ? vst_empty : v_empty;
        while (issued_k < n_tiles || issued_v < n_vtiles) {
            bool go_k = false, go_v = false;
            if (lane == 0) {
                go_k = issued_k < n_tiles &&
                       (issued_k < FK || mbar_test_wait(&ke[issued_k % FK], ((issued_k / FK) - 1) & 1));
                go_v = issued_v < n_vtiles &&
                       (issued_v < FV || mbar_test_wait(&ve[issued_v % FV], ((issued_v / FV) - 1) & 1));
            }
            go_k = __shfl_sync(0xffffffffu, go_k, 0);
            go_v = __shfl_sync(0xffffffffu, go_v, 0);
            if (go_k) issue_tile(issued_k++, 0, policy);
            if (go_v) issue_tile(issued_v++, 1, policy);
            if (go_k || go_v) {
                idle = 0;
            } else {
                const bool stop = __shfl_sync(0xffffffffu, ++idle > kWaitPollLimit || flags[0] != 0, 0);
                if (stop) {
                    if (lane == 0) flags[0] = 1;
                    break;
                }
            }
        }
        if (lane == 0 && flags[0]) {
            // let the copies in flight land before the CTA ends
            uint64_t *kf = F8 ? kst_full : k_full;
            uint64_t *vf = F8 ? vst_full : v_full;
            for (int i = max(0, issued_k - FK); i < issued_k; ++i)
                for (uint32_t n = 0; n < kWaitPollLimit && !mbar_try_wait(&kf[i % FK], (i / FK) & 1); ++n) {
                }
            for (int i = max(0, issued_v - FV); i < issued_v; ++i)
                for (uint32_t n = 0; n < kWaitPollLimit && !mbar_try_wait(&vf[i % FV], (i / FV) & 1); ++n) {
                }
            set_status(p.status, PA_DEV_TIMEOUT);
        }
    } else if (warp == 4) {
        // ---------------- MMA issue: one lane ----------------
        if (lane == 0) {
            constexpr uint32_t kIdQK = tc::idesc_bf16(128, TK, 0, F8);
            constexpr uint32_t kIdPV = tc::idesc_bf16(128, D, 1, F8);
            // Event loop: each product is issued as soon as its own inputs are
            // ready -- O += P_i V_i when the softmax warps have written P_i,
            // S_i = Q K_i^T when tile i has landed and P_{i-2}, which shares
            // S_i's columns, has been consumed.  The tensor core runs this
            // thread's MMAs in issue order, so S_i never overwrites P_{i-2}
            // before O += P_{i-2} V_{i-2} has read it.
            int next_qk = 0, next_pv = 0;
            uint32_t idle = 0;
            bool ok = true;
            while (next_pv < n_tiles) {
                bool progress = false;
                // the V tiles of score tile next_pv (VPK, fewer at a split's end) have landed
                auto v_ready = [&](int i) {
                    if constexpr (VPK == 1) {
                        return mbar_test_wait(&v_full[i % NV], (i / NV) & 1);
                    } else {
                        const int nvt = min(VPK, n_vtiles - i * VPK);
                        for (int h2 = 0; h2 < nvt; ++h2) {
                            const int vt = i * VPK + h2;
                            if (!mbar_test_wait(&v_full[vt % NV], (vt / NV) & 1)) return false;
                        }
                        return true;
                    }
                };
                if (next_pv < next_qk && mbar_test_wait(&p_full[next_pv % NSB], (next_pv / NSB) & 1) &&
                    v_ready(next_pv)) {
                    const int i = next_pv, j = i % NSB;
                    const int nvt = VPK == 1 ? 1 : min(VPK, n_vtiles - i * VPK);
                    tc::fence_after();
#pragma unroll 1
                    for (int h2 = 0; h2 < nvt; ++h2) {
                        const int vt = i * VPK + h2;
                        const uint32_t v_addr = smem_addr(smem + C::OFF_V + (vt % NV) * C::TILE_BYTES);
#pragma unroll
                        for (int ks = 0; ks < TT / 16; ++ks) {
                            // V: MN-major; 64-dim blocks TT x 128 B apart (LBO), 8-token groups 1 KiB apart (SBO)
                            const uint64_t bdesc = tc::sdesc(v_addr + ks * 16 * 128, TT * 128, 1024, 2);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                // P (head, then residual) of this 64-key half: 16 tokens = 8 columns per step
                                const uint32_t a_tm = tmem + C::SBUF(j) + h2 * TT + h * (TT / 2) + ks * 8;
                                tc::mma_bf16_ta(tmem + C::O_COL, a_tm, bdesc, kIdPV,
                                                (i > 0 || h2 > 0 || ks > 0 || h > 0) ? 1u : 0u);
                            }
                        }
                        tc::commit(&v_empty[vt % NV]);
                    }
                    tc::commit(&o_done[j]);
                    ++next_pv;
                    progress = true;
                }
                if (next_qk < n_tiles && next_qk - next_pv < NSB) {
                    const int i = next_qk, s = i % NK, j = i % NSB;
                    if (mbar_test_wait(&k_full[s], (i / NK) & 1)) {
                        tc::fence_after();
                        const uint32_t k_addr = smem_addr(smem + s * C::KTILE_BYTES);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            // 16-element k steps: +32 B inside a 128-byte swizzle row, next 64-dim block further on
                            const uint32_t koff = (kk >> 2) * (TK * 128) + (kk & 3) * 32;
                            if constexpr (QSM) {  // Q from shared memory, laid out like K with M rows
                                const uint32_t qoff = (kk >> 2) * (C::M * 128) + (kk & 3) * 32;
                                tc::mma_bf16(tmem + C::SBUF(j), tc::sdesc(smem_addr(smem + C::OFF_Q) + qoff, 16, 1024, 2),
                                             tc::sdesc(k_addr + koff, 16, 1024, 2), kIdQK, kk > 0 ? 1u : 0u);
                            } else {
                                tc::mma_bf16_ta(tmem + C::SBUF(j), tmem + C::Q_COL + kk * 8,
                                                tc::sdesc(k_addr + koff, 16, 1024, 2), kIdQK, kk > 0 ? 1u : 0u);
                            }
                        }
                        tc::commit(&k_empty[s]);
                        tc::commit(&s_full[j]);
                        ++next_qk;
                        progress = true;
                    }
                }
                if (progress) {
                    idle = 0;
                } else if (++idle > kWaitPollLimit || flags[0]) {
                    ok = false;
                    break;
                }
            }
            if (!ok) {
                flags[0] = 1;
                set_status(p.status, PA_DEV_TIMEOUT);
            }
            // Whatever happened, let every issued MMA finish before tensor
            // memory is released at the end of the CTA.
            tc::commit(mma_fin);
            for (uint32_t n = 0; n < kWaitPollLimit && !mbar_try_wait(mma_fin, 0); ++n) {
            }
        }
    } else if (warp >= 6) {
        if constexpr (F8) {
            // ---------------- fp8: widen staged e4m3 tiles into the K (warps 6, 7) / V (8, 9) ring ----------------
            const int tensor = (warp - 6) / C::CW, part = (warp - 6) % C::CW;
            constexpr int NR0 = NK, NR1 = NV;
            const int NR = tensor == 0 ? NR0 : NR1;
            uint64_t *ring_full = tensor == 0 ? k_full : v_full;
            uint64_t *ring_empty = tensor == 0 ? k_empty : v_empty;
            uint64_t *stg_full = tensor == 0 ? kst_full : vst_full;
            uint64_t *stg_empty = tensor == 0 ? kst_empty : vst_empty;
            uint8_t *ring = smem + (tensor == 0 ? 0 : C::OFF_V);
            const uint8_t *stg = smem + C::OFF_STG + tensor * NSG * C::STG_BYTES;
            const int t_end = min(L, (c_begin + n_my) * kChunk);
            // A lane widens 16 codes -- 16-byte column j of 128-code block b of
            // token t -- into two 16-byte f16 chunks of the swizzled ring row.
            // The 8 lanes of a shared-memory phase take 8 consecutive tokens of
            // one column (t & 7 = lane & 7), so both the staged reads and the
            // ring writes spread over the 8 bank groups; a lane then walks its
            // column down the tile in steps of 8 tokens (1 KiB in both layouts).
            constexpr int QG = D / 64;  // groups of 4 columns: warp `part` takes every CW-th
            const int t_lo = lane & 7, q_lo = lane >> 3;
            for (int i = 0; i < n_tiles; ++i) {
                // the staged tile has landed, and the ring slot's previous tile has been consumed
                bool ok = __all_sync(0xffffffffu, mbar_wait(&stg_full[i % NSG], (i / NSG) & 1, &flags[0]));
                if (ok && i >= NR)
                    ok = __all_sync(0xffffffffu, mbar_wait(&ring_empty[i % NR], ((i / NR) - 1) & 1, &flags[0]));
                if (!ok) {
                    flags[0] = 1;
                    break;
                }
                const int nvl = min(TT, t_end - (c_begin + i * CPT) * kChunk) - t_lo;  // rows t < nv hold keys
                const uint8_t *stg_tile = stg + (i % NSG) * C::STG_BYTES;
                uint8_t *ring_tile = ring + (i % NR) * C::TILE_BYTES;
                for (int qg = part; qg < QG; qg += C::CW) {
                    const int q = 4 * qg + q_lo, b = q >> 3, j = q & 7, c = (q & 3) * 2;
                    const uint8_t *src = stg_tile + b * (TT * 128) + t_lo * 128 + ((j ^ t_lo) << 4);
                    uint8_t *dst = ring_tile + (q >> 2) * (TT * 128) + t_lo * 128;
                    const int o_lo = (c ^ t_lo) << 4, o_hi = ((c + 1) ^ t_lo) << 4;
#pragma unroll
                    for (int u = 0; u < TT / 8; ++u) {
                        uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
                        if (8 * u < nvl) {
                            const uint4 w = *reinterpret_cast<const uint4 *>(src + u * 1024);
                            lo = e4m3x8_to_f16x8(w.x, w.y);
                            hi = e4m3x8_to_f16x8(w.z, w.w);
                        }
                        *reinterpret_cast<uint4 *>(dst + u * 1024 + o_lo) = lo;
                        *reinterpret_cast<uint4 *>(dst + u * 1024 + o_hi) = hi;
                    }
                }
                tc::fence_async_smem();  // the tensor core reads the widened tile
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&ring_full[i % NR]);
                    mbar_arrive(&stg_empty[i % NSG]);
                }
            }
        }
    } else {
        // ---------------- softmax: thread = query row = tensor-memory lane ----------------
        const int rho = row0 + threadIdx.x;  // this thread's row (tensor-memory lane threadIdx.x)
        const bool live = (int)threadIdx.x < R;
        // last visible key: the causal limit of the row, and never past this
        // split's last chunk (a tile may reach into the next split's tokens)
        const int t_end = min(L, (c_begin + n_my) * kChunk);
        const int lim = live ? min(L - p.q_len + rho / G, t_end - 1) : -1;
        const int lo = p.window > 0 ? L - p.q_len + rho / G - p.window + 1 : 0;  // first key of the row's window
        // fp8: K's scale and the inverse of q's pre-scale (a power of two) join the softmax scale
        const float sl = F8 ? p.scale_log2 * p.k_scale[kvh] * (1.f / q_pre) : p.scale_log2;
        float m_ref = -INFINITY, l_sum = 0.f;
        bool ok = true;
        // O += P_k V_k of tile k is waited for in order per barrier (tile k +
        // NSB, where it is long finished), so no wait ever tests a phase parity
        // two phases behind the barrier.
        auto wait_pv = [&](int k) {
            return __all_sync(0xffffffffu, mbar_wait(&o_done[k % NSB], (k / NSB) & 1, &flags[0]));
        };
        for (int i = 0; i < n_tiles; ++i) {
            const int j = i % NSB;
            // waits ahead of a warp-collective tensor-memory access end the same way for the whole warp
            if (!__all_sync(0xffffffffu, mbar_wait(&s_full[j], (i / NSB) & 1, &flags[0]))) {
                ok = false;
                break;
            }
            // A 64-key tile keeps its scores in registers from the max to the
            // exponentials (one load); a 128-key tile takes its max over both
            // halves first and loads each half again for P (the one-load form
            // for 128 keys would not fit the registers, and the two-pass form
            // makes the fp8 variants spill).
            if constexpr (VPK == 1) {
                tc::fence_after();
                float sv[TT];
                {
                    uint32_t r[TT / 16][16];  // the tile's scores: all loads in flight, one wait
#pragma unroll
                    for (int c0 = 0; c0 < TT / 16; ++c0) tc::ld16_nowait(lane_base + C::SBUF(j) + 16 * c0, r[c0]);
                    tc::wait_ld();
#pragma unroll
                    for (int c = 0; c < TT; ++c) sv[c] = __uint_as_float(r[c / 16][c % 16]);
                }
                if (i >= NSB && !wait_pv(i - NSB)) {
                    ok = false;
                    break;
                }

                const int t0 = (c_begin + i * CPT) * kChunk;
                float mx = -INFINITY;
                // the exponent is 2^(sv * mul - m): raw scores with mul = scale when
                // every key of the tile is visible to this row (no mask, and the
                // max of the scaled scores is the scaled max for scale > 0), else
                // scaled and masked scores with mul = 1
                float mul = 1.f;
                if (sl > 0.f && t0 + TT - 1 <= lim && t0 >= lo) {
                    float mr = sv[0];
#pragma unroll
                    for (int c = 1; c + 1 < TT; c += 2) mr = fmax3(mr, sv[c], sv[c + 1]);
                    mr = fmaxf(mr, sv[TT - 1]);
                    mx = mr * sl;
                    mul = sl;
                } else {
#pragma unroll
                    for (int c = 0; c < TT; ++c) sv[c] = (t0 + c <= lim && t0 + c >= lo) ? sv[c] * sl : -INFINITY;
#pragma unroll
                    for (int c = 0; c < TT; c += 2) mx = fmax3(mx, sv[c], sv[c + 1]);
                }
                // lazy rescale: only when the max grows by more than 2^kLazy, and
                // then only after the previous tile's P.V product has finished
                const bool raise = mx > m_ref + kLazy;
                const bool need_rescale = raise && m_ref != -INFINITY;
                if (__any_sync(0xffffffffu, need_rescale)) {
                    if (!wait_pv(i - 1)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const float alpha = need_rescale ? fast_exp2(m_ref - mx) : 1.f;
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 16) {
                        float ov[16];
                        tc::ld16(lane_base + C::O_COL + c0, ov);
#pragma unroll
                        for (int c = 0; c < 16; ++c) ov[c] *= alpha;
                        tc::st16(lane_base + C::O_COL + c0, ov);
                    }
                    if (need_rescale) l_sum *= alpha;
                }
                if (raise) m_ref = mx;
                // The tile may be short or end in a partial chunk: V rows past the
                // end hold stale data (even NaN), and 0 * NaN would reach O through
                // the tensor core, so zero them before the P.V product reads them.
                const int nv = min(TT, t_end - t0);
                if (!F8 && nv < TT) {  // (fp8: the widening warp writes those rows as zeros)
                    if (!__all_sync(0xffffffffu, mbar_wait(&v_full[i % NV], (i / NV) & 1, &flags[0]))) {
                        ok = false;
                        break;
                    }
                    uint8_t *vst = smem + C::OFF_V + (i % NV) * C::TILE_BYTES;
                    for (int idx = threadIdx.x; idx < (TT - nv) * C::DB * 8; idx += 128) {
                        const int t = nv + idx / (C::DB * 8), rem = idx % (C::DB * 8);
                        *reinterpret_cast<uint4 *>(vst + (rem >> 3) * (TT * 128) + t * 128 + (rem & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    tc::fence_async_smem();  // zeroed V rows are read by the tensor core
                }
                // P = 2^(s - m) as a bf16 head and a bf16 residual, written over S_i
                // (tokens packed two per column: head in the first 32 columns)
                // with no visible key yet (m = -inf) every p is 0: 2^(x - inf)
                const float m_use = m_ref == -INFINITY ? INFINITY : m_ref;
                float2 ps2 = make_float2(0.f, 0.f);
                uint32_t hw[TT / 2], lw[TT / 2];
#pragma unroll
                for (int c = 0; c < TT / 2; ++c) {
                    const float p0 = fast_exp2(fmaf(sv[2 * c], mul, -m_use));
                    const float p1 = fast_exp2(fmaf(sv[2 * c + 1], mul, -m_use));
                    ps2 = __fadd2_rn(ps2, make_float2(p0, p1));
                    if constexpr (F8)
                        split_f16(p0, p1, hw[c], lw[c]);
                    else
                        split_bf16(p0, p1, hw[c], lw[c]);
                }
                l_sum += ps2.x + ps2.y;
                tc::st32(lane_base + C::SBUF(j), hw);
                tc::st32(lane_base + C::SBUF(j) + TT / 2, lw);
                tc::wait_st();
                tc::fence_before();
            } else {
                tc::fence_after();
                const int t0 = (c_begin + i * CPK) * kChunk;        // first key of the score tile
                const int nvt = min(VPK, n_vtiles - i * VPK);       // its 64-key halves with keys of this split
                // The exponent is 2^(sv * mul - m): raw scores with mul = scale when
                // every key of the tile is visible to this row (no mask, and the
                // max of the scaled scores is the scaled max for scale > 0), else
                // scaled and masked scores with mul = 1.
                const bool all_visible = sl > 0.f && t0 + TK - 1 <= lim && t0 >= lo;
                const float mul = all_visible ? sl : 1.f;
                // 64 scores of half h2 (all loads in flight, one wait), masked and scaled unless all_visible
                float sv[TT];
                auto load_half = [&](int h2) {
                    uint32_t r[TT / 16][16];
#pragma unroll
                    for (int c0 = 0; c0 < TT / 16; ++c0)
                        tc::ld16_nowait(lane_base + C::SBUF(j) + h2 * TT + 16 * c0, r[c0]);
                    tc::wait_ld();
#pragma unroll
                    for (int c = 0; c < TT; ++c) sv[c] = __uint_as_float(r[c / 16][c % 16]);
                    if (!all_visible) {
                        const int th = t0 + h2 * TT;
#pragma unroll
                        for (int c = 0; c < TT; ++c) sv[c] = (th + c <= lim && th + c >= lo) ? sv[c] * sl : -INFINITY;
                    }
                };
                auto half_max = [&]() {
                    float mh;
                    if (all_visible) {
                        mh = sv[0];
#pragma unroll
                        for (int c = 1; c + 1 < TT; c += 2) mh = fmax3(mh, sv[c], sv[c + 1]);
                        mh = fmaxf(mh, sv[TT - 1]) * sl;
                    } else {
                        mh = -INFINITY;
#pragma unroll
                        for (int c = 0; c < TT; c += 2) mh = fmax3(mh, sv[c], sv[c + 1]);
                    }
                    return mh;
                };
                float mx = -INFINITY;
                for (int h2 = 0; h2 < nvt; ++h2) {  // the tile's max, over every half
                    load_half(h2);
                    mx = fmaxf(mx, half_max());
                }
                if (i >= NSB && !wait_pv(i - NSB)) {
                    ok = false;
                    break;
                }
                // lazy rescale: only when the max grows by more than 2^kLazy, and
                // then only after the previous tile's P.V product has finished
                const bool raise = mx > m_ref + kLazy;
                const bool need_rescale = raise && m_ref != -INFINITY;
                if (__any_sync(0xffffffffu, need_rescale)) {
                    if (!wait_pv(i - 1)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const float alpha = need_rescale ? fast_exp2(m_ref - mx) : 1.f;
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 16) {
                        float ov[16];
                        tc::ld16(lane_base + C::O_COL + c0, ov);
#pragma unroll
                        for (int c = 0; c < 16; ++c) ov[c] *= alpha;
                        tc::st16(lane_base + C::O_COL + c0, ov);
                    }
                    if (need_rescale) l_sum *= alpha;
                }
                if (raise) m_ref = mx;
                // A V tile may be short or end in a partial chunk: V rows past the
                // end hold stale data (even NaN), and 0 * NaN would reach O through
                // the tensor core, so zero them before the P.V product reads them.
                bool zero_ok = true;
                for (int h2 = 0; h2 < nvt && !F8; ++h2) {  // (fp8: the widening warp writes those rows as zeros)
                    const int vt = i * VPK + h2;
                    const int nv = min(TT, t_end - (t0 + h2 * TT));
                    if (nv >= TT) continue;
                    if (!__all_sync(0xffffffffu, mbar_wait(&v_full[vt % NV], (vt / NV) & 1, &flags[0]))) {
                        zero_ok = false;
                        break;
                    }
                    uint8_t *vst = smem + C::OFF_V + (vt % NV) * C::TILE_BYTES;
                    for (int idx = threadIdx.x; idx < (TT - nv) * C::DB * 8; idx += 128) {
                        const int t = nv + idx / (C::DB * 8), rem = idx % (C::DB * 8);
                        *reinterpret_cast<uint4 *>(vst + (rem >> 3) * (TT * 128) + t * 128 + (rem & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    tc::fence_async_smem();  // zeroed V rows are read by the tensor core
                }
                if (!zero_ok) {
                    ok = false;
                    break;
                }
                // P = 2^(s - m) per 64-key half as a bf16 head and a bf16 residual,
                // written over that half's S columns (tokens packed two per column:
                // head in the first 32 columns); with no visible key yet (m = -inf)
                // every p is 0: 2^(x - inf)
                const float m_use = m_ref == -INFINITY ? INFINITY : m_ref;
                for (int h2 = 0; h2 < nvt; ++h2) {
                    if (VPK > 1) load_half(h2);  // (one half: its scores are still in sv)
                    float2 ps2 = make_float2(0.f, 0.f);
                    uint32_t hw[TT / 2], lw[TT / 2];
#pragma unroll
                    for (int c = 0; c < TT / 2; ++c) {
                        const float p0 = fast_exp2(fmaf(sv[2 * c], mul, -m_use));
                        const float p1 = fast_exp2(fmaf(sv[2 * c + 1], mul, -m_use));
                        ps2 = __fadd2_rn(ps2, make_float2(p0, p1));
                        if constexpr (F8)
                            split_f16(p0, p1, hw[c], lw[c]);
                        else
                            split_bf16(p0, p1, hw[c], lw[c]);
                    }
                    l_sum += ps2.x + ps2.y;
                    tc::st32(lane_base + C::SBUF(j) + h2 * TT, hw);
                    tc::st32(lane_base + C::SBUF(j) + h2 * TT + TT / 2, lw);
                }
                tc::wait_st();
                tc::fence_before();
            }
            mbar_arrive(&p_full[j]);
        }
        // Epilogue: wait for the last P.V MMA, normalise and write this row.
        if (ok && !wait_pv(n_tiles - 1)) ok = false;
        ok = __all_sync(0xffffffffu, ok);  // the loads below are warp-collective
        if (!ok) flags[0] = 1;
        tc::fence_after();
        const bool poisoned = !ok || flags[1] != 0;
        const float inv = (poisoned || !(l_sum > 0.f)) ? 0.f : (F8 ? p.v_scale[kvh] : 1.f) / l_sum;
        const size_t orow = live ? ((size_t)b * p.q_len + rho / G) * p.num_q_heads + kvh * G + rho % G : 0;
        const bool direct = p.num_splits == 1;  // the final output, else this split's record
        if (ok) {
            // Every tile has been consumed by the tensor core, so the K/V rings
            // are free: the row is staged there (rows SROW bytes apart, so the
            // 16-byte stores of 8 consecutive rows fall in 8 different bank
            // groups) and leaves with one bulk copy, instead of a warp's 32
            // rows going out as 32 separate segments per store.
            const bool bf = direct && p.out_bf16;
            uint8_t *srow = smem + threadIdx.x * C::SROW;
#pragma unroll 1
            for (int c1 = 0; c1 < D; c1 += 64) {
                uint32_t r[4][16];  // 64 columns: four loads in flight, one wait
#pragma unroll
                for (int k = 0; k < 4; ++k) tc::ld16_nowait(lane_base + C::O_COL + c1 + 16 * k, r[k]);
                tc::wait_ld();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int c0 = c1 + 16 * k;
                    float ov[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) ov[c] = __uint_as_float(r[k][c]) * inv;
                    if (bf) {
                        uint32_t w[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c) w[c] = pack_bf16(ov[2 * c], ov[2 * c + 1]);
                        *reinterpret_cast<uint4 *>(srow + 2 * c0) = make_uint4(w[0], w[1], w[2], w[3]);
                        *reinterpret_cast<uint4 *>(srow + 2 * c0 + 16) = make_uint4(w[4], w[5], w[6], w[7]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 16; c += 4)
                            *reinterpret_cast<float4 *>(srow + 4 * (c0 + c)) =
                                make_float4(ov[c], ov[c + 1], ov[c + 2], ov[c + 3]);
                    }
                }
            }
            if (live) {
                tc::fence_async_smem();  // the staged row is read by the copy engine
                uint8_t *dst = direct ? static_cast<uint8_t *>(p.out) + orow * D * (bf ? 2 : 4)
                                      : reinterpret_cast<uint8_t *>(p.part_o + (orow * p.num_splits + split) * D);
                bulk_store_s2g(dst, srow, bf ? D * 2 : D * 4);
                bulk_commit();
                bulk_wait_read();  // the row has left shared memory before the CTA ends
            }
        } else if (live) {
            // a wait was abandoned (copies may still land in the rings): zero the row with plain stores
#pragma unroll 1
            for (int c = 0; c < D; ++c) {
                if (direct)
                    store_out(p.out, orow * D + c, 0.f, p.out_bf16);
                else
                    p.part_o[(orow * p.num_splits + split) * D + c] = 0.f;
            }
        }
        if (live && !direct)
            p.part_ml[orow * p.num_splits + split] = make_float2(m_ref, poisoned ? -1.f : l_sum);
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 4) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace pa
