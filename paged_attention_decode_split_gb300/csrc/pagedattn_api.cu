// pagedattn_api.cu -- the C ABI: argument validation, split planning, TMA
// descriptors, and the reshape_and_cache kernel.
//
// Split planning follows the split-KV fix of "Hybrid SSM decode rate on dual
// Radeon under vLLM": with one CTA per (sequence, KV head) a batch-1 decode of
// a 4-KV-head model leaves most SMs idle, so each (sequence, KV head) context
// is cut into S splits of whole 16-token chunks, enough that the grid
// (S, Hkv, B) covers every SM; the partition reduce then merges the splits.
// More splits cost more partial traffic and a longer reduce (the grid-versus-
// partials trade-off that "Qwen3.8 on MI350P" spells out for split-K GEMMs),
// so a split never drops below kMinChunksPerSplit chunks.  The plan depends
// only on the description and the SM count, so it is deterministic.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/pagedattn.h"
#include "pa_internal.h"

namespace pa {

namespace {

// 64 tokens: at 1K tokens, 16 splits of 4 chunks take 5.12 us per hybrid call
// against 5.63 us for 32 of 2 (500 tokens: 5.00 against 5.04 us); from 2K up
// and for the dense shape the plan is the same either way
constexpr int kMinChunksPerSplit = 4;
constexpr int kMaxChunksPerSplit = 256; // 4096 tokens: bounds the longest CTA for load balance
constexpr int kMaxDevices = 64;
constexpr int kKernelSlots = 160;

thread_local pa_plan_info g_last_plan;
thread_local bool g_have_plan = false;

struct Plan {
    int num_sms;
    int num_splits;
    int chunks_per_split;
    size_t ws_bytes;
    size_t off_part_ml;  // workspace: split outputs [rows, S, D] fp32, then (max, sum) [rows, S] from here
};

inline size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sm_count(int *out) {
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0) {
        *out = cache[dev];
        return 0;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
    if (dev >= 0 && dev < kMaxDevices) cache[dev] = n;
    *out = n;
    return 0;
}

// Validates a description; `verify` selects the q_len rule.
pa_status check_desc(const pa_attn_desc *d, bool verify) {
    if (!d) return PA_ERR_INVALID_ARG;
    if (d->num_seqs < 0 || d->q_len < 1 || d->num_q_heads < 1 || d->num_kv_heads < 1 || d->head_dim < 1 ||
        d->block_size < 1 || d->max_pages_per_seq < 0 || d->max_seq_len < 0 || d->num_pages < 1 ||
        d->num_splits < 0 || d->num_sms < 0 || (d->flags & ~PA_FLAG_EARLY_KV_READ) != 0 || d->window < 0)
        return PA_ERR_INVALID_ARG;
    if (!verify && d->q_len != 1) return PA_ERR_INVALID_ARG;
    if (d->num_q_heads % d->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (d->out_dtype != PA_OUT_F32 && d->out_dtype != PA_OUT_BF16) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(d->scale)) return PA_ERR_INVALID_ARG;
    const int64_t need_pages = (static_cast<int64_t>(d->max_seq_len) + d->block_size - 1) / d->block_size;
    if (need_pages > d->max_pages_per_seq) return PA_ERR_INVALID_ARG;
    if (d->num_pages > INT32_MAX) return PA_ERR_UNSUPPORTED;  // TMA coordinates are 32-bit
    // grid.z = num_seqs (split kernels), grid.y = num_seqs * q_len (reduce), grid.y = Hkv x row blocks
    if (static_cast<int64_t>(d->num_seqs) * d->q_len > 65535 || d->num_kv_heads > 65535)
        return PA_ERR_UNSUPPORTED;
    if (verify && static_cast<int64_t>(d->num_kv_heads) *
                          ((static_cast<int64_t>(d->q_len) * (d->num_q_heads / d->num_kv_heads) + 127) / 128) >
                      65535)
        return PA_ERR_UNSUPPORTED;
    if (d->block_size % kChunk != 0) return PA_ERR_UNSUPPORTED;
    const int group = d->num_q_heads / d->num_kv_heads;
    if (verify) {
        if (!verify_supported(d->head_dim, d->q_len * group)) return PA_ERR_UNSUPPORTED;
    } else {
        if (!decode_supported(d->head_dim, group)) return PA_ERR_UNSUPPORTED;
    }
    return PA_OK;
}

pa_status make_plan(const pa_attn_desc *d, bool verify, Plan *pl) {
    pa_status st = check_desc(d, verify);
    if (st != PA_OK) return st;
    int sms = d->num_sms;
    if (sms <= 0 && device_sm_count(&sms) != 0) return PA_ERR_CUDA;
    int n_chunks = (d->max_seq_len + kChunk - 1) / kChunk;
    // with a sliding window a unit reads at most window + q_len - 1 keys, from
    // a chunk-aligned start: the splits cover that span only
    if (d->window > 0)
        n_chunks = static_cast<int>(std::min<int64_t>(
            n_chunks, (static_cast<int64_t>(d->window) + d->q_len - 1 + kChunk - 1) / kChunk + 1));
    // verify: each (sequence, KV head) unit has ceil(q_len G / 128) row blocks of its own
    const int64_t row_blocks =
        verify ? (static_cast<int64_t>(d->q_len) * (d->num_q_heads / d->num_kv_heads) + 127) / 128 : 1;
    const int64_t units = static_cast<int64_t>(d->num_seqs) * d->num_kv_heads * row_blocks;
    int splits;
    if (d->num_splits > 0) {
        splits = d->num_splits;
    } else if (units == 0 || n_chunks == 0) {
        splits = 1;
    } else {
        // as many splits as whole waves allow: a grid of units x splits CTAs
        // never spills a few CTAs into a second wave
        splits = static_cast<int>(std::max<int64_t>(1, sms / units));
        splits = std::min(splits, std::max(1, n_chunks / kMinChunksPerSplit));
        // decode: long contexts are cut further to bound the longest CTA (a
        // batch of mixed lengths then balances over several waves).  Verify
        // CTAs carry a large fixed cost (Q into tensor memory, the pipeline
        // fill), so verify stays at whole waves: for 8 sequences x 16 rows of
        // the 32/8/128 shape, 2 splits (128 CTAs) take 74 us where the 3 the
        // rule asks for (192 CTAs) take 100 us.
        if (units < sms && !verify)
            splits = std::max(splits, (n_chunks + kMaxChunksPerSplit - 1) / kMaxChunksPerSplit);
    }
    splits = std::max(1, std::min(splits, std::max(1, n_chunks)));
    int cps = std::max(1, (n_chunks + splits - 1) / splits);
    if (verify) cps = (cps + 3) & ~3;  // the tensor-core path walks 64-token tiles: splits of whole tiles
    splits = std::max(1, (n_chunks + cps - 1) / cps);  // no trailing empty split for the longest sequence
    pl->num_sms = sms;
    pl->num_splits = splits;
    pl->chunks_per_split = cps;
    pl->ws_bytes = pl->off_part_ml = 0;
    if (splits > 1) {
        const size_t rows = static_cast<size_t>(d->num_seqs) * d->q_len * d->num_q_heads;
        pl->off_part_ml = round256(rows * splits * d->head_dim * sizeof(float));
        pl->ws_bytes = pl->off_part_ml + rows * splits * sizeof(float2);
    }
    return PA_OK;
}

// ---- TMA descriptors of a [P, BS, Hkv, D] bf16 or fp8 cache -----------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Encoded tensor maps are kept per host thread: a serving loop passes the same
// cache tensors every step, and an encode costs microseconds of host time.  A
// map depends only on the key (address and geometry), so a hit is exact.
struct MapKey {
    const void *base;
    int64_t num_pages;
    int32_t block_size, num_kv_heads, head_dim, box_d, kind;  // kind 0: chunk box of box_d dims; 1: 5-D column-block box of box_d tokens
    bool swizzle128, fp8;
    bool operator==(const MapKey &o) const {
        return base == o.base && num_pages == o.num_pages && block_size == o.block_size &&
               num_kv_heads == o.num_kv_heads && head_dim == o.head_dim && box_d == o.box_d && kind == o.kind &&
               swizzle128 == o.swizzle128 && fp8 == o.fp8;
    }
};
struct MapEntry {
    CUtensorMap map;
    MapKey key;
    bool valid;
};
constexpr int kMapCache = 64;
thread_local MapEntry g_maps[kMapCache];
thread_local int g_map_next = 0;

template <typename Encode>
bool cached_map(CUtensorMap *map, const MapKey &key, Encode encode) {
    for (const MapEntry &e : g_maps)
        if (e.valid && e.key == key) {
            *map = e.map;
            return true;
        }
    if (!encode(map)) return false;
    g_maps[g_map_next].map = *map;
    g_maps[g_map_next].key = key;
    g_maps[g_map_next].valid = true;
    g_map_next = (g_map_next + 1) % kMapCache;
    return true;
}

// Box = [box_d elements of d, 1 head, 16 tokens, 1 page]; fp8: one-byte elements.
bool encode_cache_map_uncached(CUtensorMap *map, const void *base, const pa_attn_desc *d, int box_d,
                               bool swizzle128, bool fp8) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)d->head_dim, (cuuint64_t)d->num_kv_heads, (cuuint64_t)d->block_size,
                                (cuuint64_t)d->num_pages};
    const cuuint64_t row = (cuuint64_t)d->head_dim * (fp8 ? 1 : 2);
    const cuuint64_t strides[3] = {row, row * d->num_kv_heads, row * d->num_kv_heads * d->block_size};
    const cuuint32_t box[4] = {(cuuint32_t)box_d, 1, (cuuint32_t)kChunk, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                    const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 5-D view for the tensor-core paths: {128-byte column block, tokens, blocks,
// head, page}; one box of {block, `tokens` tokens, all blocks, 1, 1} lands in
// shared memory as [blocks][tokens][128 B] with the 128-byte swizzle -- the
// K-major (and MN-major) operand layout the tcgen05 MMA reads, and the layout
// in which ldmatrix rows never share a bank group -- in a single copy.
// Verify copies 64-token tiles, decode 16-token chunks.  bf16: 64-dim blocks;
// fp8: 128-code blocks.
bool encode_cache_map_blocks_uncached(CUtensorMap *map, const void *base, const pa_attn_desc *d, bool fp8,
                                      int tokens) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    const int esz = fp8 ? 1 : 2, blk = 128 / esz;
    const cuuint64_t row = (cuuint64_t)d->head_dim * esz;
    const cuuint64_t dims[5] = {(cuuint64_t)blk, (cuuint64_t)d->block_size, (cuuint64_t)(d->head_dim / blk),
                                (cuuint64_t)d->num_kv_heads, (cuuint64_t)d->num_pages};
    const cuuint64_t strides[4] = {row * d->num_kv_heads, 128, row, row * d->num_kv_heads * d->block_size};
    const cuuint32_t box[5] = {(cuuint32_t)blk, (cuuint32_t)tokens, (cuuint32_t)(d->head_dim / blk), 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                    const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_cache_map(CUtensorMap *map, const void *base, const pa_attn_desc *d, int box_d, bool swizzle128,
                      bool fp8 = false) {
    const MapKey key{base, d->num_pages, d->block_size, d->num_kv_heads, d->head_dim, box_d, 0, swizzle128, fp8};
    return cached_map(map, key, [&](CUtensorMap *m) {
        return encode_cache_map_uncached(m, base, d, box_d, swizzle128, fp8);
    });
}

bool encode_cache_map_blocks(CUtensorMap *map, const void *base, const pa_attn_desc *d, bool fp8 = false,
                             int tokens = 64) {
    const MapKey key{base, d->num_pages, d->block_size, d->num_kv_heads, d->head_dim, tokens, 1, true, fp8};
    return cached_map(map, key,
                      [&](CUtensorMap *m) { return encode_cache_map_blocks_uncached(m, base, d, fp8, tokens); });
}

void record_plan(int path, const Plan &pl, const pa_attn_desc *d, int ctas) {
    g_last_plan.path_id = path;
    g_last_plan.num_splits = pl.num_splits;
    g_last_plan.chunks_per_split = pl.chunks_per_split;
    g_last_plan.grid_ctas = ctas;
    g_last_plan.block_size = d->block_size;
    g_last_plan.reduce_launched = pl.num_splits > 1 ? 1 : 0;
    g_have_plan = true;
}

pa_status check_common_ptrs(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                            const int32_t *seq_lens, const void *out) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out) return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

pa_status check_workspace(const Plan &pl, void *workspace, size_t ws_bytes) {
    if (pl.ws_bytes == 0) return PA_OK;
    if (!workspace || ws_bytes < pl.ws_bytes || !aligned16(workspace)) return PA_ERR_WORKSPACE;
    return PA_OK;
}

}  // namespace

cudaError_t ensure_smem_limit(const void *fn, int bytes, int slot) {
    static bool done[kMaxDevices][kKernelSlots] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= kKernelSlots)
        return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev][slot]) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[dev][slot] = true;
    return e;
}

// ---- reshape_and_cache kernel ------------------------------------------------
// One CTA per new token copies its [Hkv, D] rows of K and V into the slot's
// cache row with 16-byte vector accesses.
__global__ void __launch_bounds__(128) pa_reshape_and_cache_kernel(const uint4 *__restrict__ k_new,
                                                                   const uint4 *__restrict__ v_new,
                                                                   uint4 *__restrict__ k_cache,
                                                                   uint4 *__restrict__ v_cache,
                                                                   const int64_t *__restrict__ slots, int row_vecs,
                                                                   int64_t num_slots, int32_t *status) {
    pdl_launch_dependents();  // the attention kernel behind may start its set-up
    pdl_wait_primary();       // the work before it on the stream has finished
    const int i = blockIdx.x;
    const int64_t s = slots[i];
    if (s < 0) return;  // padding token
    if (s >= num_slots) {
        if (threadIdx.x == 0) set_status(status, PA_DEV_BAD_SLOT);
        return;
    }
    const uint4 *ks = k_new + (size_t)i * row_vecs;
    const uint4 *vs = v_new + (size_t)i * row_vecs;
    uint4 *kd = k_cache + (size_t)s * row_vecs;
    uint4 *vd = v_cache + (size_t)s * row_vecs;
    for (int j = threadIdx.x; j < row_vecs; j += blockDim.x) {
        kd[j] = ks[j];
        vd[j] = vs[j];
    }
}

// fp8 variant: a thread turns 8 bf16 of a row into 8 e4m3 codes, code =
// e4m3(x / scale[kv head]) with the division in binary32, rounding to nearest
// even and saturating to +-448 (cvt ... satfinite).
__global__ void __launch_bounds__(128) pa_reshape_and_cache_fp8_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new, uint2 *__restrict__ k_cache,
    uint2 *__restrict__ v_cache, const int64_t *__restrict__ slots, const float *__restrict__ k_scale,
    const float *__restrict__ v_scale, int row_vecs, int head_vecs, int64_t num_slots, int32_t *status) {
    pdl_launch_dependents();
    pdl_wait_primary();
    const int i = blockIdx.x;
    const int64_t s = slots[i];
    if (s < 0) return;
    if (s >= num_slots) {
        if (threadIdx.x == 0) set_status(status, PA_DEV_BAD_SLOT);
        return;
    }
    const uint4 *ks = k_new + (size_t)i * row_vecs;
    const uint4 *vs = v_new + (size_t)i * row_vecs;
    uint2 *kd = k_cache + (size_t)s * row_vecs;
    uint2 *vd = v_cache + (size_t)s * row_vecs;
    for (int j = threadIdx.x; j < row_vecs; j += blockDim.x) {
        const int h = j / head_vecs;
        kd[j] = e4m3x8_div(ks[j], k_scale[h]);
        vd[j] = e4m3x8_div(vs[j], v_scale[h]);
    }
}

pa_status decode_call(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                      const float *v_scale, const int32_t *block_table, const int32_t *seq_lens,
                      const pa_attn_desc *desc, void *out, void *workspace, size_t workspace_bytes,
                      int32_t *device_status, void *stream, const void *k_new = nullptr,
                      const void *v_new = nullptr);
pa_status verify_call(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                      const float *v_scale, const int32_t *block_table, const int32_t *seq_lens,
                      const pa_attn_desc *desc, void *out, void *workspace, size_t workspace_bytes,
                      int32_t *device_status, void *stream);

}  // namespace pa

using namespace pa;

extern "C" {

const char *pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG: invalid argument";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: shape outside the compiled kernels";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
        case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA call or launch failed";
    }
    return "unknown pa_status";
}

pa_status pa_last_plan(pa_plan_info *info) {
    if (!info || !g_have_plan) return PA_ERR_INVALID_ARG;
    *info = g_last_plan;
    return PA_OK;
}

size_t pa_workspace_bytes(const pa_attn_desc *desc) {
    Plan pl;
    const bool verify = desc && desc->q_len > 1;
    if (make_plan(desc, verify, &pl) != PA_OK) return static_cast<size_t>(-1);
    return pl.ws_bytes;
}

int64_t pa_hybrid_page_tokens(int64_t state_page_bytes, int64_t attn_bytes_per_token, int32_t alignment_tokens) {
    if (state_page_bytes <= 0 || attn_bytes_per_token <= 0 || alignment_tokens <= 0) return -1;
    // bytes of one alignment group; past INT64_MAX / alignment one group already holds any state page
    if (attn_bytes_per_token > INT64_MAX / alignment_tokens) return alignment_tokens;
    const int64_t group_bytes = attn_bytes_per_token * alignment_tokens;
    const int64_t groups = state_page_bytes / group_bytes + (state_page_bytes % group_bytes != 0);
    if (groups > INT64_MAX / alignment_tokens) return -1;
    return groups * alignment_tokens;
}

pa_status pa_reshape_and_cache(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                               const int64_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int64_t num_pages, int32_t *device_status,
                               void *stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_pages < 1)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * 2;
    if (row_bytes % 16 != 0 || row_bytes / 16 > INT32_MAX) return PA_ERR_UNSUPPORTED;
    // programmatic dependent launch: scheduled early, waits before any access
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_tokens));
    cfg.blockDim = dim3(128);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, pa_reshape_and_cache_kernel, static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slot_mapping, static_cast<int>(row_bytes / 16),
        num_pages * block_size, device_status);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_reshape_and_cache_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                   const int64_t *slot_mapping, const float *k_scale, const float *v_scale,
                                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int64_t num_pages, int32_t *device_status, void *stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_pages < 1)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping || !k_scale || !v_scale)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(v_scale) & 3u))
        return PA_ERR_INVALID_ARG;
    // a thread converts 8 elements of one head: head_dim must be a multiple of 8
    if (head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
    const int64_t row_vecs = static_cast<int64_t>(num_kv_heads) * head_dim / 8;
    if (row_vecs > INT32_MAX) return PA_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_tokens));
    cfg.blockDim = dim3(128);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, pa_reshape_and_cache_fp8_kernel, static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
        static_cast<uint2 *>(k_cache), static_cast<uint2 *>(v_cache), slot_mapping, k_scale, v_scale,
        static_cast<int>(row_vecs), head_dim / 8, num_pages * block_size, device_status);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_paged_attention_decode(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_table, const int32_t *seq_lens, const pa_attn_desc *desc,
                                    void *out, void *workspace, size_t workspace_bytes, int32_t *device_status,
                                    void *stream) {
    return decode_call(q, k_cache, v_cache, nullptr, nullptr, block_table, seq_lens, desc, out, workspace,
                       workspace_bytes, device_status, stream);
}

pa_status pa_paged_attention_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                        const float *k_scale, const float *v_scale, const int32_t *block_table,
                                        const int32_t *seq_lens, const pa_attn_desc *desc, void *out,
                                        void *workspace, size_t workspace_bytes, int32_t *device_status,
                                        void *stream) {
    if (!k_scale || !v_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(v_scale) & 3u))
        return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, desc, out, workspace,
                       workspace_bytes, device_status, stream);
}

pa_status pa_paged_attention_decode_append(const void *q, const void *k_new, const void *v_new, void *k_cache,
                                           void *v_cache, const int32_t *block_table, const int32_t *seq_lens,
                                           const pa_attn_desc *desc, void *out, void *workspace,
                                           size_t workspace_bytes, int32_t *device_status, void *stream) {
    if (!k_new || !v_new) return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, nullptr, nullptr, block_table, seq_lens, desc, out, workspace,
                       workspace_bytes, device_status, stream, k_new, v_new);
}

pa_status pa_paged_attention_decode_append_fp8(const void *q, const void *k_new, const void *v_new, void *k_cache,
                                               void *v_cache, const float *k_scale, const float *v_scale,
                                               const int32_t *block_table, const int32_t *seq_lens,
                                               const pa_attn_desc *desc, void *out, void *workspace,
                                               size_t workspace_bytes, int32_t *device_status, void *stream) {
    if (!k_new || !v_new || !k_scale || !v_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(v_scale) & 3u))
        return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, desc, out, workspace,
                       workspace_bytes, device_status, stream, k_new, v_new);
}

pa_status pa_paged_attention_verify(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_table, const int32_t *seq_lens, const pa_attn_desc *desc,
                                    void *out, void *workspace, size_t workspace_bytes, int32_t *device_status,
                                    void *stream) {
    return verify_call(q, k_cache, v_cache, nullptr, nullptr, block_table, seq_lens, desc, out, workspace,
                       workspace_bytes, device_status, stream);
}

pa_status pa_paged_attention_verify_fp8(const void *q, const void *k_cache, const void *v_cache,
                                        const float *k_scale, const float *v_scale, const int32_t *block_table,
                                        const int32_t *seq_lens, const pa_attn_desc *desc, void *out,
                                        void *workspace, size_t workspace_bytes, int32_t *device_status,
                                        void *stream) {
    if (!k_scale || !v_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(v_scale) & 3u))
        return PA_ERR_INVALID_ARG;
    return verify_call(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, desc, out, workspace,
                       workspace_bytes, device_status, stream);
}

}  // extern "C"

namespace pa {

// Decode over a bf16 cache (k_scale == nullptr) or an fp8 e4m3 cache; with
// k_new / v_new, the fused append of each sequence's new token first.
pa_status decode_call(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                      const float *v_scale, const int32_t *block_table, const int32_t *seq_lens,
                      const pa_attn_desc *desc, void *out, void *workspace, size_t workspace_bytes,
                      int32_t *device_status, void *stream, const void *k_new, const void *v_new) {
    const bool fp8 = k_scale != nullptr;
    pa_status st = check_desc(desc, false);
    if (st != PA_OK) return st;
    if (desc->num_seqs == 0) return PA_OK;
    st = check_common_ptrs(q, k_cache, v_cache, block_table, seq_lens, out);
    if (st != PA_OK) return st;
    if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_INVALID_ARG;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_INVALID_ARG;
    Plan pl;
    st = make_plan(desc, false, &pl);
    if (st != PA_OK) return st;
    st = check_workspace(pl, workspace, workspace_bytes);
    if (st != PA_OK) return st;

    // 16-token chunks as [column blocks][16 tokens][128 B], 128-byte swizzle
    CUtensorMap tk, tv;
    if (!encode_cache_map_blocks(&tk, k_cache, desc, fp8, kChunk) ||
        !encode_cache_map_blocks(&tv, v_cache, desc, fp8, kChunk))
        return PA_ERR_CUDA;

    const int group = desc->num_q_heads / desc->num_kv_heads;
    DecodeParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = out;
    p.part_o = static_cast<float *>(workspace);
    p.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(workspace) + pl.off_part_ml);
    p.status = device_status;
    p.num_pages = desc->num_pages;
    p.num_q_heads = desc->num_q_heads;
    p.max_pages_per_seq = desc->max_pages_per_seq;
    p.max_seq_len = desc->max_seq_len;
    p.block_size = desc->block_size;
    p.chunks_per_split = pl.chunks_per_split;
    p.num_splits = pl.num_splits;
    p.scale_log2 = desc->scale * 1.4426950408889634f;
    p.out_bf16 = desc->out_dtype == PA_OUT_BF16;
    p.early_kv = (desc->flags & PA_FLAG_EARLY_KV_READ) != 0;
    p.window = desc->window;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.k_cache = static_cast<uint8_t *>(const_cast<void *>(k_cache));
    p.v_cache = static_cast<uint8_t *>(const_cast<void *>(v_cache));

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 grid(pl.num_splits, desc->num_kv_heads, desc->num_seqs);
    const cudaError_t e = fp8 ? launch_decode_fp8(desc->head_dim, group, tk, tv, p, grid, s)
                              : launch_decode(desc->head_dim, group, tk, tv, p, grid, s);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    if (pl.num_splits > 1) {
        ReduceParams r;
        r.part_o = p.part_o;
        r.part_ml = p.part_ml;
        r.out = out;
        r.num_q_heads = desc->num_q_heads;
        r.num_splits = pl.num_splits;
        r.out_bf16 = p.out_bf16;
        if (launch_reduce(desc->head_dim, r, desc->num_seqs, pl.num_sms, s) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    record_plan(PA_PATH_DECODE_MMA, pl, desc, pl.num_splits * desc->num_kv_heads * desc->num_seqs);
    return PA_OK;
}

// Verify over a bf16 cache (k_scale == nullptr) or an fp8 e4m3 cache.
pa_status verify_call(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                      const float *v_scale, const int32_t *block_table, const int32_t *seq_lens,
                      const pa_attn_desc *desc, void *out, void *workspace, size_t workspace_bytes,
                      int32_t *device_status, void *stream) {
    const bool fp8 = k_scale != nullptr;
    pa_status st = check_desc(desc, true);
    if (st != PA_OK) return st;
    if (desc->num_seqs == 0) return PA_OK;
    st = check_common_ptrs(q, k_cache, v_cache, block_table, seq_lens, out);
    if (st != PA_OK) return st;
    Plan pl;
    st = make_plan(desc, true, &pl);
    if (st != PA_OK) return st;
    st = check_workspace(pl, workspace, workspace_bytes);
    if (st != PA_OK) return st;

    CUtensorMap tk, tv;
    CUtensorMap tk64, tv64;  // whole-tile copies; only used where a 64-token tile fits in a page
    if (fp8) {
        // e4m3 in 128-code column blocks, 128-byte swizzle: a 16-token chunk
        // per block, or a whole 64-token tile in one 5-D box
        if (!encode_cache_map(&tk, k_cache, desc, 128, true, true) ||
            !encode_cache_map(&tv, v_cache, desc, 128, true, true))
            return PA_ERR_CUDA;
        if (desc->block_size < 64) {
            tk64 = tk;  // never used: no 64-token tile fits in a smaller page
            tv64 = tv;
        } else if (!encode_cache_map_blocks(&tk64, k_cache, desc, true) ||
                   !encode_cache_map_blocks(&tv64, v_cache, desc, true)) {
            return PA_ERR_CUDA;
        }
    } else if (!encode_cache_map(&tk, k_cache, desc, 64, true) || !encode_cache_map(&tv, v_cache, desc, 64, true)) {
        return PA_ERR_CUDA;
    } else if (desc->block_size >= 64) {
        if (!encode_cache_map_blocks(&tk64, k_cache, desc) || !encode_cache_map_blocks(&tv64, v_cache, desc))
            return PA_ERR_CUDA;
    } else {
        tk64 = tk;  // never used: no 64-token tile fits in a smaller page
        tv64 = tv;
    }
    const int group = desc->num_q_heads / desc->num_kv_heads;
    // 128-token K tiles of one page, for the verify shapes that run 128-key score tiles
    CUtensorMap tk128 = tk64;
    if (!fp8 && desc->block_size >= 128 && verify_wide_score_tiles(desc->head_dim, desc->q_len * group) &&
        !encode_cache_map_blocks(&tk128, k_cache, desc, false, 128))
        return PA_ERR_CUDA;

    VerifyParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = out;
    p.part_o = static_cast<float *>(workspace);
    p.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(workspace) + pl.off_part_ml);
    p.status = device_status;
    p.num_pages = desc->num_pages;
    p.num_q_heads = desc->num_q_heads;
    p.q_len = desc->q_len;
    p.group = group;
    p.max_pages_per_seq = desc->max_pages_per_seq;
    p.max_seq_len = desc->max_seq_len;
    p.block_size = desc->block_size;
    p.chunks_per_split = pl.chunks_per_split;
    p.num_splits = pl.num_splits;
    p.scale_log2 = desc->scale * 1.4426950408889634f;
    p.out_bf16 = desc->out_dtype == PA_OUT_BF16;
    p.early_kv = (desc->flags & PA_FLAG_EARLY_KV_READ) != 0;
    p.window = desc->window;
    p.num_kv_heads = desc->num_kv_heads;
    p.k_scale = k_scale;
    p.v_scale = v_scale;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int row_blocks = (desc->q_len * group + 127) / 128;
    const dim3 grid(pl.num_splits, desc->num_kv_heads * row_blocks, desc->num_seqs);
    const cudaError_t e = fp8 ? launch_verify_fp8(desc->head_dim, tk, tv, tk64, tv64, p, grid, s)
                              : launch_verify(desc->head_dim, desc->q_len * group, tk, tv, tk64, tv64, tk128, p,
                                              grid, s);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    if (pl.num_splits > 1) {
        ReduceParams r;
        r.part_o = p.part_o;
        r.part_ml = p.part_ml;
        r.out = out;
        r.num_q_heads = desc->num_q_heads;
        r.num_splits = pl.num_splits;
        r.out_bf16 = p.out_bf16;
        if (launch_reduce(desc->head_dim, r, desc->num_seqs * desc->q_len, pl.num_sms, s) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    record_plan(PA_PATH_VERIFY_TCGEN05, pl, desc, pl.num_splits * desc->num_kv_heads * row_blocks * desc->num_seqs);
    return PA_OK;
}

}  // namespace pa
