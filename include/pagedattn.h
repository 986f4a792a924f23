/*
 * pagedattn.h -- C ABI of the GB300 (sm_103a) paged-attention library.
 *
 * The library computes, per query head, softmax(q . K^T * scale) . V over a KV
 * cache cut into fixed-size physical pages that each sequence reaches through
 * its own block table.  It is the full-attention decode path of a hybrid
 * Gated-DeltaNet/attention model (24 query heads on 4 KV heads, head_dim 256,
 * pages of 784 or 832 tokens; dense models use 16-token pages).
 *
 * Sources (web pages; cited by title and section):
 *   "DCU page832 attention" (luanjiahao.me), Sec.1 block-table address math,
 *     Sec.4 cache shape, Sec.5 tiled loop with online softmax, Sec.6 the
 *     varlen interface (q, k, v, seqused_k, block_table, max_seqlen_k, causal),
 *     Sec.7 page-contiguous decode loop.
 *   "Hybrid SSM decode rate on dual Radeon under vLLM" (cadamcat.github.io),
 *     section on the upstream split-KV fix: the KV range of one (sequence,
 *     KV head) is cut across many workgroups, then reduced.
 *   "Qwen3.8 on MI350P" (flozi.net), Lektion 3: several verify rows share each
 *     K/V tile, with a causal mask per row and merged softmax statistics.
 *   "Qwen3.5-27B 6x faster on one RTX 3090" (coreui.cn): new K/V rows are
 *     written into the cache by a copy (ggml_cpy) before attention reads them.
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device addresses owned by the caller; the library
 *     never allocates, frees or synchronises.  Calls are asynchronous on the
 *     given stream (a cudaStream_t passed as void*; NULL = legacy default stream).
 *   - Tensors are dense row-major (C order).  bf16 data is IEEE bfloat16.
 *     Every data pointer must be 16-byte aligned.
 *   - Host-detectable errors are returned synchronously as a pa_status; nothing
 *     is launched in that case.  A failed launch returns PA_ERR_CUDA.
 *   - Device-side errors (which the host cannot see: seq_lens and block tables
 *     live in device memory) are OR-ed as PA_DEV_* bits into *device_status if
 *     that pointer is non-NULL.  Kernels never trap; the affected output rows
 *     are written as zeros.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, inconsistent or negative sizes */
    PA_ERR_UNSUPPORTED = 2,  /* valid request outside the compiled kernel set */
    PA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than pa_workspace_bytes() */
    PA_ERR_CUDA = 4          /* a CUDA runtime/driver call or a launch failed */
} pa_status;

/* Output element type. */
typedef enum { PA_OUT_F32 = 0, PA_OUT_BF16 = 1 } pa_out_dtype;

/* Bits OR-ed into *device_status by the kernels. */
#define PA_DEV_BAD_SEQLEN 1  /* seq_lens[b] < 0, > max_seq_len, or (verify) < q_len */
#define PA_DEV_BAD_PAGE 2    /* a block_table entry that is read lies outside [0, num_pages) */
#define PA_DEV_BAD_SLOT 4    /* reshape_and_cache: slot >= num_pages * block_size */
#define PA_DEV_TIMEOUT 8     /* a bounded wait inside a kernel gave up (never expected) */

/* Shape and launch description of one attention call.
 *   num_seqs          B, number of sequences (>= 0; 0 is a no-op)
 *   q_len             query rows per sequence: 1 for decode, > 1 for verify
 *   num_q_heads       Hq;  num_kv_heads Hkv; Hq % Hkv == 0, G = Hq / Hkv.
 *                     Decode is compiled for G in {1, 2, 3, 4, 5, 6, 8, 12, 16}
 *                     at D = 256 and D = 128 (PA_ERR_UNSUPPORTED otherwise);
 *                     verify takes any G with G * q_len <= 32768
 *   head_dim          D (128 or 256)
 *   block_size        BS, tokens per physical page (a multiple of 16: 16, 784, 832 ...)
 *   max_pages_per_seq columns of block_table
 *   max_seq_len       host-side upper bound of seq_lens (plans the split count,
 *                     like max_seqlen_k of the varlen interface)
 *   num_pages         P, physical pages in each cache tensor
 *   scale             softmax scale (1/sqrt(D) for the models here)
 *   out_dtype         pa_out_dtype
 *   num_splits        0 = automatic; > 0 forces the split count (benchmarks, tests)
 *   num_sms           0 = query the current device; > 0 plans for that SM count
 *   flags             0, or PA_FLAG_EARLY_KV_READ (below)
 *   window            0 = full attention; W > 0 = sliding window: every query
 *                     row sees only its last W visible keys (its own position
 *                     included), as the RTX 3090 page's 2048-position window
 */
typedef struct {
    int32_t num_seqs;
    int32_t q_len;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t max_pages_per_seq;
    int32_t max_seq_len;
    int64_t num_pages;
    float scale;
    int32_t out_dtype;
    int32_t num_splits;
    int32_t num_sms;
    int32_t flags;
    int32_t window;
} pa_attn_desc;

/* desc->flags bits.
 *
 * Every kernel of this library is launched as a programmatic dependent of the
 * work before it on the stream: it may be scheduled while that work is still
 * running and overlap its own set-up with it.  By default each kernel then
 * waits for that work to finish before it reads or writes global memory.
 *
 * PA_FLAG_EARLY_KV_READ lets a decode or verify call start streaming cached
 * K/V before that wait.  Before the preceding work has finished it reads only
 * block_table, seq_lens and the cached K/V rows of positions 0 .. L_b - q_len - 1
 * (the context before the new rows); q, the new rows' cache slots, the
 * workspace and the output are touched only after the wait.  The caller
 * guarantees that no work that may still be running when the call starts
 * writes any of those early-read inputs.  Kernels of this library honour that
 * on their own (reshape_and_cache writes only the new rows' slots; the
 * attention kernels write only workspaces and outputs).  The guarantee is
 * broken by, for example, a kernel just before the call that fills the block
 * table or seq_lens on the device. */
#define PA_FLAG_EARLY_KV_READ 1

/* What the last successful attention call on this host thread ran: the path
 * marker the tests and benchmarks record. */
typedef struct {
    int32_t path_id;           /* PA_PATH_* */
    int32_t num_splits;        /* splits of the context per (sequence, KV head) */
    int32_t chunks_per_split;  /* 16-token chunks per split */
    int32_t grid_ctas;         /* CTAs of the main kernel */
    int32_t block_size;
    int32_t reduce_launched;   /* 1 if the partition-reduce kernel ran */
} pa_plan_info;

#define PA_PATH_DECODE_CUDA_CORE 1  /* retired: split-KV decode on the CUDA cores (no longer reported) */
#define PA_PATH_DECODE_MMA 2        /* split-KV decode, both products on the tensor cores (mma.sync) */
#define PA_PATH_VERIFY_TCGEN05 3    /* multi-row verify, tcgen05 + TMEM */

/* Bytes of device workspace an attention call with this description needs
 * (split partials: out vectors, max and sum per split).  0 when the plan does
 * not split.  Returns (size_t)-1 if the description is invalid.  Host only;
 * queries the device SM count unless desc->num_sms > 0.  The workspace may
 * hold anything before a call: every split writes the record the merge reads,
 * so one workspace serves any calls whose descriptions fit, without clearing. */
size_t pa_workspace_bytes(const pa_attn_desc *desc);

/* Page length, in tokens, for a hybrid model whose attention KV cache and
 * recurrent-state cache share one page granularity: the state page measured
 * in attention tokens, rounded up to whole groups of alignment_tokens,
 *     ceil(state_page_bytes / (alignment_tokens * attn_bytes_per_token)) * alignment_tokens
 * (DCU page-832 article, section "Why Qwen3.5's Hybrid Cache Makes This
 * Problem More Complex", the path without prefix caching).  A state page
 * worth 769..784 attention tokens gives 784 at 16-token alignment and 832 at
 * the 64-token access unit of the article's section 2.
 *   state_page_bytes      bytes of one recurrent-state page
 *   attn_bytes_per_token  one token's K+V bytes (2 * Hkv * D * 2 for bf16)
 *   alignment_tokens      page granularity in tokens (16, 64 ...)
 * Returns the page length, or -1 if an argument is not positive or the
 * result does not fit in int64.  Host arithmetic only.  The attention calls
 * accept any page length that is a multiple of 16. */
int64_t pa_hybrid_page_tokens(int64_t state_page_bytes, int64_t attn_bytes_per_token, int32_t alignment_tokens);

/* reshape_and_cache -- write new K/V rows into their page slots.
 * For every new token i with slot s = slot_mapping[i]:
 *     k_cache[s / BS, s % BS, h, :] = k_new[i, h, :]   (and the same for V)
 * with the page/offset split of the block-table address math.  s < 0 marks a
 * padding token and is skipped; s >= num_pages * BS sets PA_DEV_BAD_SLOT and is
 * skipped.  The copy is bit-exact.
 *   k_new, v_new   device bf16 [num_tokens, num_kv_heads, head_dim]
 *   k_cache,
 *   v_cache        device bf16 [num_pages, block_size, num_kv_heads, head_dim], written in place
 *   slot_mapping   device int64 [num_tokens]
 * head_dim * 2 bytes must be a multiple of 16. */
pa_status pa_reshape_and_cache(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                               const int64_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int64_t num_pages,
                               int32_t *device_status, void *stream);

/* paged_attention_decode -- one query row per sequence (desc->q_len == 1).
 * out[b, h, :] = sum_{t < L_b} softmax_t(scale * q[b, h, :] . K_t) V_t
 * with K_t, V_t the rows of token t of KV head h / G, found at
 * (block_table[b, t / BS], t % BS).  L_b = seq_lens[b] counts every cached
 * token, including the one just written.  L_b == 0 gives a zero row.
 * The context is cut into desc-planned splits per (sequence, KV head); each
 * split runs on its own CTA ("Hybrid SSM decode rate on dual Radeon under
 * vLLM", the split-KV fix: the KV range cut across workgroups, then
 * reduced); a log-sum-exp reduce merges them.  The arithmetic per split is
 * the tiled loop of "DCU page832 attention", Sec.5, over the page walk of its
 * Sec.7.
 *   q            device bf16 [B, Hq, D]
 *   k_cache,
 *   v_cache      device bf16 [P, BS, Hkv, D]
 *   block_table  device int32 [B, max_pages_per_seq]; entries past the last
 *                page a sequence uses are never read
 *   seq_lens     device int32 [B]
 *   out          device [B, Hq, D] of desc->out_dtype
 *   workspace    device, >= pa_workspace_bytes(desc) bytes (may be NULL if 0);
 *                calls that share a workspace must not overlap on the GPU
 *   device_status nullable device int32, PA_DEV_* bits are OR-ed in */
pa_status pa_paged_attention_decode(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_table, const int32_t *seq_lens,
                                    const pa_attn_desc *desc, void *out, void *workspace,
                                    size_t workspace_bytes, int32_t *device_status, void *stream);

/* paged_attention_decode_append -- the decode step's two calls in one kernel:
 * reshape_and_cache of each sequence's new token, then paged_attention_decode.
 * For every sequence b with L_b = seq_lens[b] >= 1, the new token is position
 * L_b - 1; its rows k_new[b], v_new[b] are written into the cache slot of that
 * position, (block_table[b, (L_b - 1) / BS], (L_b - 1) % BS) -- the address
 * math of "DCU page832 attention", Sec.1 -- bit-exactly as pa_reshape_and_cache
 * with that slot would, and the decode then reads them ("Qwen3.5-27B 6x faster
 * on one RTX 3090": new K/V rows are copied into the cache before attention
 * reads it).  The CTA whose split holds position L_b - 1 writes the rows before
 * it copies the chunk that holds them, so the step needs no separate kernel.
 * The result (output and caches) equals pa_reshape_and_cache followed by
 * pa_paged_attention_decode on the same stream.
 *   k_new, v_new  device bf16 [B, Hkv, D], 16-byte aligned; read after the
 *                 stream dependency (PA_FLAG_EARLY_KV_READ does not cover them)
 *   k_cache,
 *   v_cache       written in place (the new rows) and read
 * A position L_b - 1 whose page index lies outside [0, P) is not written
 * (PA_DEV_BAD_PAGE, zero row, as for decode); L_b == 0 writes nothing.  Other
 * arguments, results and errors as for pa_paged_attention_decode. */
pa_status pa_paged_attention_decode_append(const void *q, const void *k_new, const void *v_new, void *k_cache,
                                           void *v_cache, const int32_t *block_table, const int32_t *seq_lens,
                                           const pa_attn_desc *desc, void *out, void *workspace,
                                           size_t workspace_bytes, int32_t *device_status, void *stream);

/* paged_attention_verify -- desc->q_len > 1 new rows per sequence, causal among
 * them (speculative verify: "Qwen3.8 on MI350P", Lektion 3, the verify rows
 * of one request sharing every K/V tile under a per-row causal mask).  Rows are ordered (sequence, new row): q and out
 * are [B * q_len, Hq, D].  Row r (0-based) of sequence b attends to keys
 * 0 .. L_b - q_len + r inclusive; the q_len new rows must already be in the
 * cache (L_b >= q_len, else PA_DEV_BAD_SEQLEN and zero rows).  The G * q_len
 * rows of one KV head are processed in blocks of 128 that share every K/V tile
 * on the tensor cores; a block reads only the keys its last row can see, so a
 * large q_len (a chunked-prefill step) skips the masked upper triangle tile by
 * tile.  Supported:
 * G * q_len <= 32768 and num_kv_heads * ceil(G * q_len / 128) <= 65535.  Other
 * arguments as for decode. */
pa_status pa_paged_attention_verify(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_table, const int32_t *seq_lens,
                                    const pa_attn_desc *desc, void *out, void *workspace,
                                    size_t workspace_bytes, int32_t *device_status, void *stream);

/* ---- fp8 e4m3 KV cache ------------------------------------------------------
 * The RTX 3090 page ("24 GB of VRAM for a 128K context") shrinks the KV cache
 * with a quantised format (ggml's Q4_0) because decode time is KV bytes.  The
 * counterpart here is an fp8 e4m3 cache (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, largest finite 448) with one binary32 scale
 * per KV head for K and one for V, chosen by the caller (for example max |x|
 * / 448 over a calibration set): an element x is stored as the code
 *     e4m3(x / scale[kv_head])     (binary32 division, round to nearest even,
 *                                   saturating to +-448; NaN stays NaN)
 * and read back as decoded(code) * scale[kv_head].  Half the bytes of bf16. */

/* reshape_and_cache into an fp8 cache: the slot rules of pa_reshape_and_cache,
 * each element quantised as above.
 *   k_new, v_new     device bf16 [num_tokens, num_kv_heads, head_dim]
 *   k_cache, v_cache device uint8 e4m3 codes [num_pages, block_size, num_kv_heads, head_dim]
 *   k_scale, v_scale device float [num_kv_heads]
 * head_dim must be a multiple of 8 (PA_ERR_UNSUPPORTED otherwise). */
pa_status pa_reshape_and_cache_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                   const int64_t *slot_mapping, const float *k_scale, const float *v_scale,
                                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int64_t num_pages, int32_t *device_status,
                                   void *stream);

/* paged_attention_decode over an fp8 cache: out as pa_paged_attention_decode
 * with K_t = decoded(k code) * k_scale[kv head], V_t likewise.  The split
 * plan and workspace are those of the bf16 call with the same description
 * (pa_workspace_bytes).  Window and PA_FLAG_EARLY_KV_READ behave as there.
 *   k_cache, v_cache device uint8 e4m3 codes [P, BS, Hkv, D]
 *   k_scale, v_scale device float [Hkv], read after the stream dependency
 * Other arguments, results and errors as for pa_paged_attention_decode. */
pa_status pa_paged_attention_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                        const float *k_scale, const float *v_scale,
                                        const int32_t *block_table, const int32_t *seq_lens,
                                        const pa_attn_desc *desc, void *out, void *workspace,
                                        size_t workspace_bytes, int32_t *device_status, void *stream);

/* paged_attention_decode_append over an fp8 cache: the new rows quantised as
 * pa_reshape_and_cache_fp8 does (bit-exact), then the decode of
 * pa_paged_attention_decode_fp8.  Arguments as for pa_paged_attention_decode_append
 * plus the scales of pa_paged_attention_decode_fp8. */
pa_status pa_paged_attention_decode_append_fp8(const void *q, const void *k_new, const void *v_new, void *k_cache,
                                               void *v_cache, const float *k_scale, const float *v_scale,
                                               const int32_t *block_table, const int32_t *seq_lens,
                                               const pa_attn_desc *desc, void *out, void *workspace,
                                               size_t workspace_bytes, int32_t *device_status, void *stream);

/* paged_attention_verify over an fp8 cache: out as pa_paged_attention_verify
 * with K and V decoded as for pa_paged_attention_decode_fp8.  The tensor-core
 * products run in f16 (exact for the e4m3 values; q enters as f16), with the
 * scales applied to the scores and to the final normaliser.  Same plan,
 * workspace, limits and errors as pa_paged_attention_verify. */
pa_status pa_paged_attention_verify_fp8(const void *q, const void *k_cache, const void *v_cache,
                                        const float *k_scale, const float *v_scale,
                                        const int32_t *block_table, const int32_t *seq_lens,
                                        const pa_attn_desc *desc, void *out, void *workspace,
                                        size_t workspace_bytes, int32_t *device_status, void *stream);

/* Size of the scratch array that pa_paged_attention_decode_noalloc keeps in
 * device memory (8 MiB per GPU that loads the library, held until exit). */
#define PA_NOALLOC_SCRATCH_BYTES (8u << 20)

/* pa_paged_attention_decode_noalloc -- the same decode as
 * pa_paged_attention_decode, for callers that cannot allocate device memory
 * (for example a plugin inside a serving engine that has already claimed
 * nearly all of HBM for its own KV-cache pool and owns every allocation, so
 * it has no spare buffer to hand over).  The pages have no counterpart of
 * this entry point; it is a convenience of this library.
 *   - No workspace argument: the split partials go to a scratch array of
 *     PA_NOALLOC_SCRATCH_BYTES compiled into the library.  A description whose
 *     pa_workspace_bytes() exceeds that size is rejected with PA_ERR_WORKSPACE
 *     before anything is launched.
 *   - The first call on a device looks up the array's device address (a
 *     cudaGetSymbolAddress on the current device); make that first call before
 *     any stream capture.  The call allocates nothing (no cudaMalloc/cudaFree).
 *   - Every call on a device shares the one array, and it keeps the last
 *     call's contents; nothing in it needs to start at zero, because each call
 *     writes every partial it later reads.  Calls whose kernels overlap on the
 *     GPU (different streams, no ordering between them) race on the array and
 *     give wrong results: order them.
 *   - The array's address is cached per device ordinal for the life of the
 *     process: a device reset (cudaDeviceReset) after the first call on that
 *     device is not supported.
 * Other arguments, results and errors as for pa_paged_attention_decode. */
pa_status pa_paged_attention_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                            const int32_t *block_table, const int32_t *seq_lens,
                                            const pa_attn_desc *desc, void *out, int32_t *device_status,
                                            void *stream);

/* Human-readable name of a status code (static storage). */
const char *pa_status_string(pa_status status);

/* Copies the plan of the last successful attention call made on this host
 * thread.  PA_ERR_INVALID_ARG if info is NULL or no call was made yet. */
pa_status pa_last_plan(pa_plan_info *info);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
