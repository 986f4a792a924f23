// decode_noalloc.cu -- pa_paged_attention_decode_noalloc: decode for callers
// that cannot allocate device memory.
//
// Some callers run inside an engine that reserved nearly all of HBM for its own
// KV-cache pool and hands a plugin only the tensors of the call; they have no
// way to obtain the workspace that pa_paged_attention_decode asks for.  This
// entry point keeps that workspace (the split partials) in a fixed-size array
// compiled into the library instead, and otherwise runs the ordinary decode.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pagedattn.h"

// The split partials of every no-alloc call on a device.  Host code sees only a
// stand-in for this name, never its device address; the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
pa_status scratch_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_paged_attention_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                                       const int32_t *block_table, const int32_t *seq_lens,
                                                       const pa_attn_desc *desc, void *out, int32_t *device_status,
                                                       void *stream) {
    if (!desc) return PA_ERR_INVALID_ARG;
    // A description the ordinary decode rejects (q_len != 1 among them) gets
    // that call's exact error before any size is compared, and nothing runs.
    const size_t need = desc->q_len == 1 ? pa_workspace_bytes(desc) : static_cast<size_t>(-1);
    if (need == static_cast<size_t>(-1))  // invalid description: report its exact error, launch nothing
        return pa_paged_attention_decode(q, k_cache, v_cache, block_table, seq_lens, desc, out, nullptr, 0,
                                         device_status, stream);
    if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;  // plan larger than the built-in scratch
    void *scratch = nullptr;
    if (need > 0) {
        const pa_status st = scratch_address(&scratch);
        if (st != PA_OK) return st;
    }
    return pa_paged_attention_decode(q, k_cache, v_cache, block_table, seq_lens, desc, out, scratch,
                                     need > 0 ? static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES) : 0, device_status,
                                     stream);
}
