// pa_binding.cpp -- the compiled half of the Python binding: each call checks
// its tensors against the attention description (element type, shape, CUDA
// device, contiguity) and hands their pointers to the C ABI of
// include/pagedattn.h.  It computes nothing.
//
// The C ABI sees bare pointers and cannot tell a buffer's size, so a tensor of
// the wrong type or shape would be read or written past its end; the checks
// come before the call.  They run here rather than in Python because a
// decode step is one call per layer and the Python attribute lookups of eleven
// tensors cost more host time per call than the kernel takes on the GPU.
//
// The library is not linked: the Python side passes the addresses of the C
// entry points it loaded (set_entry), so the process holds one copy of the
// library and its host-side state (last plan, tensor-map cache).
#include <torch/extension.h>

#include <c10/cuda/CUDAFunctions.h>
#include <c10/cuda/CUDAStream.h>

#include <array>
#include <initializer_list>
#include <string>
#include <utility>

#include "pagedattn.h"

namespace {

using at::Tensor;
using c10::optional;

using AttnFn = pa_status (*)(const void *, const void *, const void *, const int32_t *, const int32_t *,
                             const pa_attn_desc *, void *, void *, size_t, int32_t *, void *);
using AttnFp8Fn = pa_status (*)(const void *, const void *, const void *, const float *, const float *,
                                const int32_t *, const int32_t *, const pa_attn_desc *, void *, void *, size_t,
                                int32_t *, void *);
using AppendFn = pa_status (*)(const void *, const void *, const void *, void *, void *, const int32_t *,
                               const int32_t *, const pa_attn_desc *, void *, void *, size_t, int32_t *, void *);
using AppendFp8Fn = pa_status (*)(const void *, const void *, const void *, void *, void *, const float *,
                                  const float *, const int32_t *, const int32_t *, const pa_attn_desc *, void *,
                                  void *, size_t, int32_t *, void *);
using NoAllocFn = pa_status (*)(const void *, const void *, const void *, const int32_t *, const int32_t *,
                                const pa_attn_desc *, void *, int32_t *, void *);
using ReshapeFn = pa_status (*)(const void *, const void *, void *, void *, const int64_t *, int32_t, int32_t,
                                int32_t, int32_t, int64_t, int32_t *, void *);
using ReshapeFp8Fn = pa_status (*)(const void *, const void *, void *, void *, const int64_t *, const float *,
                                   const float *, int32_t, int32_t, int32_t, int32_t, int64_t, int32_t *, void *);

struct Entries {
    AttnFn decode = nullptr, verify = nullptr;
    AttnFp8Fn decode_fp8 = nullptr, verify_fp8 = nullptr;
    AppendFn decode_append = nullptr;
    AppendFp8Fn decode_append_fp8 = nullptr;
    NoAllocFn decode_noalloc = nullptr;
    ReshapeFn reshape = nullptr;
    ReshapeFp8Fn reshape_fp8 = nullptr;
} g_entries;

void set_entry(const std::string &name, int64_t addr) {
    void *p = reinterpret_cast<void *>(addr);
    if (name == "pa_paged_attention_decode") g_entries.decode = reinterpret_cast<AttnFn>(p);
    else if (name == "pa_paged_attention_verify") g_entries.verify = reinterpret_cast<AttnFn>(p);
    else if (name == "pa_paged_attention_decode_fp8") g_entries.decode_fp8 = reinterpret_cast<AttnFp8Fn>(p);
    else if (name == "pa_paged_attention_verify_fp8") g_entries.verify_fp8 = reinterpret_cast<AttnFp8Fn>(p);
    else if (name == "pa_paged_attention_decode_append") g_entries.decode_append = reinterpret_cast<AppendFn>(p);
    else if (name == "pa_paged_attention_decode_append_fp8")
        g_entries.decode_append_fp8 = reinterpret_cast<AppendFp8Fn>(p);
    else if (name == "pa_paged_attention_decode_noalloc") g_entries.decode_noalloc = reinterpret_cast<NoAllocFn>(p);
    else if (name == "pa_reshape_and_cache") g_entries.reshape = reinterpret_cast<ReshapeFn>(p);
    else if (name == "pa_reshape_and_cache_fp8") g_entries.reshape_fp8 = reinterpret_cast<ReshapeFp8Fn>(p);
    else TORCH_CHECK_VALUE(false, "unknown entry point ", name);
}

bool is_fp8_cache_type(at::ScalarType t) { return t == at::kByte || t == at::ScalarType::Float8_e4m3fn; }

// Element type and shape (when `check_shape`) of one tensor.  The device and
// layout checks come after every tensor's type and shape (`placed`), so that a
// call's first error names the argument that does not fit the description.
void expect(const Tensor &t, const char *name, bool type_ok, const char *want, c10::IntArrayRef shape,
            bool check_shape = true) {
    TORCH_CHECK_VALUE(type_ok, name, ": dtype ", t.scalar_type(), "; expected ", want);
    if (check_shape) TORCH_CHECK_VALUE(t.sizes().equals(shape), name, ": shape ", t.sizes(), "; expected ", shape);
}

// The library launches on the current device, so every tensor must live there.
void placed(std::initializer_list<std::pair<const Tensor *, const char *>> ts) {
    int dev = -1;
    for (const auto &[t, name] : ts) {
        if (t == nullptr) continue;
        TORCH_CHECK_VALUE(t->is_cuda(), name, ": a CUDA tensor is required (got ", t->device(), ")");
        if (dev < 0) dev = c10::cuda::current_device();
        TORCH_CHECK_VALUE(t->get_device() == dev, name, ": on ", t->device(), ", but the current device is cuda:", dev);
        TORCH_CHECK_VALUE(t->is_contiguous(), name, ": the tensor must be contiguous");
    }
}

const Tensor *opt(const optional<Tensor> &t) { return t.has_value() ? &*t : nullptr; }

void *stream_of(int64_t s) {
    return s == -1 ? static_cast<void *>(c10::cuda::getCurrentCUDAStream().stream()) : reinterpret_cast<void *>(s);
}

template <typename T>
T *ptr_of(const optional<Tensor> &t) {
    return t.has_value() ? static_cast<T *>(t->data_ptr()) : nullptr;
}

enum Kind { kDecode = 0, kDecodeAppend, kVerify, kDecodeFp8, kDecodeAppendFp8, kVerifyFp8, kDecodeNoAlloc };

// One attention call of the given kind (the C entry point it maps to is in the
// switch below); returns the pa_status of the call.
int64_t attention(int64_t kind, const Tensor &q, const Tensor &k_cache, const Tensor &v_cache,
                  const optional<Tensor> &k_scale, const optional<Tensor> &v_scale, const optional<Tensor> &k_new,
                  const optional<Tensor> &v_new, const Tensor &block_table, const Tensor &seq_lens,
                  int64_t desc_addr, const Tensor &out, const optional<Tensor> &workspace,
                  const optional<Tensor> &status, int64_t stream) {
    TORCH_CHECK_VALUE(desc_addr != 0, "desc: a description is required");
    const pa_attn_desc *d = reinterpret_cast<const pa_attn_desc *>(desc_addr);
    const bool fp8 = kind == kDecodeFp8 || kind == kDecodeAppendFp8 || kind == kVerifyFp8;
    const bool append = kind == kDecodeAppend || kind == kDecodeAppendFp8;
    const int64_t rows = static_cast<int64_t>(d->num_seqs) * d->q_len;
    const std::array<int64_t, 3> row_shape{rows, d->num_q_heads, d->head_dim};
    const std::array<int64_t, 4> cache_shape{d->num_pages, d->block_size, d->num_kv_heads, d->head_dim};
    expect(q, "q", q.scalar_type() == at::kBFloat16, "bfloat16", row_shape);
    const bool kc_ok = fp8 ? is_fp8_cache_type(k_cache.scalar_type()) : k_cache.scalar_type() == at::kBFloat16;
    const bool vc_ok = fp8 ? is_fp8_cache_type(v_cache.scalar_type()) : v_cache.scalar_type() == at::kBFloat16;
    const char *cache_want = fp8 ? "uint8 or float8_e4m3fn (e4m3 codes)" : "bfloat16";
    expect(k_cache, "k_cache", kc_ok, cache_want, cache_shape);
    expect(v_cache, "v_cache", vc_ok, cache_want, cache_shape);
    expect(block_table, "block_table", block_table.scalar_type() == at::kInt, "int32",
           std::array<int64_t, 2>{d->num_seqs, d->max_pages_per_seq});
    expect(seq_lens, "seq_lens", seq_lens.scalar_type() == at::kInt, "int32", std::array<int64_t, 1>{d->num_seqs});
    const bool out_bf16 = d->out_dtype == PA_OUT_BF16;
    expect(out, "out", out.scalar_type() == (out_bf16 ? at::kBFloat16 : at::kFloat), out_bf16 ? "bfloat16" : "float32",
           row_shape);
    const std::array<int64_t, 1> scale_shape{d->num_kv_heads};
    TORCH_CHECK_VALUE(!fp8 || (k_scale.has_value() && v_scale.has_value()), "k_scale, v_scale: an e4m3 cache needs both");
    if (k_scale.has_value()) expect(*k_scale, "k_scale", k_scale->scalar_type() == at::kFloat, "float32", scale_shape);
    if (v_scale.has_value()) expect(*v_scale, "v_scale", v_scale->scalar_type() == at::kFloat, "float32", scale_shape);
    if (append) {
        TORCH_CHECK_VALUE(k_new.has_value() && v_new.has_value(), "k_new, v_new: the new rows are required");
        const std::array<int64_t, 3> new_shape{d->num_seqs, d->num_kv_heads, d->head_dim};
        expect(*k_new, "k_new", k_new->scalar_type() == at::kBFloat16, "bfloat16", new_shape);
        expect(*v_new, "v_new", v_new->scalar_type() == at::kBFloat16, "bfloat16", new_shape);
    }
    size_t ws_bytes = 0;
    if (workspace.has_value()) ws_bytes = workspace->numel() * workspace->element_size();
    if (status.has_value())
        expect(*status, "status", status->scalar_type() == at::kInt && status->numel() >= 1, "int32 (one element)",
               {}, false);
    placed({{&q, "q"}, {&k_cache, "k_cache"}, {&v_cache, "v_cache"}, {&block_table, "block_table"},
            {&seq_lens, "seq_lens"}, {&out, "out"}, {opt(k_scale), "k_scale"}, {opt(v_scale), "v_scale"},
            {opt(k_new), "k_new"}, {opt(v_new), "v_new"}, {opt(workspace), "workspace"}, {opt(status), "status"}});

    const void *qp = q.data_ptr();
    void *kc = k_cache.data_ptr(), *vc = v_cache.data_ptr(), *op = out.data_ptr(), *wp = ptr_of<void>(workspace);
    const int32_t *bt = block_table.data_ptr<int32_t>(), *sl = seq_lens.data_ptr<int32_t>();
    int32_t *st = ptr_of<int32_t>(status);
    const float *ks = ptr_of<float>(k_scale), *vs = ptr_of<float>(v_scale);
    const void *kn = ptr_of<void>(k_new), *vn = ptr_of<void>(v_new);
    void *s = stream_of(stream);
    switch (kind) {
        case kDecode:
            TORCH_CHECK(g_entries.decode, "entry point not set");
            return g_entries.decode(qp, kc, vc, bt, sl, d, op, wp, ws_bytes, st, s);
        case kVerify:
            TORCH_CHECK(g_entries.verify, "entry point not set");
            return g_entries.verify(qp, kc, vc, bt, sl, d, op, wp, ws_bytes, st, s);
        case kDecodeFp8:
            TORCH_CHECK(g_entries.decode_fp8, "entry point not set");
            return g_entries.decode_fp8(qp, kc, vc, ks, vs, bt, sl, d, op, wp, ws_bytes, st, s);
        case kVerifyFp8:
            TORCH_CHECK(g_entries.verify_fp8, "entry point not set");
            return g_entries.verify_fp8(qp, kc, vc, ks, vs, bt, sl, d, op, wp, ws_bytes, st, s);
        case kDecodeAppend:
            TORCH_CHECK(g_entries.decode_append, "entry point not set");
            return g_entries.decode_append(qp, kn, vn, kc, vc, bt, sl, d, op, wp, ws_bytes, st, s);
        case kDecodeAppendFp8:
            TORCH_CHECK(g_entries.decode_append_fp8, "entry point not set");
            return g_entries.decode_append_fp8(qp, kn, vn, kc, vc, ks, vs, bt, sl, d, op, wp, ws_bytes, st, s);
        case kDecodeNoAlloc:
            TORCH_CHECK(g_entries.decode_noalloc, "entry point not set");
            return g_entries.decode_noalloc(qp, kc, vc, bt, sl, d, op, st, s);
    }
    TORCH_CHECK_VALUE(false, "unknown call kind ", kind);
    return PA_ERR_INVALID_ARG;
}

// reshape_and_cache (bf16) or reshape_and_cache_fp8: the geometry comes from
// the cache tensor itself.
int64_t reshape(bool fp8, const Tensor &k_new, const Tensor &v_new, const Tensor &k_cache, const Tensor &v_cache,
                const Tensor &slot_mapping, const optional<Tensor> &k_scale, const optional<Tensor> &v_scale,
                const optional<Tensor> &status, int64_t stream) {
    TORCH_CHECK_VALUE(k_cache.dim() == 4, "k_cache: a [pages, block_size, kv_heads, head_dim] tensor is required");
    TORCH_CHECK_VALUE(slot_mapping.dim() == 1, "slot_mapping: a one-dimensional tensor is required");
    const int64_t n = slot_mapping.size(0), hkv = k_cache.size(2), dim = k_cache.size(3);
    const char *cache_want = fp8 ? "uint8 or float8_e4m3fn (e4m3 codes)" : "bfloat16";
    expect(k_cache, "k_cache", fp8 ? is_fp8_cache_type(k_cache.scalar_type()) : k_cache.scalar_type() == at::kBFloat16,
           cache_want, {}, false);
    expect(v_cache, "v_cache", v_cache.scalar_type() == k_cache.scalar_type(), cache_want, k_cache.sizes());
    const std::array<int64_t, 3> new_shape{n, hkv, dim};
    expect(k_new, "k_new", k_new.scalar_type() == at::kBFloat16, "bfloat16", new_shape);
    expect(v_new, "v_new", v_new.scalar_type() == at::kBFloat16, "bfloat16", new_shape);
    expect(slot_mapping, "slot_mapping", slot_mapping.scalar_type() == at::kLong, "int64", {}, false);
    const std::array<int64_t, 1> scale_shape{hkv};
    TORCH_CHECK_VALUE(!fp8 || (k_scale.has_value() && v_scale.has_value()), "k_scale, v_scale: an e4m3 cache needs both");
    if (k_scale.has_value()) expect(*k_scale, "k_scale", k_scale->scalar_type() == at::kFloat, "float32", scale_shape);
    if (v_scale.has_value()) expect(*v_scale, "v_scale", v_scale->scalar_type() == at::kFloat, "float32", scale_shape);
    if (status.has_value())
        expect(*status, "status", status->scalar_type() == at::kInt && status->numel() >= 1, "int32 (one element)",
               {}, false);
    placed({{&k_new, "k_new"}, {&v_new, "v_new"}, {&k_cache, "k_cache"}, {&v_cache, "v_cache"},
            {&slot_mapping, "slot_mapping"}, {opt(k_scale), "k_scale"}, {opt(v_scale), "v_scale"},
            {opt(status), "status"}});
    int32_t *st = ptr_of<int32_t>(status);
    void *s = stream_of(stream);
    if (fp8) {
        TORCH_CHECK(g_entries.reshape_fp8, "entry point not set");
        return g_entries.reshape_fp8(k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                     slot_mapping.data_ptr<int64_t>(), ptr_of<float>(k_scale), ptr_of<float>(v_scale),
                                     static_cast<int32_t>(n), static_cast<int32_t>(hkv), static_cast<int32_t>(dim),
                                     static_cast<int32_t>(k_cache.size(1)), k_cache.size(0), st, s);
    }
    TORCH_CHECK(g_entries.reshape, "entry point not set");
    return g_entries.reshape(k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                             slot_mapping.data_ptr<int64_t>(), static_cast<int32_t>(n), static_cast<int32_t>(hkv),
                             static_cast<int32_t>(dim), static_cast<int32_t>(k_cache.size(1)), k_cache.size(0), st, s);
}

}  // namespace

PYBIND11_MODULE(TORCH_EXTENSION_NAME, m) {
    m.def("set_entry", &set_entry);
    m.def("attention", &attention);
    m.def("reshape", &reshape);
}
