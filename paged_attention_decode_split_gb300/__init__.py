"""Paged-attention split-KV decode for GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libpagedattn.so`` (the C ABI of
``include/pagedattn.h``).  It only marshals arguments: torch tensors supply
device pointers and the current CUDA stream (after their element types and
shapes are checked against the attention description, since the C ABI cannot
see a buffer's size); every step of the computation runs in the library's CUDA
kernels.  If the library is missing or cannot be loaded,
every call raises -- there is no fallback.

Names follow the C ABI: ``reshape_and_cache``, ``paged_attention_decode``,
``paged_attention_decode_append``, ``paged_attention_verify``,
``workspace_bytes``, ``last_plan``.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "AttnDesc", "PlanInfo", "PagedAttnError", "load_library", "make_desc", "workspace_bytes",
    "hybrid_page_tokens", "reshape_and_cache_fp8", "paged_attention_decode_fp8", "paged_attention_verify_fp8",
    "reshape_and_cache", "paged_attention_decode", "paged_attention_verify", "last_plan",
    "paged_attention_decode_append", "paged_attention_decode_append_fp8",
    "status_string", "PA_OK", "PA_ERR_INVALID_ARG", "PA_ERR_UNSUPPORTED", "PA_ERR_WORKSPACE",
    "PA_ERR_CUDA", "PA_OUT_F32", "PA_OUT_BF16", "PA_DEV_BAD_SEQLEN", "PA_DEV_BAD_PAGE",
    "PA_DEV_BAD_SLOT", "PA_DEV_TIMEOUT", "PA_PATH_DECODE_CUDA_CORE", "PA_PATH_DECODE_MMA",
    "PA_PATH_VERIFY_TCGEN05", "PA_FLAG_EARLY_KV_READ", "PA_NOALLOC_SCRATCH_BYTES", "paged_attention_decode_noalloc",
]

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = 0, 1, 2, 3, 4
PA_OUT_F32, PA_OUT_BF16 = 0, 1
PA_DEV_BAD_SEQLEN, PA_DEV_BAD_PAGE, PA_DEV_BAD_SLOT, PA_DEV_TIMEOUT = 1, 2, 4, 8
PA_PATH_DECODE_CUDA_CORE, PA_PATH_DECODE_MMA, PA_PATH_VERIFY_TCGEN05 = 1, 2, 3
PA_FLAG_EARLY_KV_READ = 1
PA_NOALLOC_SCRATCH_BYTES = 8 << 20

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpagedattn.so")


class AttnDesc(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32), ("q_len", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32), ("max_seq_len", ctypes.c_int32), ("num_pages", ctypes.c_int64),
        ("scale", ctypes.c_float), ("out_dtype", ctypes.c_int32), ("num_splits", ctypes.c_int32),
        ("num_sms", ctypes.c_int32), ("flags", ctypes.c_int32), ("window", ctypes.c_int32),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("path_id", ctypes.c_int32), ("num_splits", ctypes.c_int32), ("chunks_per_split", ctypes.c_int32),
        ("grid_ctas", ctypes.c_int32), ("block_size", ctypes.c_int32), ("reduce_launched", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p


def load_library(path: str | None = None):
    """Load libpagedattn.so (built by ``_build.build()``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"libpagedattn.so not found at {path}; build it with "
                "`python -m paged_attention_decode_split_gb300._build` (no CPU fallback exists)")
        lib = ctypes.CDLL(path)
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_status_string.argtypes = [ctypes.c_int]
        lib.pa_workspace_bytes.restype = ctypes.c_size_t
        lib.pa_workspace_bytes.argtypes = [ctypes.POINTER(AttnDesc)]
        lib.pa_hybrid_page_tokens.restype = ctypes.c_int64
        lib.pa_hybrid_page_tokens.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32]
        lib.pa_last_plan.restype = ctypes.c_int
        lib.pa_last_plan.argtypes = [ctypes.POINTER(PlanInfo)]
        lib.pa_reshape_and_cache.restype = ctypes.c_int
        lib.pa_reshape_and_cache.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _vp, _vp]
        lib.pa_reshape_and_cache_fp8.restype = ctypes.c_int
        lib.pa_reshape_and_cache_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _vp, _vp]
        for name in ("pa_paged_attention_decode_fp8", "pa_paged_attention_verify_fp8"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(AttnDesc), _vp, _vp, ctypes.c_size_t,
                           _vp, _vp]
        lib.pa_paged_attention_decode_append.restype = ctypes.c_int
        lib.pa_paged_attention_decode_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(AttnDesc),
                                                         _vp, _vp, ctypes.c_size_t, _vp, _vp]
        lib.pa_paged_attention_decode_append_fp8.restype = ctypes.c_int
        lib.pa_paged_attention_decode_append_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                                             ctypes.POINTER(AttnDesc), _vp, _vp, ctypes.c_size_t,
                                                             _vp, _vp]
        lib.pa_paged_attention_decode_noalloc.restype = ctypes.c_int
        lib.pa_paged_attention_decode_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.POINTER(AttnDesc), _vp,
                                                          _vp, _vp]
        for name in ("pa_paged_attention_decode", "pa_paged_attention_verify"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.POINTER(AttnDesc), _vp, _vp, ctypes.c_size_t, _vp, _vp]
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().pa_status_string(int(status)).decode()


def make_desc(*, num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
              max_pages_per_seq: int, max_seq_len: int, num_pages: int, scale: float, q_len: int = 1,
              out_dtype: int = PA_OUT_F32, num_splits: int = 0, num_sms: int = 0, flags: int = 0,
              window: int = 0) -> AttnDesc:
    return AttnDesc(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_pages_per_seq,
                    max_seq_len, num_pages, scale, out_dtype, num_splits, num_sms, flags, window)


def workspace_bytes(desc: AttnDesc) -> int:
    n = load_library().pa_workspace_bytes(ctypes.byref(desc))
    if n == ctypes.c_size_t(-1).value:
        raise PagedAttnError(PA_ERR_INVALID_ARG, "pa_workspace_bytes")
    return int(n)


def hybrid_page_tokens(state_page_bytes: int, attn_bytes_per_token: int, alignment_tokens: int) -> int:
    """Page length (tokens) shared by a hybrid model's attention and state caches."""
    n = load_library().pa_hybrid_page_tokens(state_page_bytes, attn_bytes_per_token, alignment_tokens)
    if n < 0:
        raise PagedAttnError(PA_ERR_INVALID_ARG, "pa_hybrid_page_tokens")
    return int(n)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    assert t.is_contiguous(), "tensors passed to the library must be contiguous"
    return t.data_ptr()


def _current_stream_handle() -> int:
    """The current CUDA stream of the current device as a raw handle.  The raw
    query avoids building a torch.cuda.Stream object on every call (about 5 us
    of host time); the public path is the fallback."""
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _stream(stream) -> int | None:
    if stream is None:
        return _current_stream_handle()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedAttnError(status, what)


# The C ABI takes bare pointers and cannot tell a buffer's size or element
# type, so a tensor of the wrong type or shape would be read or written past
# its end.  The binding checks every tensor against the description before the
# call (raw integer pointers pass through unchecked).
def _expect(t, name: str, dtypes, shape=None) -> None:
    if t is None or isinstance(t, int):
        return
    dts = dtypes if isinstance(dtypes, tuple) else (dtypes,)
    if t.dtype not in dts:
        raise ValueError(f"{name}: dtype {t.dtype}; expected {' or '.join(str(d) for d in dts)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}; expected {tuple(shape)}")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: a CUDA tensor is required (got {t.device})")


def _fp8_cache_dtypes():
    import torch
    return (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())


def _check_attention(desc: AttnDesc, q, k_cache, v_cache, block_table, seq_lens, out, workspace, status,
                     fp8: bool, k_scale=None, v_scale=None, k_new=None, v_new=None) -> None:
    import torch
    rows = desc.num_seqs * desc.q_len
    cache = (desc.num_pages, desc.block_size, desc.num_kv_heads, desc.head_dim)
    cache_dt = _fp8_cache_dtypes() if fp8 else torch.bfloat16
    _expect(q, "q", torch.bfloat16, (rows, desc.num_q_heads, desc.head_dim))
    _expect(k_cache, "k_cache", cache_dt, cache)
    _expect(v_cache, "v_cache", cache_dt, cache)
    _expect(block_table, "block_table", torch.int32, (desc.num_seqs, desc.max_pages_per_seq))
    _expect(seq_lens, "seq_lens", torch.int32, (desc.num_seqs,))
    _expect(out, "out", torch.bfloat16 if desc.out_dtype == PA_OUT_BF16 else torch.float32,
            (rows, desc.num_q_heads, desc.head_dim))
    if workspace is not None and not isinstance(workspace, int) and workspace.device.type != "cuda":
        raise ValueError("workspace: a CUDA tensor is required")
    _expect(status, "status", torch.int32)
    _expect(k_scale, "k_scale", torch.float32, (desc.num_kv_heads,))
    _expect(v_scale, "v_scale", torch.float32, (desc.num_kv_heads,))
    _expect(k_new, "k_new", torch.bfloat16, (desc.num_seqs, desc.num_kv_heads, desc.head_dim))
    _expect(v_new, "v_new", torch.bfloat16, (desc.num_seqs, desc.num_kv_heads, desc.head_dim))


def _check_reshape(k_new, v_new, k_cache, v_cache, slot_mapping, status, fp8: bool) -> None:
    import torch
    n = int(slot_mapping.shape[0])
    _, _, hkv, d = k_cache.shape
    _expect(k_cache, "k_cache", _fp8_cache_dtypes() if fp8 else torch.bfloat16)
    _expect(v_cache, "v_cache", _fp8_cache_dtypes() if fp8 else torch.bfloat16, tuple(k_cache.shape))
    _expect(k_new, "k_new", torch.bfloat16, (n, hkv, d))
    _expect(v_new, "v_new", torch.bfloat16, (n, hkv, d))
    _expect(slot_mapping, "slot_mapping", torch.int64, (n,))
    _expect(status, "status", torch.int32)


def reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping, status=None, stream=None) -> None:
    """Write new K/V rows ([N, Hkv, D] bf16) into cache slots (int64 [N])."""
    num_pages, block_size, num_kv_heads, head_dim = k_cache.shape
    _check_reshape(k_new, v_new, k_cache, v_cache, slot_mapping, status, fp8=False)
    rc = load_library().pa_reshape_and_cache(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), int(slot_mapping.shape[0]),
        num_kv_heads, head_dim, block_size, num_pages, _ptr(status), _stream(stream))
    _check(rc, "pa_reshape_and_cache")


def paged_attention_decode(q, k_cache, v_cache, block_table, seq_lens, desc: AttnDesc, out, workspace=None,
                           status=None, stream=None) -> None:
    """out[b, h, :] = softmax(scale q K^T) V through the block table (q_len 1)."""
    _check_attention(desc, q, k_cache, v_cache, block_table, seq_lens, out, workspace, status, fp8=False)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().pa_paged_attention_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), ctypes.byref(desc), _ptr(out),
        _ptr(workspace), ws, _ptr(status), _stream(stream))
    _check(rc, "pa_paged_attention_decode")


def paged_attention_decode_append(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, desc: AttnDesc, out,
                                  workspace=None, status=None, stream=None) -> None:
    """reshape_and_cache of each sequence's new token (rows k_new, v_new
    [B, Hkv, D] bf16 into the slot of token seq_lens[b] - 1) fused with the
    decode that reads it: one kernel, the same result as the two calls."""
    _check_attention(desc, q, k_cache, v_cache, block_table, seq_lens, out, workspace, status, fp8=False,
                     k_new=k_new, v_new=v_new)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().pa_paged_attention_decode_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        ctypes.byref(desc), _ptr(out), _ptr(workspace), ws, _ptr(status), _stream(stream))
    _check(rc, "pa_paged_attention_decode_append")


def paged_attention_decode_append_fp8(q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                                      desc: AttnDesc, out, workspace=None, status=None, stream=None) -> None:
    """The fused append and decode over an e4m3 cache (the new rows quantised
    as reshape_and_cache_fp8 does)."""
    _check_attention(desc, q, k_cache, v_cache, block_table, seq_lens, out, workspace, status, fp8=True,
                     k_scale=k_scale, v_scale=v_scale, k_new=k_new, v_new=v_new)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().pa_paged_attention_decode_append_fp8(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_table), _ptr(seq_lens), ctypes.byref(desc), _ptr(out), _ptr(workspace), ws, _ptr(status),
        _stream(stream))
    _check(rc, "pa_paged_attention_decode_append_fp8")


def paged_attention_decode_noalloc(q, k_cache, v_cache, block_table, seq_lens, desc: AttnDesc, out, status=None,
                                   stream=None) -> None:
    """Decode without a workspace argument (split partials in the library's
    device scratch array; calls that overlap on the GPU must be ordered)."""
    _check_attention(desc, q, k_cache, v_cache, block_table, seq_lens, out, None, status, fp8=False)
    rc = load_library().pa_paged_attention_decode_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), ctypes.byref(desc), _ptr(out),
        _ptr(status), _stream(stream))
    _check(rc, "pa_paged_attention_decode_noalloc")


def paged_attention_verify(q, k_cache, v_cache, block_table, seq_lens, desc: AttnDesc, out, workspace=None,
                           status=None, stream=None) -> None:
    """q_len > 1 rows per sequence, causal among them; q/out are [B*q_len, Hq, D]."""
    _check_attention(desc, q, k_cache, v_cache, block_table, seq_lens, out, workspace, status, fp8=False)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().pa_paged_attention_verify(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), ctypes.byref(desc), _ptr(out),
        _ptr(workspace), ws, _ptr(status), _stream(stream))
    _check(rc, "pa_paged_attention_verify")


def reshape_and_cache_fp8(k_new, v_new, k_cache, v_cache, slot_mapping, k_scale, v_scale, status=None,
                          stream=None) -> None:
    """Quantise new K/V rows ([N, Hkv, D] bf16) into e4m3 cache slots (uint8
    caches [P, BS, Hkv, D]; float32 scales [Hkv])."""
    import torch
    num_pages, block_size, num_kv_heads, head_dim = k_cache.shape
    _check_reshape(k_new, v_new, k_cache, v_cache, slot_mapping, status, fp8=True)
    _expect(k_scale, "k_scale", torch.float32, (num_kv_heads,))
    _expect(v_scale, "v_scale", torch.float32, (num_kv_heads,))
    rc = load_library().pa_reshape_and_cache_fp8(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), _ptr(k_scale), _ptr(v_scale),
        int(slot_mapping.shape[0]), num_kv_heads, head_dim, block_size, num_pages, _ptr(status), _stream(stream))
    _check(rc, "pa_reshape_and_cache_fp8")


def paged_attention_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, desc: AttnDesc, out,
                               workspace=None, status=None, stream=None) -> None:
    """Decode over an e4m3 cache: K = code x k_scale[kv head], V likewise."""
    _check_attention(desc, q, k_cache, v_cache, block_table, seq_lens, out, workspace, status, fp8=True,
                     k_scale=k_scale, v_scale=v_scale)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().pa_paged_attention_decode_fp8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens),
        ctypes.byref(desc), _ptr(out), _ptr(workspace), ws, _ptr(status), _stream(stream))
    _check(rc, "pa_paged_attention_decode_fp8")


def paged_attention_verify_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, desc: AttnDesc, out,
                               workspace=None, status=None, stream=None) -> None:
    """Verify (q_len > 1) over an e4m3 cache: K = code x k_scale[kv head], V likewise."""
    _check_attention(desc, q, k_cache, v_cache, block_table, seq_lens, out, workspace, status, fp8=True,
                     k_scale=k_scale, v_scale=v_scale)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().pa_paged_attention_verify_fp8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens),
        ctypes.byref(desc), _ptr(out), _ptr(workspace), ws, _ptr(status), _stream(stream))
    _check(rc, "pa_paged_attention_verify_fp8")


def last_plan() -> dict:
    info = PlanInfo()
    _check(load_library().pa_last_plan(ctypes.byref(info)), "pa_last_plan")
    return info.as_dict()
