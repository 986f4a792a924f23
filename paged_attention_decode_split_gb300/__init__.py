"""Paged-attention split-KV decode for GB300 (sm_103a): Python binding.

A thin layer over ``libpagedattn.so`` (the C ABI of ``include/pagedattn.h``).
It only marshals arguments; every step of the computation runs in the
library's CUDA kernels.  The library is loaded with ctypes (descriptions, plan
queries and the raw entry points); the tensor calls go through a small
compiled module (``binding/pa_binding.cpp``) that checks each tensor's element
type, shape, device and layout against the attention description -- the C ABI
cannot see a buffer's size -- and passes its device pointer and the current
CUDA stream to the C entry point.  If the library or the compiled module is
missing or cannot be loaded, every call raises -- there is no fallback.

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
_bind = None
_vp = ctypes.c_void_p

# the C entry points the compiled module calls (it takes their addresses from
# the library loaded here, so the process holds one copy of the library)
_BOUND_ENTRIES = ("pa_paged_attention_decode", "pa_paged_attention_verify", "pa_paged_attention_decode_fp8",
                  "pa_paged_attention_verify_fp8", "pa_paged_attention_decode_append",
                  "pa_paged_attention_decode_append_fp8", "pa_paged_attention_decode_noalloc", "pa_reshape_and_cache",
                  "pa_reshape_and_cache_fp8")


def _load_binding(lib):
    """Import the compiled tensor binding built beside the library and hand it
    the library's entry points."""
    import importlib.util
    import sysconfig

    import torch  # noqa: F401  (the module links against torch's libraries)
    path = os.path.join(_PKG, "_build", "_pa_binding" + sysconfig.get_config_var("EXT_SUFFIX"))
    if not os.path.exists(path):
        raise RuntimeError(f"compiled binding not found at {path}; build it with "
                           "`python -m paged_attention_decode_split_gb300._build`")
    spec = importlib.util.spec_from_file_location("_pa_binding", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    for name in _BOUND_ENTRIES:
        mod.set_entry(name, ctypes.cast(getattr(lib, name), ctypes.c_void_p).value)
    return mod


def load_library(path: str | None = None):
    """Load libpagedattn.so and the compiled tensor binding (both built by
    ``_build.build()``); raises if either is absent."""
    global _lib, _bind
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
        _bind = _load_binding(lib)
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


def _stream(stream) -> int:
    """The stream handle the binding takes: -1 for the current CUDA stream
    (read in C++), else the raw handle."""
    if stream is None:
        return -1
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedAttnError(status, what)


# Call kinds of the compiled binding's attention(); each maps to one C entry point.
_DECODE, _DECODE_APPEND, _VERIFY, _DECODE_FP8, _DECODE_APPEND_FP8, _VERIFY_FP8, _DECODE_NOALLOC = range(7)


def _bound():
    return _bind if _bind is not None else (load_library(), _bind)[1]


def reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping, status=None, stream=None) -> None:
    """Write new K/V rows ([N, Hkv, D] bf16) into cache slots (int64 [N])."""
    _check(_bound().reshape(False, k_new, v_new, k_cache, v_cache, slot_mapping, None, None, status,
                            _stream(stream)), "pa_reshape_and_cache")


def paged_attention_decode(q, k_cache, v_cache, block_table, seq_lens, desc: AttnDesc, out, workspace=None,
                           status=None, stream=None) -> None:
    """out[b, h, :] = softmax(scale q K^T) V through the block table (q_len 1)."""
    _check(_bound().attention(_DECODE, q, k_cache, v_cache, None, None, None, None, block_table, seq_lens,
                              ctypes.addressof(desc), out, workspace, status, _stream(stream)),
           "pa_paged_attention_decode")


def paged_attention_decode_append(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, desc: AttnDesc, out,
                                  workspace=None, status=None, stream=None) -> None:
    """reshape_and_cache of each sequence's new token (rows k_new, v_new
    [B, Hkv, D] bf16 into the slot of token seq_lens[b] - 1) fused with the
    decode that reads it: one kernel, the same result as the two calls."""
    _check(_bound().attention(_DECODE_APPEND, q, k_cache, v_cache, None, None, k_new, v_new, block_table, seq_lens,
                              ctypes.addressof(desc), out, workspace, status, _stream(stream)),
           "pa_paged_attention_decode_append")


def paged_attention_decode_append_fp8(q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                                      desc: AttnDesc, out, workspace=None, status=None, stream=None) -> None:
    """The fused append and decode over an e4m3 cache (the new rows quantised
    as reshape_and_cache_fp8 does)."""
    _check(_bound().attention(_DECODE_APPEND_FP8, q, k_cache, v_cache, k_scale, v_scale, k_new, v_new, block_table,
                              seq_lens, ctypes.addressof(desc), out, workspace, status, _stream(stream)),
           "pa_paged_attention_decode_append_fp8")


def paged_attention_decode_noalloc(q, k_cache, v_cache, block_table, seq_lens, desc: AttnDesc, out, status=None,
                                   stream=None) -> None:
    """Decode without a workspace argument (split partials in the library's
    device scratch array; calls that overlap on the GPU must be ordered)."""
    _check(_bound().attention(_DECODE_NOALLOC, q, k_cache, v_cache, None, None, None, None, block_table, seq_lens,
                              ctypes.addressof(desc), out, None, status, _stream(stream)),
           "pa_paged_attention_decode_noalloc")


def paged_attention_verify(q, k_cache, v_cache, block_table, seq_lens, desc: AttnDesc, out, workspace=None,
                           status=None, stream=None) -> None:
    """q_len > 1 rows per sequence, causal among them; q/out are [B*q_len, Hq, D]."""
    _check(_bound().attention(_VERIFY, q, k_cache, v_cache, None, None, None, None, block_table, seq_lens,
                              ctypes.addressof(desc), out, workspace, status, _stream(stream)),
           "pa_paged_attention_verify")


def reshape_and_cache_fp8(k_new, v_new, k_cache, v_cache, slot_mapping, k_scale, v_scale, status=None,
                          stream=None) -> None:
    """Quantise new K/V rows ([N, Hkv, D] bf16) into e4m3 cache slots (uint8
    caches [P, BS, Hkv, D]; float32 scales [Hkv])."""
    _check(_bound().reshape(True, k_new, v_new, k_cache, v_cache, slot_mapping, k_scale, v_scale, status,
                            _stream(stream)), "pa_reshape_and_cache_fp8")


def paged_attention_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, desc: AttnDesc, out,
                               workspace=None, status=None, stream=None) -> None:
    """Decode over an e4m3 cache: K = code x k_scale[kv head], V likewise."""
    _check(_bound().attention(_DECODE_FP8, q, k_cache, v_cache, k_scale, v_scale, None, None, block_table, seq_lens,
                              ctypes.addressof(desc), out, workspace, status, _stream(stream)),
           "pa_paged_attention_decode_fp8")


def paged_attention_verify_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, desc: AttnDesc, out,
                               workspace=None, status=None, stream=None) -> None:
    """Verify (q_len > 1) over an e4m3 cache: K = code x k_scale[kv head], V likewise."""
    _check(_bound().attention(_VERIFY_FP8, q, k_cache, v_cache, k_scale, v_scale, None, None, block_table, seq_lens,
                              ctypes.addressof(desc), out, workspace, status, _stream(stream)),
           "pa_paged_attention_verify_fp8")


def last_plan() -> dict:
    info = PlanInfo()
    _check(load_library().pa_last_plan(ctypes.byref(info)), "pa_last_plan")
    return info.as_dict()
