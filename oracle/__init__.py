"""CPU fp64 oracle for paged attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
path (``paged_attention_decode_split_gb300``) never imports, links or runs it,
and it shares no code with the CUDA kernels.

The arithmetic lives in ``pa_oracle.c`` (plain C, IEEE double), compiled with
gcc into ``oracle/_build/liboracle.so`` on first use (``build()`` compiles it
eagerly).  This module only marshals numpy arrays into it.

Inputs use raw bf16 bit patterns (``numpy.uint16``); outputs are float64.
Parity is pinned by ``tests/test_oracle.py`` against closed forms, invariants
and a brute-force dense softmax; no function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` with gcc (no -ffast-math: IEEE semantics kept)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_reshape_and_cache.restype = ctypes.c_int
            lib.oracle_reshape_and_cache.argtypes = [
                _u16p, _u16p, _u16p, _u16p, _i64p, ctypes.c_int64,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64]
            common = [_u16p, _u16p, _u16p, _i32p, _i32p,
                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_double]
            lib.oracle_paged_attention.restype = ctypes.c_int
            lib.oracle_paged_attention.argtypes = common + [_f64p, ctypes.c_int]
            lib.oracle_paged_attention_window.restype = ctypes.c_int
            lib.oracle_paged_attention_window.argtypes = common + [ctypes.c_int64, _f64p, ctypes.c_int]
            lib.oracle_attention_partial.restype = ctypes.c_int
            lib.oracle_attention_partial.argtypes = common + [
                ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _f64p, _f64p, _f64p]
            lib.oracle_lse_combine.restype = ctypes.c_int
            lib.oracle_lse_combine.argtypes = [_f64p, _f64p, _f64p, ctypes.c_int, ctypes.c_int, _f64p]
            lib.oracle_hybrid_page_tokens.restype = ctypes.c_int64
            lib.oracle_e4m3_encode.restype = ctypes.c_int
            lib.oracle_e4m3_encode.argtypes = [_f32p, _u8p, ctypes.c_int64]
            lib.oracle_e4m3_decode.restype = ctypes.c_int
            lib.oracle_e4m3_decode.argtypes = [_u8p, _f64p, ctypes.c_int64]
            lib.oracle_reshape_and_cache_fp8.restype = ctypes.c_int
            lib.oracle_reshape_and_cache_fp8.argtypes = [
                _u16p, _u16p, _u8p, _u8p, _i64p, ctypes.c_int64,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, _f32p, _f32p]
            lib.oracle_paged_attention_fp8.restype = ctypes.c_int
            lib.oracle_paged_attention_fp8.argtypes = [
                _u16p, _u8p, _u8p, _f32p, _f32p, _i32p, _i32p,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_double,
                ctypes.c_int64, _f64p, ctypes.c_int]
            lib.oracle_hybrid_page_tokens.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctype)


def _bits(a) -> np.ndarray:
    """Accept a numpy uint16 array or a torch bf16 tensor; return uint16 bits."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16, "bf16 data is passed as uint16 bit patterns"
        return np.ascontiguousarray(a)
    import torch  # only for the tensor -> bits view
    assert a.dtype == torch.bfloat16
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(a) -> np.ndarray:
    if not isinstance(a, np.ndarray):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def reshape_and_cache(k_new, v_new, k_cache: np.ndarray, v_cache: np.ndarray, slot_mapping) -> None:
    """Scatter new K/V rows into cache slots, in place on the uint16 caches."""
    k_new, v_new = _bits(k_new), _bits(v_new)
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    slots = slot_mapping if isinstance(slot_mapping, np.ndarray) else slot_mapping.detach().cpu().numpy()
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    num_pages, block_size, num_kv_heads, head_dim = k_cache.shape
    rc = _load().oracle_reshape_and_cache(
        _ptr(k_new, _u16p), _ptr(v_new, _u16p), _ptr(k_cache, _u16p), _ptr(v_cache, _u16p),
        _ptr(slots, _i64p), slots.shape[0], num_kv_heads, head_dim, block_size, num_pages)
    if rc != 0:
        raise ValueError(f"oracle_reshape_and_cache failed ({rc})")


def _problem(q, k_cache, v_cache, block_table, seq_lens, scale, q_len):
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    bt, sl = _i32(block_table), _i32(seq_lens)
    num_pages, block_size, num_kv_heads, head_dim = kb.shape
    rows, num_q_heads, hd = qb.shape
    assert hd == head_dim and vb.shape == kb.shape
    num_seqs = sl.shape[0]
    assert rows == num_seqs * q_len and bt.shape[0] == num_seqs
    keep = (qb, kb, vb, bt, sl)
    args = [_ptr(qb, _u16p), _ptr(kb, _u16p), _ptr(vb, _u16p), _ptr(bt, _i32p), _ptr(sl, _i32p),
            num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, bt.shape[1],
            num_pages, float(scale)]
    return keep, args, (rows, num_q_heads, head_dim)


def paged_attention(q, k_cache, v_cache, block_table, seq_lens, scale: float, q_len: int = 1,
                    num_threads: int | None = None, window: int = 0) -> np.ndarray:
    """Exact softmax attention through the block table; returns float64 [rows, Hq, D].
    window > 0: each row sees only its last `window` visible keys (sliding window)."""
    keep, args, shape = _problem(q, k_cache, v_cache, block_table, seq_lens, scale, q_len)
    out = np.zeros(shape, dtype=np.float64)
    if num_threads is None:
        num_threads = os.cpu_count() or 1
    if window:
        rc = _load().oracle_paged_attention_window(*args, int(window), _ptr(out, _f64p), int(num_threads))
    else:
        rc = _load().oracle_paged_attention(*args, _ptr(out, _f64p), int(num_threads))
    del keep
    if rc != 0:
        raise ValueError(f"oracle_paged_attention failed ({rc})")
    return out


def attention_partial(q, k_cache, v_cache, block_table, seq_lens, scale: float, row: int, head: int,
                      t_begin: int, t_end: int, q_len: int = 1):
    """One split: attention of (row, head) over keys [t_begin, t_end). Returns (o, m, l)."""
    keep, args, shape = _problem(q, k_cache, v_cache, block_table, seq_lens, scale, q_len)
    o = np.zeros(shape[2], dtype=np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    rc = _load().oracle_attention_partial(*args, row, head, t_begin, t_end, _ptr(o, _f64p),
                                          ctypes.byref(m), ctypes.byref(l))
    del keep
    if rc != 0:
        raise ValueError(f"oracle_attention_partial failed ({rc})")
    return o, m.value, l.value


def lse_combine(o_parts: np.ndarray, m_parts: np.ndarray, l_parts: np.ndarray) -> np.ndarray:
    """Merge split results: weights l_i exp(m_i - max m), normalised."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    m_parts = np.ascontiguousarray(m_parts, dtype=np.float64)
    l_parts = np.ascontiguousarray(l_parts, dtype=np.float64)
    n, head_dim = o_parts.shape
    out = np.zeros(head_dim, dtype=np.float64)
    rc = _load().oracle_lse_combine(_ptr(o_parts, _f64p), _ptr(m_parts, _f64p), _ptr(l_parts, _f64p),
                                    n, head_dim, _ptr(out, _f64p))
    if rc != 0:
        raise ValueError(f"oracle_lse_combine failed ({rc})")
    return out


def hybrid_page_tokens(state_page_bytes: int, attn_bytes_per_token: int, alignment: int) -> int:
    """Shared page length of a hybrid attention/recurrent-state cache: the state
    page in attention tokens, rounded up to whole alignment groups (-1 if an
    argument is not positive)."""
    return int(_load().oracle_hybrid_page_tokens(state_page_bytes, attn_bytes_per_token, alignment))


# -- fp8 e4m3 KV cache --------------------------------------------------------------

def _np(a, dtype) -> np.ndarray:
    if not isinstance(a, np.ndarray):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=dtype)


def _u8(a) -> np.ndarray:
    """Accept a numpy uint8 array or a torch uint8 / float8_e4m3fn tensor."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint8
        return np.ascontiguousarray(a)
    import torch  # only for the tensor -> bytes view
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.uint8).numpy())


def e4m3_encode(x) -> np.ndarray:
    """binary32 values -> e4m3 codes (nearest, ties to even, saturating to +-448)."""
    xf = _np(x, np.float32)
    out = np.zeros(xf.shape, dtype=np.uint8)
    if _load().oracle_e4m3_encode(_ptr(xf, _f32p), _ptr(out, _u8p), xf.size) != 0:
        raise ValueError("oracle_e4m3_encode failed")
    return out


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 codes -> their exact values as float64 (NaN for the NaN codes)."""
    c = _u8(codes)
    out = np.zeros(c.shape, dtype=np.float64)
    if _load().oracle_e4m3_decode(_ptr(c, _u8p), _ptr(out, _f64p), c.size) != 0:
        raise ValueError("oracle_e4m3_decode failed")
    return out


def reshape_and_cache_fp8(k_new, v_new, k_cache: np.ndarray, v_cache: np.ndarray, slot_mapping,
                          k_scale, v_scale) -> None:
    """Quantise new bf16 K/V rows into uint8 e4m3 cache slots, in place:
    code = e4m3(x / scale[kv_head]) with the division in binary32."""
    k_new, v_new = _bits(k_new), _bits(v_new)
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    slots = _np(slot_mapping, np.int64)
    ks, vs = _np(k_scale, np.float32), _np(v_scale, np.float32)
    num_pages, block_size, num_kv_heads, head_dim = k_cache.shape
    assert ks.shape == (num_kv_heads,) and vs.shape == (num_kv_heads,)
    rc = _load().oracle_reshape_and_cache_fp8(
        _ptr(k_new, _u16p), _ptr(v_new, _u16p), _ptr(k_cache, _u8p), _ptr(v_cache, _u8p),
        _ptr(slots, _i64p), slots.shape[0], num_kv_heads, head_dim, block_size, num_pages,
        _ptr(ks, _f32p), _ptr(vs, _f32p))
    if rc != 0:
        raise ValueError(f"oracle_reshape_and_cache_fp8 failed ({rc})")


def paged_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, scale: float,
                        q_len: int = 1, num_threads: int | None = None, window: int = 0) -> np.ndarray:
    """Exact softmax attention over an fp8 cache (K = decoded code x k_scale[kv
    head], V likewise); returns float64 [rows, Hq, D]."""
    qb, kb, vb = _bits(q), _u8(k_cache), _u8(v_cache)
    bt, sl = _i32(block_table), _i32(seq_lens)
    ks, vs = _np(k_scale, np.float32), _np(v_scale, np.float32)
    num_pages, block_size, num_kv_heads, head_dim = kb.shape
    rows, num_q_heads, hd = qb.shape
    assert hd == head_dim and vb.shape == kb.shape
    assert ks.shape == (num_kv_heads,) and vs.shape == (num_kv_heads,)
    num_seqs = sl.shape[0]
    assert rows == num_seqs * q_len and bt.shape[0] == num_seqs
    out = np.zeros((rows, num_q_heads, head_dim), dtype=np.float64)
    if num_threads is None:
        num_threads = os.cpu_count() or 1
    rc = _load().oracle_paged_attention_fp8(
        _ptr(qb, _u16p), _ptr(kb, _u8p), _ptr(vb, _u8p), _ptr(ks, _f32p), _ptr(vs, _f32p),
        _ptr(bt, _i32p), _ptr(sl, _i32p), num_seqs, q_len, num_q_heads, num_kv_heads, head_dim,
        block_size, bt.shape[1], num_pages, float(scale), int(window), _ptr(out, _f64p), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention_fp8 failed ({rc})")
    return out
