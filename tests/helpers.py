"""Test-side helpers: layout builders and a dense fp64 reference.

These are written independently of both the oracle and the CUDA path: the
paged layout is produced here from contiguous per-sequence K/V by direct
placement, and the dense reference is torch's own softmax in float64.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bit patterns (CPU copy)."""
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def place_in_pages(k_list, v_list, block_size: int, num_pages: int, seed: int, fill: float = 0.0):
    """Scatter contiguous per-sequence K/V ([L_b, Hkv, D] bf16) into a shared
    pool of ``num_pages`` pages in a random order.  Returns (k_cache, v_cache,
    block_table int32 [B, max_pages] with -1 padding)."""
    hkv, d = k_list[0].shape[1], k_list[0].shape[2]
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)
    k_cache = torch.full((num_pages, block_size, hkv, d), fill, dtype=torch.bfloat16)
    v_cache = torch.full((num_pages, block_size, hkv, d), fill, dtype=torch.bfloat16)
    pages = [math.ceil(k.shape[0] / block_size) for k in k_list]
    assert sum(pages) <= num_pages
    bt = torch.full((len(k_list), max([1] + pages)), -1, dtype=torch.int32)
    cur = 0
    for b, (k, v) in enumerate(zip(k_list, v_list)):
        for lp in range(pages[b]):
            phys = int(perm[cur])
            cur += 1
            bt[b, lp] = phys
            lo = lp * block_size
            hi = min(k.shape[0], lo + block_size)
            k_cache[phys, : hi - lo] = k[lo:hi]
            v_cache[phys, : hi - lo] = v[lo:hi]
    return k_cache, v_cache, bt


def dense_attention(q, k_list, v_list, scale: float, q_len: int, num_kv_heads: int,
                    window: int = 0) -> torch.Tensor:
    """torch fp64 softmax(Q K^T scale) V per sequence with the causal rule for
    the q_len new rows; query head h uses KV head h // (Hq / Hkv).  window > 0
    keeps only each row's last `window` visible keys."""
    rows, hq, d = q.shape
    g = hq // num_kv_heads
    out = torch.zeros(rows, hq, d, dtype=torch.float64)
    for b, (k, v) in enumerate(zip(k_list, v_list)):
        L = k.shape[0]
        kf = k.double()
        vf = v.double()
        for r in range(q_len):
            n = L - q_len + r + 1
            if n <= 0:
                continue
            a = max(0, n - window) if window > 0 else 0
            qr = q[b * q_len + r].double()  # [Hq, D]
            for h in range(hq):
                s = (kf[a:n, h // g, :] @ qr[h]) * scale
                p = torch.softmax(s, dim=0)
                out[b * q_len + r, h] = p @ vf[a:n, h // g, :]
    return out


def randn_bf16(shape, gen):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)
