"""Seeded synthetic inputs shaped like the pages' workloads.

This module draws random numbers and lays out pages; it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can consume its
output without sharing any of the method.

Recipe (every draw comes from one ``torch.Generator`` seeded per problem):
  1. per-sequence context lengths (fixed, or uniform integers in a range);
  2. a random permutation of the physical page pool; sequence b takes the next
     ceil(L_b / BS) entries of it as its block-table row, so every sequence's
     pages lie scattered at random through one shared pool;
  3. q ~ N(0, 1) in bf16, shape [B * q_len, Hq, D];
  4. for each layer, k_cache and v_cache ~ N(0, 1) in bf16, [P, BS, Hkv, D]
     (unused slots hold random data too, or NaN with ``poison_unused``);
     with ``kv_fp8`` the caches hold e4m3 codes instead: N(0, 1) draws clipped
     to +-6.5, divided by the per-KV-head scale and cast by torch's
     float8_e4m3fn type, with scales k_scale[h] = (1 + h/4) / 64 and
     v_scale[h] = (1 + h/8) / 48 (so |x / scale| < 448), NaN code 0x7F in
     poisoned slots.
Unused block-table entries are -1 so that a kernel that reads past the pages
of a sequence trips its bounds check.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16_NAN_BITS = 0x7FC0
E4M3_NAN_CODE = 0x7F


@dataclass
class PagedProblem:
    num_seqs: int
    q_len: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_pages: int
    scale: float
    seq_lens: torch.Tensor          # int32 [B]
    block_table: torch.Tensor       # int32 [B, max_pages_per_seq]
    q: list = field(default_factory=list)        # per layer: bf16 [B*q_len, Hq, D]
    k_cache: list = field(default_factory=list)  # per layer: bf16 [P, BS, Hkv, D]
    v_cache: list = field(default_factory=list)
    kv_fp8: bool = False
    k_scale: list = field(default_factory=list)  # fp8 only, per layer: float32 [Hkv]
    v_scale: list = field(default_factory=list)

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.num_seqs else 0

    @property
    def num_layers(self) -> int:
        return len(self.k_cache)

    def context_tokens(self) -> int:
        return int(self.seq_lens.to(torch.int64).sum().item())

    def new_token_slots(self) -> torch.Tensor:
        """int64 slot of each of the q_len newest tokens of every sequence,
        ordered like the q rows (sequence, new row): the slot_mapping a caller
        hands to reshape_and_cache after appending those tokens."""
        slots = []
        bt = self.block_table.cpu()
        for b, L in enumerate(self.seq_lens.cpu().tolist()):
            for t in range(L - self.q_len, L):
                slots.append(int(bt[b, t // self.block_size]) * self.block_size + t % self.block_size)
        return torch.tensor(slots, dtype=torch.int64)


def _randn_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(torch.bfloat16)


def fp8_scales(num_kv_heads: int, device: str = "cpu"):
    """The synthetic per-KV-head scales of an fp8 cache (K, V)."""
    h = torch.arange(num_kv_heads, dtype=torch.float32, device=device)
    return (1 + h / 4) / 64, (1 + h / 8) / 48


def _e4m3_codes(shape, gen, device, scale):
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device).clamp_(-6.5, 6.5)
    x /= scale.view(1, 1, -1, 1)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def make_problem(seed: int, *, num_seqs: int, seq_lens, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, block_size: int, q_len: int = 1, num_layers: int = 1,
                 pool_pages: int | None = None, pool_factor: float = 1.1, scale: float | None = None,
                 device: str = "cpu", poison_unused: bool = False, kv_fp8: bool = False) -> PagedProblem:
    """Draw one paged-attention problem.

    ``seq_lens`` is an int (same length for all), a list of ints, or a tuple
    ("uniform", lo, hi) for integers drawn uniformly in [lo, hi].
    ``pool_pages`` fixes the pool size; otherwise it is ceil(pool_factor * pages used).
    Random draws happen on ``device`` (a CUDA generator when device is cuda).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    if isinstance(seq_lens, int):
        lens = [seq_lens] * num_seqs
    elif isinstance(seq_lens, tuple) and seq_lens[0] == "uniform":
        lo, hi = seq_lens[1], seq_lens[2]
        lens = torch.randint(lo, hi + 1, (num_seqs,), generator=gen, device=device).cpu().tolist()
    else:
        lens = list(seq_lens)
    assert len(lens) == num_seqs
    pages_per_seq = [math.ceil(L / block_size) for L in lens]
    used = sum(pages_per_seq)
    if pool_pages is None:
        pool_pages = max(1, math.ceil(pool_factor * used))
    assert pool_pages >= used, "page pool smaller than the pages in use"
    max_pages = max([1] + pages_per_seq)

    perm = torch.randperm(pool_pages, generator=gen, device=device).cpu()
    block_table = torch.full((num_seqs, max_pages), -1, dtype=torch.int32)
    cursor = 0
    for b, n in enumerate(pages_per_seq):
        block_table[b, :n] = perm[cursor:cursor + n].to(torch.int32)
        cursor += n

    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    prob = PagedProblem(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, pool_pages,
                        float(scale), torch.tensor(lens, dtype=torch.int32), block_table, kv_fp8=kv_fp8)
    cache_shape = (pool_pages, block_size, num_kv_heads, head_dim)
    for _ in range(num_layers):
        prob.q.append(_randn_bf16((num_seqs * q_len, num_q_heads, head_dim), gen, device))
        if kv_fp8:
            ks, vs = fp8_scales(num_kv_heads, device)
            prob.k_scale.append(ks)
            prob.v_scale.append(vs)
            prob.k_cache.append(_e4m3_codes(cache_shape, gen, device, ks))
            prob.v_cache.append(_e4m3_codes(cache_shape, gen, device, vs))
        else:
            prob.k_cache.append(_randn_bf16(cache_shape, gen, device))
            prob.v_cache.append(_randn_bf16(cache_shape, gen, device))
    if poison_unused:
        poison_unused_slots(prob)
    return prob


def poison_unused_slots(prob: PagedProblem) -> None:
    """Fill every cache slot no sequence uses with NaN (bf16 NaN bits, or the
    e4m3 NaN code in an fp8 cache)."""
    for kc, vc in zip(prob.k_cache, prob.v_cache):
        used = torch.zeros((prob.num_pages, prob.block_size), dtype=torch.bool)
        bt = prob.block_table.cpu()
        for b, L in enumerate(prob.seq_lens.tolist()):
            for lp in range((L + prob.block_size - 1) // prob.block_size):
                n = min(prob.block_size, L - lp * prob.block_size)
                used[int(bt[b, lp]), :n] = True
        mask = (~used).to(kc.device)
        if prob.kv_fp8:
            nan = torch.tensor(E4M3_NAN_CODE, dtype=torch.uint8, device=kc.device)
        else:
            nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16, device=kc.device).view(torch.bfloat16)
        kc[mask] = nan
        vc[mask] = nan


def make_new_tokens(seed: int, num_tokens: int, num_kv_heads: int, head_dim: int, device: str = "cpu"):
    """Fresh K/V rows (bf16 N(0,1)) for reshape_and_cache."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    k = _randn_bf16((num_tokens, num_kv_heads, head_dim), gen, device)
    v = _randn_bf16((num_tokens, num_kv_heads, head_dim), gen, device)
    return k, v


# The five workloads of the pages, by name.  Sizes follow the pages: 24 query
# heads on 4 KV heads with head_dim 256 for the hybrid model, 32/8/128 for the
# dense control; pages of 16, 784 and 832 tokens.
WORKLOADS = {
    "decode_l512_bs16": dict(num_seqs=1, seq_lens=512, num_q_heads=24, num_kv_heads=4, head_dim=256,
                             block_size=16, pool_pages=64, scale=1.0 / 16, q_len=1, num_layers=1),
    "hybrid_step_l32768_bs784_x16": dict(num_seqs=1, seq_lens=32768, num_q_heads=24, num_kv_heads=4,
                                         head_dim=256, block_size=784, scale=1.0 / 16, q_len=1,
                                         num_layers=16),
    "batch32_uniform_bs784": dict(num_seqs=32, seq_lens=("uniform", 1024, 32768), num_q_heads=24,
                                  num_kv_heads=4, head_dim=256, block_size=784, scale=1.0 / 16, q_len=1,
                                  num_layers=1),
    "verify_b8_q16_l8192_bs832": dict(num_seqs=8, seq_lens=8192 + 16, num_q_heads=24, num_kv_heads=4,
                                      head_dim=256, block_size=832, scale=1.0 / 16, q_len=16,
                                      num_layers=1),
    # wider GQA: 48 query heads on the same 4 KV heads (12 per group)
    # the hybrid layer over an fp8 e4m3 cache (half the KV bytes)
    "decode_fp8_l32768_bs784": dict(num_seqs=1, seq_lens=32768, num_q_heads=24, num_kv_heads=4,
                                    head_dim=256, block_size=784, scale=1.0 / 16, q_len=1,
                                    num_layers=16, kv_fp8=True),
    "decode_g12_l32768_bs784": dict(num_seqs=1, seq_lens=32768, num_q_heads=48, num_kv_heads=4,
                                    head_dim=256, block_size=784, scale=1.0 / 16, q_len=1,
                                    num_layers=16),
    # the dense control at full depth: 32 query heads on 8 KV heads, head_dim
    # 128, 16-token pages (the same 4096 B of K+V per token as the hybrid)
    "decode_dense_l32768_bs16": dict(num_seqs=1, seq_lens=32768, num_q_heads=32, num_kv_heads=8,
                                     head_dim=128, block_size=16, scale=1.0 / math.sqrt(128), q_len=1,
                                     num_layers=16),
    # speculative verify with 12 query heads per KV head: 5 positions x 12 heads
    # = 60 rows per (sequence, KV head), 32 sequences of 2048 positions
    "verify_g12_b32_q5_l2048_bs784": dict(num_seqs=32, seq_lens=2048, num_q_heads=48, num_kv_heads=4,
                                          head_dim=256, block_size=784, scale=1.0 / 16, q_len=5,
                                          num_layers=1),
    # a chunked-prefill step: 2048 new rows of one sequence over 14336 cached tokens
    "prefill_q2048_l16384_bs832": dict(num_seqs=1, seq_lens=16384, num_q_heads=24, num_kv_heads=4,
                                       head_dim=256, block_size=832, scale=1.0 / 16, q_len=2048,
                                       num_layers=1),
}

SWEEP_DEPTHS = [500, 1024, 2048, 4096, 6144, 8192, 12288, 16384, 20480, 24576, 32768]


def sweep_workload(depth: int, dense: bool, num_layers: int = 16) -> dict:
    """One depth of the context sweep: the hybrid shape on 832-token pages, or
    the dense control (32 query / 8 KV heads, head_dim 128, 16-token pages)."""
    if dense:
        return dict(num_seqs=1, seq_lens=depth, num_q_heads=32, num_kv_heads=8, head_dim=128,
                    block_size=16, scale=1.0 / math.sqrt(128), q_len=1, num_layers=num_layers)
    return dict(num_seqs=1, seq_lens=depth, num_q_heads=24, num_kv_heads=4, head_dim=256,
                block_size=832, scale=1.0 / 16, q_len=1, num_layers=num_layers)
