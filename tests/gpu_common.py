"""GPU-side test helpers: run the library on a problem and compare with the oracle.

The parity gate (the stated tolerance for bf16 inputs with fp32 accumulation):
  * every output finite;
  * max |gpu - oracle| <= 2e-3 over all elements;
  * |gpu - oracle| / |oracle| <= 1e-2 wherever |oracle| >= 0.2 (= 2e-3 / 1e-2,
    the magnitude above which the relative bound is the tighter one);
  * relative L2 error per (row, head) <= ``rel_l2`` = 1e-4, a tighter internal
    target (fp32 accumulation; the verify kernel carries P as a bf16 head plus
    a bf16 residual into its tensor-core P.V product).
A row whose oracle output is exactly zero (no visible key) must be exactly zero.
"""
from __future__ import annotations

import numpy as np
import torch

import paged_attention_decode_split_gb300 as pa

ATOL = 2e-3
RTOL = 1e-2
REL_L2_DECODE = 1e-4
REL_L2_VERIFY = 1e-4


def to_dev(prob, layer=0, device="cuda"):
    return (prob.q[layer].to(device), prob.k_cache[layer].to(device), prob.v_cache[layer].to(device),
            prob.block_table.to(device), prob.seq_lens.to(device))


def desc_for(prob, *, num_splits=0, out_dtype=pa.PA_OUT_F32, max_seq_len=None, window=0, flags=0):
    return pa.make_desc(num_seqs=prob.num_seqs, q_len=prob.q_len, num_q_heads=prob.num_q_heads,
                        num_kv_heads=prob.num_kv_heads, head_dim=prob.head_dim, block_size=prob.block_size,
                        max_pages_per_seq=prob.max_pages_per_seq,
                        max_seq_len=prob.max_seq_len if max_seq_len is None else max_seq_len,
                        num_pages=prob.num_pages, scale=prob.scale, out_dtype=out_dtype, num_splits=num_splits,
                        window=window, flags=flags)


def scales_dev(prob, layer=0, device="cuda"):
    return prob.k_scale[layer].to(device), prob.v_scale[layer].to(device)


def run_attention(prob, layer=0, *, num_splits=0, out_dtype=pa.PA_OUT_F32, max_seq_len=None, tensors=None,
                  window=0, flags=0):
    """Runs decode (q_len 1; over the fp8 cache for an fp8 problem) or verify
    through the C ABI; returns (out on CPU, status, plan)."""
    q, kc, vc, bt, sl = tensors if tensors is not None else to_dev(prob, layer)
    desc = desc_for(prob, num_splits=num_splits, out_dtype=out_dtype, max_seq_len=max_seq_len, window=window,
                    flags=flags)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device=q.device)
    dtype = torch.float32 if out_dtype == pa.PA_OUT_F32 else torch.bfloat16
    out = torch.full((prob.num_seqs * prob.q_len, prob.num_q_heads, prob.head_dim), float("nan"), dtype=dtype,
                     device=q.device)
    status = torch.zeros(1, dtype=torch.int32, device=q.device)
    if prob.kv_fp8:
        ks, vs = scales_dev(prob, layer, q.device)
        fn = pa.paged_attention_decode_fp8 if prob.q_len == 1 else pa.paged_attention_verify_fp8
        fn(q, kc, vc, ks, vs, bt, sl, desc, out, ws, status)
    else:
        fn = pa.paged_attention_decode if prob.q_len == 1 else pa.paged_attention_verify
        fn(q, kc, vc, bt, sl, desc, out, ws, status)
    torch.cuda.synchronize()
    return out.float().cpu(), int(status.item()), pa.last_plan()


def oracle_out(oracle_mod, prob, layer=0, rows=None, window=0):
    """Oracle output [rows, Hq, D] (float64); ``rows`` restricts to some sequences."""
    q, bt, sl = prob.q[layer].cpu(), prob.block_table.cpu(), prob.seq_lens.cpu()
    if rows is not None:
        idx = torch.tensor(rows)
        qi = torch.cat([torch.arange(b * prob.q_len, (b + 1) * prob.q_len) for b in rows])
        q, bt, sl = q[qi].contiguous(), bt[idx].contiguous(), sl[idx].contiguous()
    if prob.kv_fp8:
        return oracle_mod.paged_attention_fp8(q, prob.k_cache[layer].cpu(), prob.v_cache[layer].cpu(),
                                              prob.k_scale[layer].cpu(), prob.v_scale[layer].cpu(), bt.numpy(),
                                              sl.numpy(), prob.scale, q_len=prob.q_len, window=window)
    return oracle_mod.paged_attention(q, prob.k_cache[layer].cpu(), prob.v_cache[layer].cpu(), bt.numpy(),
                                      sl.numpy(), prob.scale, q_len=prob.q_len, window=window)


def assert_cache_written(oracle_mod, k_before, v_before, k_new, v_new, slots, k_dev, v_dev):
    """The bf16 caches that the GPU's reshape_and_cache wrote (k_dev, v_dev)
    equal, bit for bit, the oracle's scatter of the same new rows into CPU
    copies of the caches as they were before the call.  Tests that hand a
    GPU-written cache to the oracle check it with this first, so a slot
    error cannot be read identically by both sides."""
    from tests.helpers import bits
    k_ref, v_ref = bits(k_before).copy(), bits(v_before).copy()
    oracle_mod.reshape_and_cache(bits(k_new), bits(v_new), k_ref, v_ref, np.asarray(slots.cpu().numpy(), np.int64))
    assert np.array_equal(bits(k_dev), k_ref), "reshape_and_cache wrote K differently from the oracle"
    assert np.array_equal(bits(v_dev), v_ref), "reshape_and_cache wrote V differently from the oracle"


def parity_report(gpu: torch.Tensor, ref: np.ndarray) -> dict:
    g = gpu.double().numpy()
    err = np.abs(g - ref)
    big = np.abs(ref) >= ATOL / RTOL
    num = np.linalg.norm((g - ref).reshape(-1, g.shape[-1]), axis=1)
    den = np.linalg.norm(ref.reshape(-1, g.shape[-1]), axis=1)
    nz = den > 0
    return {
        "finite": bool(np.isfinite(g).all()),
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_rel_big": float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
        "max_rel_l2": float((num[nz] / den[nz]).max()) if nz.any() else 0.0,
        "zero_rows_exact": bool(np.all(g.reshape(-1, g.shape[-1])[~nz] == 0.0)),
    }


def assert_parity(gpu: torch.Tensor, ref: np.ndarray, rel_l2: float = REL_L2_DECODE, what: str = "") -> dict:
    r = parity_report(gpu, ref)
    assert r["finite"], f"{what}: non-finite output"
    assert r["max_abs"] <= ATOL, f"{what}: max abs err {r['max_abs']:.3g} > {ATOL}"
    assert r["max_rel_big"] <= RTOL, f"{what}: max rel err {r['max_rel_big']:.3g} > {RTOL}"
    assert r["max_rel_l2"] <= rel_l2, f"{what}: rel L2 {r['max_rel_l2']:.3g} > {rel_l2}"
    assert r["zero_rows_exact"], f"{what}: rows without keys are not exactly zero"
    return r
