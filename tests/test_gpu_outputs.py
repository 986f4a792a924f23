"""GPU parity of the ways results leave the kernels: the verify kernel's
staged epilogue (its rows copied out of shared memory, fp32 or bf16, as the
final output or as split records) and the few-split merge, whose warps each
take 1, 2 or 4 (row, head) pairs depending on how many pairs a call has, with
2, 4 or 8 split slots.  Small problems only reach one pair per warp, so these
cases use batches with enough rows: every (slots, pairs per warp) variant runs."""
import math

import numpy as np
import pytest
import torch

import paged_attention_decode_split_gb300 as pa
from paged_attention_decode_split_gb300 import _build
from paged_attention_decode_split_gb300.inputs import make_new_tokens, make_problem
from tests.gpu_common import (REL_L2_DECODE, REL_L2_VERIFY, assert_cache_written, assert_parity, oracle_out,
                              run_attention)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    pa.load_library()


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def write_new_rows(oracle_mod, prob, seed):
    """reshape_and_cache of the q_len newest tokens (GPU), checked bit for bit
    against the oracle's scatter before anything reads the cache."""
    k_new, v_new = make_new_tokens(seed, prob.num_seqs * prob.q_len, prob.num_kv_heads, prob.head_dim)
    slots = prob.new_token_slots()
    kc, vc = prob.k_cache[0].cuda(), prob.v_cache[0].cuda()
    pa.reshape_and_cache(k_new.cuda(), v_new.cuda(), kc, vc, slots.cuda())
    torch.cuda.synchronize()
    assert_cache_written(oracle_mod, prob.k_cache[0], prob.v_cache[0], k_new, v_new, slots, kc, vc)
    prob.k_cache[0], prob.v_cache[0] = kc.cpu(), vc.cpu()


def assert_bf16_close(out, ref):
    """bf16 output against the oracle rounded to bf16: one bf16 rounding on
    each side of a difference within the fp32 gate."""
    ref_bf16 = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    got = out.double().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - ref_bf16).max() <= 2e-3 + 2 * 2.0 ** -8 * np.abs(ref).max()


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("d", [256, 128])
def test_verify_bf16_output(oracle_mod, splits, d):
    """One split: the CTA's staged rows are the bf16 output; three: fp32
    split records, merged into bf16."""
    if d == 256:
        prob = make_problem(63, num_seqs=2, seq_lens=[700, 40], num_q_heads=24, num_kv_heads=4, head_dim=256,
                            block_size=832, q_len=16, scale=1 / 16, poison_unused=True)
    else:
        prob = make_problem(64, num_seqs=2, seq_lens=[700, 40], num_q_heads=32, num_kv_heads=8, head_dim=128,
                            block_size=16, q_len=16, scale=1 / math.sqrt(128), poison_unused=True)
    write_new_rows(oracle_mod, prob, 21)
    out, status, plan = run_attention(prob, out_dtype=pa.PA_OUT_BF16, num_splits=splits)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05 and plan["num_splits"] == splits
    assert_bf16_close(out, oracle_out(oracle_mod, prob))


@pytest.mark.parametrize("splits", [1, 2])
def test_verify_fp8_bf16_output(oracle_mod, splits):
    prob = make_problem(65, num_seqs=2, seq_lens=[900, 33], num_q_heads=24, num_kv_heads=4, head_dim=256,
                        block_size=784, q_len=16, scale=1 / 16, kv_fp8=True, poison_unused=True)
    out, status, plan = run_attention(prob, out_dtype=pa.PA_OUT_BF16, num_splits=splits)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05 and plan["num_splits"] == splits
    assert_bf16_close(out, oracle_out(oracle_mod, prob))


# seqs x 16 rows x 24 heads (row, head) pairs: 4 sequences give 1536 pairs (2
# per merge warp on 152 SMs), 16 give 6144 (4 per warp, or 2 with 8 slots)
@pytest.mark.parametrize("splits", [2, 3, 7])
@pytest.mark.parametrize("seqs", [4, 16])
def test_verify_few_split_merge_pairs_per_warp(oracle_mod, splits, seqs):
    lens = [300 + 39 * i for i in range(seqs)]  # split counts 2, 3, 7 come out exactly as forced
    prob = make_problem(71 + seqs + splits, num_seqs=seqs, seq_lens=lens, num_q_heads=24, num_kv_heads=4,
                        head_dim=256, block_size=832, q_len=16, scale=1 / 16, poison_unused=True)
    write_new_rows(oracle_mod, prob, 23)
    pairs = seqs * 16 * 24
    assert pairs > 8 * sm_count()  # more than one pair per merge warp
    out, status, plan = run_attention(prob, num_splits=splits)
    assert status == 0 and plan["num_splits"] == splits
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what=f"merge seqs={seqs} splits={splits}")


@pytest.mark.parametrize("splits", [2, 5])
@pytest.mark.parametrize("out_dtype", [pa.PA_OUT_F32, pa.PA_OUT_BF16])
def test_decode_few_split_merge_wide_batch(oracle_mod, splits, out_dtype):
    """64 sequences x 24 heads = 1536 pairs: two pairs per merge warp."""
    lens = [1 + (97 * i) % 1500 for i in range(64)]
    prob = make_problem(81 + splits, num_seqs=64, seq_lens=lens, num_q_heads=24, num_kv_heads=4, head_dim=256,
                        block_size=16, scale=1 / 16, poison_unused=True)
    out, status, plan = run_attention(prob, num_splits=splits, out_dtype=out_dtype)
    assert status == 0 and plan["num_splits"] == splits
    ref = oracle_out(oracle_mod, prob)
    if out_dtype == pa.PA_OUT_BF16:
        assert_bf16_close(out, ref)
    else:
        assert_parity(out, ref, rel_l2=REL_L2_DECODE, what=f"wide batch splits={splits}")
