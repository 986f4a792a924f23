"""GPU parity of the sliding window (a query row sees only its last W
visible keys, the RTX 3090 page's 2048-position window): decode and verify
through the C ABI against the oracle's windowed attention, at window edges
that fall inside chunks and pages, with forced splits, and with the early
K/V flag (bit-identical to the default order)."""
import pytest
import torch

import paged_attention_decode_split_gb300 as pa
from paged_attention_decode_split_gb300 import _build
from paged_attention_decode_split_gb300.inputs import make_new_tokens, make_problem
from tests.gpu_common import REL_L2_VERIFY, assert_parity, oracle_out, run_attention, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    pa.load_library()


def hybrid(seed, lens, bs, **kw):
    args = dict(num_seqs=len(lens), seq_lens=list(lens), num_q_heads=24, num_kv_heads=4, head_dim=256,
                block_size=bs, scale=1 / 16, poison_unused=True)
    args.update(kw)
    return make_problem(seed, **args)


def write_new_rows(prob, seed):
    k_new, v_new = make_new_tokens(seed, prob.num_seqs * prob.q_len, prob.num_kv_heads, prob.head_dim)
    kc, vc = prob.k_cache[0].cuda(), prob.v_cache[0].cuda()
    pa.reshape_and_cache(k_new.cuda(), v_new.cuda(), kc, vc, prob.new_token_slots().cuda())
    torch.cuda.synchronize()
    prob.k_cache[0], prob.v_cache[0] = kc.cpu(), vc.cpu()


@pytest.mark.parametrize("window", [2048, 1000, 17, 1])
@pytest.mark.parametrize("bs", [784, 16])
def test_decode_window(oracle_mod, window, bs):
    prob = hybrid(401 + window + bs, [5000, 2049, 1000, 100, 1, 0], bs)
    out, status, plan = run_attention(prob, window=window)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=window), what=f"decode window={window} bs={bs}")


@pytest.mark.parametrize("splits", [1, 3, 13])
def test_decode_window_forced_splits(oracle_mod, splits):
    prob = hybrid(411 + splits, [4000, 333], 784)
    out, status, _ = run_attention(prob, window=700, num_splits=splits)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=700), what=f"decode window splits={splits}")


def test_decode_window_dense_d128(oracle_mod):
    import math
    prob = make_problem(421, num_seqs=2, seq_lens=[3000, 64], num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, scale=1 / math.sqrt(128), poison_unused=True)
    out, status, _ = run_attention(prob, window=500)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=500), what="decode window d128")


@pytest.mark.parametrize("hd", [256, 128])
def test_decode_window_g12(oracle_mod, hd):
    import math
    prob = hybrid(425 + hd, [3000, 700, 5], 784, num_q_heads=48, num_kv_heads=4, head_dim=hd,
                  scale=1 / math.sqrt(hd))
    out, status, _ = run_attention(prob, window=1000)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=1000), what=f"decode window G=12 d{hd}")


@pytest.mark.parametrize("q_len,lens,window", [(16, [3000, 500, 16], 1024), (16, [900], 40), (200, [1500], 300)])
def test_verify_window(oracle_mod, q_len, lens, window):
    prob = hybrid(431 + window, lens, 832, q_len=q_len)
    write_new_rows(prob, 21)
    out, status, _ = run_attention(prob, window=window)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=window), rel_l2=REL_L2_VERIFY,
                  what=f"verify window={window} q_len={q_len}")


def test_window_early_kv_bitwise():
    prob = hybrid(441, [5000, 300], 784)
    t = to_dev(prob)
    ref, _, _ = run_attention(prob, tensors=t, window=2048)
    got, _, _ = run_attention(prob, tensors=t, window=2048, flags=pa.PA_FLAG_EARLY_KV_READ)
    assert torch.equal(got, ref)
