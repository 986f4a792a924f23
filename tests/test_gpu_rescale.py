"""GPU parity on inputs that make the online softmax raise its running max
in the middle of a split.

With N(0, 1) data the logits have sigma ~ 1, and the first chunks of a split
nearly always hold a max that later chunks never beat by the kernels' lazy
threshold of 2^8.  These problems give every query row a logit ramp on top of
the noise: q[..., 0] = a and K[t, :, 0] = ramp(t) / (a * scale), so the
logit of key t is ramp(t) plus noise.  Patterns:
  saw    a rising sawtooth of period 1024 and height 12 nats: splits that
         start low raise their max by more than 8 log2 units part-way;
  rise   a steady rise of 48 nats over the sequence: every split's max is far
         above the one before it, so the reduce raises its running max at
         every split;
  spike  one key 30 nats above the rest, inside a split: the output is that
         key's V, and the chunk holding it rescales everything before it;
  step   a block of 200 keys 20 nats up in the middle of the sequence.
Each test first checks on the oracle side that its input does raise the
running max mid-split (the max over a split's keys exceeds the max over the
split's first 256 keys by more than 8 ln 2; every chunk stream of a decode
CTA, and the first tile of a verify split, starts inside those 256 keys),
then compares the GPU output element by element with the oracle.
"""
import math

import numpy as np
import pytest
import torch

import paged_attention_decode_split_gb300 as pa
from paged_attention_decode_split_gb300 import _build
from paged_attention_decode_split_gb300.inputs import make_new_tokens, make_problem
from tests.gpu_common import REL_L2_VERIFY, assert_cache_written, assert_parity, oracle_out, run_attention
from tests.helpers import bits

pytestmark = pytest.mark.gpu

LAZY_NATS = 8 * math.log(2)  # the kernels' lazy threshold, 2^8, in natural-log units


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    pa.load_library()


def ramp(pattern: str, L: int) -> np.ndarray:
    t = np.arange(L, dtype=np.float64)
    if pattern == "saw":
        return 12.0 * (t % 1024) / 1024
    if pattern == "rise":
        return 48.0 * t / max(1, L - 1)
    if pattern == "spike":
        r = np.zeros(L)
        r[(2 * L) // 3] = 30.0
        return r
    if pattern == "step":
        r = np.zeros(L)
        r[L // 2:L // 2 + 200] = 20.0
        return r
    raise ValueError(pattern)


def ramp_problem(seed, lens, bs, pattern, *, G=6, hkv=4, D=256, q_len=1, fp8=False):
    """A problem whose logits follow ramp(t) per sequence (plus noise).  Row r
    of a verify block gets q[..., 0] scaled by (1 + r / 8), so its ramp is
    steeper than the row before it."""
    scale = 1 / math.sqrt(D)
    prob = make_problem(seed, num_seqs=len(lens), seq_lens=list(lens), num_q_heads=G * hkv, num_kv_heads=hkv,
                        head_dim=D, block_size=bs, q_len=q_len, scale=scale, kv_fp8=fp8, poison_unused=True)
    a = 64.0 if fp8 else 16.0  # keeps the fp8 codes of the ramp below 448
    q = prob.q[0].float()
    q[:, :, 0] = (a * (1 + torch.arange(q_len, dtype=torch.float32) / 8)).repeat(len(lens))[:, None]
    prob.q[0] = q.to(torch.bfloat16)
    kc = prob.k_cache[0]
    if not fp8:
        kc = (kc.float() * 0.5).to(torch.bfloat16)  # exact: halves the noise logits
    for b, L in enumerate(lens):
        t = torch.arange(L)
        pages = prob.block_table[b, (t // bs)].long()
        offs = t % bs
        f = torch.from_numpy(ramp(pattern, L) / (a * scale)).float()
        if fp8:
            x = (f[:, None] / prob.k_scale[0][None, :]).clamp(-448, 448)  # the cast would give NaN beyond
            codes = x.to(torch.float8_e4m3fn).view(torch.uint8)
            kc[pages, offs, :, 0] = codes
        else:
            kc[pages, offs, :, 0] = f.to(torch.bfloat16)[:, None].expand(L, hkv)
    prob.k_cache[0] = kc
    return prob


def bf16_view(oracle_mod, prob):
    """(k_cache, v_cache) as bf16 bit patterns; for an fp8 cache the decoded
    values times the head scale, which are exact in bf16 (at most 7
    significant bits) -- used only to find where the running max rises."""
    if not prob.kv_fp8:
        return bits(prob.k_cache[0]), bits(prob.v_cache[0])
    out = []
    for c, s in ((prob.k_cache[0], prob.k_scale[0]), (prob.v_cache[0], prob.v_scale[0])):
        x = oracle_mod.e4m3_decode(c) * s.double().numpy()[None, None, :, None]
        out.append(bits(torch.from_numpy(x).to(torch.bfloat16)))
    return tuple(out)


def split_raises(oracle_mod, prob, plan, seq=0, row=None, head=0, head_tokens=256):
    """Number of splits of `seq` whose max logit exceeds the max over their
    first `head_tokens` keys by more than the lazy threshold (oracle partials)."""
    kc, vc = bf16_view(oracle_mod, prob)
    q = bits(prob.q[0])
    L = int(prob.seq_lens[seq])
    row = seq * prob.q_len if row is None else row
    limit = L - prob.q_len + (row - seq * prob.q_len) + 1  # keys the row sees
    span = plan["chunks_per_split"] * 16
    bt, sl = prob.block_table.numpy(), prob.seq_lens.numpy()
    n = 0
    for t0 in range(0, limit, span):
        t1 = min(limit, t0 + span)
        if t1 - t0 <= head_tokens:
            continue
        _, m_all, _ = oracle_mod.attention_partial(q, kc, vc, bt, sl, prob.scale, row, head, t0, t1,
                                                   q_len=prob.q_len)
        _, m_first, _ = oracle_mod.attention_partial(q, kc, vc, bt, sl, prob.scale, row, head, t0,
                                                     t0 + head_tokens, q_len=prob.q_len)
        n += (m_all - m_first) > LAZY_NATS
    return n


# -- decode ---------------------------------------------------------------------

@pytest.mark.parametrize("pattern", ["saw", "rise", "spike", "step"])
@pytest.mark.parametrize("fp8", [False, True])
def test_decode_rescale_patterns_g6_d256(oracle_mod, pattern, fp8):
    prob = ramp_problem(301, [6000, 2500], 784, pattern, fp8=fp8)
    out, status, plan = run_attention(prob, num_splits=5)
    assert status == 0 and plan["num_splits"] == 5
    assert split_raises(oracle_mod, prob, plan) >= 1
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"{pattern} fp8={fp8}")


@pytest.mark.parametrize("G,D,fp8", [(12, 256, False), (12, 256, True), (6, 128, False), (6, 128, True),
                                     (16, 128, False), (1, 256, False)])
@pytest.mark.parametrize("pattern", ["saw", "rise"])
def test_decode_rescale_shapes(oracle_mod, G, D, fp8, pattern):
    prob = ramp_problem(311 + G + D, [5000, 1100], 16 if D == 128 else 832, pattern, G=G, D=D, fp8=fp8,
                        hkv=2 if G == 16 else 4)
    out, status, plan = run_attention(prob, num_splits=3)
    assert status == 0 and plan["num_splits"] == 3
    assert split_raises(oracle_mod, prob, plan) >= 1
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"G={G} D={D} fp8={fp8} {pattern}")


@pytest.mark.parametrize("splits", [1, 2, 7, 40, 120])
def test_decode_rescale_forced_splits(oracle_mod, splits):
    """The sawtooth under split counts from one (the whole context in one CTA)
    to more than 64 (the reduce loads its splits in several rounds, and its
    own running max rises from split to split)."""
    prob = ramp_problem(321 + splits, [9000], 784, "saw")
    out, status, plan = run_attention(prob, num_splits=splits)
    assert status == 0
    if plan["chunks_per_split"] * 16 >= 1024:  # long enough splits for a rise within one
        assert split_raises(oracle_mod, prob, plan) >= 1
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"saw splits={splits}")


@pytest.mark.parametrize("pattern", ["saw", "rise"])
@pytest.mark.parametrize("fp8", [False, True])
def test_decode_rescale_window(oracle_mod, pattern, fp8):
    prob = ramp_problem(331, [7000, 3000], 784, pattern, fp8=fp8)
    out, status, plan = run_attention(prob, window=2048)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=2048), what=f"window {pattern} fp8={fp8}")


def test_decode_rescale_full_context_workload_shape(oracle_mod):
    """The 32K hybrid layer shape in its automatic plan with the sawtooth."""
    prob = ramp_problem(341, [32768], 784, "saw")
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["num_splits"] > 1
    assert split_raises(oracle_mod, prob, plan) >= 1
    assert_parity(out, oracle_out(oracle_mod, prob), what="saw 32K")


# -- verify ----------------------------------------------------------------------

def write_ramp_rows(oracle_mod, prob, seed):
    """reshape_and_cache of the new rows, with the written cache checked bit
    for bit against the oracle's scatter before anything reads it.  The new
    rows keep the ramp: their dim 0 is copied from the cache they replace."""
    n = prob.num_seqs * prob.q_len
    k_new, v_new = make_new_tokens(seed, n, prob.num_kv_heads, prob.head_dim)
    slots = prob.new_token_slots()
    kc_old = prob.k_cache[0]
    for i, s in enumerate(slots.tolist()):
        k_new[i, :, 0] = kc_old[s // prob.block_size, s % prob.block_size, :, 0]
    kc, vc = prob.k_cache[0].cuda(), prob.v_cache[0].cuda()
    pa.reshape_and_cache(k_new.cuda(), v_new.cuda(), kc, vc, slots.cuda())
    torch.cuda.synchronize()
    assert_cache_written(oracle_mod, prob.k_cache[0], prob.v_cache[0], k_new, v_new, slots, kc, vc)
    prob.k_cache[0], prob.v_cache[0] = kc.cpu(), vc.cpu()


@pytest.mark.parametrize("pattern", ["saw", "rise", "spike"])
@pytest.mark.parametrize("splits", [1, 3])
def test_verify_rescale_rows_differ(oracle_mod, pattern, splits):
    """16 verify rows whose ramps have different slopes (and causal limits),
    the context in one split or in three."""
    prob = ramp_problem(351, [3000, 1700], 832, pattern, q_len=16)
    write_ramp_rows(oracle_mod, prob, 7)
    out, status, plan = run_attention(prob, num_splits=splits)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05 and plan["num_splits"] == splits
    assert split_raises(oracle_mod, prob, plan, row=15) >= 1
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what=f"verify {pattern} splits={splits}")


def test_verify_rescale_window(oracle_mod):
    prob = ramp_problem(361, [4000], 784, "saw", q_len=16)
    write_ramp_rows(oracle_mod, prob, 9)
    out, status, plan = run_attention(prob, window=2048)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=2048), rel_l2=REL_L2_VERIFY, what="verify window saw")


@pytest.mark.parametrize("pattern", ["saw", "rise", "spike", "step"])
@pytest.mark.parametrize("splits", [1, 3])
def test_verify_rescale_row_blocks(oracle_mod, pattern, splits):
    """24 rows x 6 heads = 144 rows per KV head: two row blocks, the shape
    that runs 128-key score tiles, where a tile's max is taken over both of
    its 64-key halves before any of its P is written.  (With 48 rows the
    steepest ramps reach a rel-L2 of 1.35e-4 from the fp32 scores alone, the
    same with 64-key tiles.)"""
    prob = ramp_problem(381, [3000, 1700], 832, pattern, q_len=24)
    write_ramp_rows(oracle_mod, prob, 11)
    out, status, plan = run_attention(prob, num_splits=splits)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05 and plan["num_splits"] == splits
    assert split_raises(oracle_mod, prob, plan, row=23) >= 1
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY,
                  what=f"verify row blocks {pattern} splits={splits}")


def test_verify_rescale_row_blocks_window(oracle_mod):
    prob = ramp_problem(391, [4000], 784, "saw", q_len=24)
    write_ramp_rows(oracle_mod, prob, 13)
    out, status, plan = run_attention(prob, window=2048)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=2048), rel_l2=REL_L2_VERIFY,
                  what="verify row blocks window saw")


def test_verify_rescale_fp8(oracle_mod):
    """The fp8 verify over the sawtooth (the cache is built directly; no new
    rows are written)."""
    prob = ramp_problem(371, [3000, 900], 832, "saw", q_len=16, fp8=True)
    out, status, plan = run_attention(prob, num_splits=3)
    assert status == 0 and plan["num_splits"] == 3
    assert split_raises(oracle_mod, prob, plan, row=15) >= 1
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what="verify fp8 saw")
