"""GPU parity of the fp8 e4m3 KV cache: the quantising reshape_and_cache must
give the oracle's codes bit for bit, and decode over the codes must match the
oracle's attention over the decoded values (K = code x k_scale[kv head], V
likewise) within the bf16-path tolerance.  Edge cases: ties and saturation in
the quantiser, NaN-poisoned unused slots, ragged tails, forced splits, every
compiled group size, a sliding window, bf16 output, the early-K/V flag and the
chain reshape_and_cache -> decode on one stream."""
import ctypes
import math

import numpy as np
import pytest
import torch

import paged_attention_decode_split_gb300 as pa
from paged_attention_decode_split_gb300 import _build
from paged_attention_decode_split_gb300.inputs import WORKLOADS, make_new_tokens, make_problem
from tests.gpu_common import (REL_L2_DECODE, REL_L2_VERIFY, assert_parity, desc_for, oracle_out, run_attention,
                              scales_dev, to_dev)
from tests.helpers import bits

pytestmark = pytest.mark.gpu

TAIL_LENGTHS = [1, 15, 16, 17, 63, 64, 65, 783, 784, 785, 831, 832, 833]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    pa.load_library()


def hybrid(seed, lens, bs, **kw):
    args = dict(num_seqs=len(lens), seq_lens=list(lens), num_q_heads=24, num_kv_heads=4, head_dim=256,
                block_size=bs, scale=1 / 16, kv_fp8=True)
    args.update(kw)
    return make_problem(seed, **args)


# -- quantising reshape_and_cache -------------------------------------------------------

def _reshape_fp8_both(oracle_mod, k_new, v_new, ks, vs, slots, P, bs):
    hkv, d = k_new.shape[1], k_new.shape[2]
    kc = torch.full((P, bs, hkv, d), 0x33, dtype=torch.uint8)
    vc = torch.full((P, bs, hkv, d), 0x44, dtype=torch.uint8)
    kc_d, vc_d = kc.cuda(), vc.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.reshape_and_cache_fp8(k_new.cuda(), v_new.cuda(), kc_d, vc_d, slots.cuda(), ks.cuda(), vs.cuda(), status)
    torch.cuda.synchronize()
    k_ref, v_ref = kc.numpy().copy(), vc.numpy().copy()
    oracle_mod.reshape_and_cache_fp8(bits(k_new), bits(v_new), k_ref, v_ref, slots.numpy(), ks.numpy(), vs.numpy())
    return kc_d.cpu().numpy(), vc_d.cpu().numpy(), k_ref, v_ref, int(status.item())


@pytest.mark.parametrize("hkv,d", [(4, 256), (8, 128), (1, 8)])
def test_reshape_and_cache_fp8_bit_exact(oracle_mod, hkv, d):
    P, bs, n = 7, 16, 40
    k_new, v_new = make_new_tokens(31 + d, n, hkv, d)
    k_new = k_new * 3  # spread over more binades
    g = torch.Generator().manual_seed(d)
    slots = torch.randperm(P * bs, generator=g)[:n].to(torch.int64)
    slots[5] = -1
    ks = torch.tensor([0.013 * (1 + h) for h in range(hkv)], dtype=torch.float32)
    vs = torch.tensor([0.05 / (1 + h) for h in range(hkv)], dtype=torch.float32)
    kg, vg, kr, vr, st = _reshape_fp8_both(oracle_mod, k_new, v_new, ks, vs, slots, P, bs)
    assert st == 0
    assert np.array_equal(kg, kr) and np.array_equal(vg, vr)


def test_reshape_and_cache_fp8_ties_saturation_and_subnormals(oracle_mod):
    """Values at e4m3 rounding midpoints (scale 1: the division is exact), past
    448 and +-inf, subnormal and underflowing ones: nearest-even and
    saturation agree with the oracle bit for bit."""
    vals = oracle_mod.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    pos = sorted(set(vals.tolist()))
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]  # need 4 mantissa bits: exact in bf16
    special = [448.0, 450.0, 464.0, 480.0, 8192.0, float("inf"), 2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11, 0.0]
    row = torch.tensor(mids + special + [-x for x in mids + special], dtype=torch.float64)
    d = 8
    n = math.ceil(row.numel() / d)
    row = torch.cat([row, torch.zeros(n * d - row.numel(), dtype=torch.float64)])
    assert torch.equal(row.to(torch.bfloat16).double(), row)  # every value is exact in bf16
    k_new = row.to(torch.bfloat16).view(n, 1, d)
    v_new = (-row).to(torch.bfloat16).view(n, 1, d)
    one = torch.ones(1, dtype=torch.float32)
    slots = torch.arange(n, dtype=torch.int64)
    kg, vg, kr, vr, st = _reshape_fp8_both(oracle_mod, k_new, v_new, one, one, slots, math.ceil(n / 16), 16)
    assert st == 0
    assert np.array_equal(kg, kr) and np.array_equal(vg, vr)


def test_reshape_and_cache_fp8_bad_slot_flagged(oracle_mod):
    """A slot past the pool sets PA_DEV_BAD_SLOT and writes nothing; the other
    tokens land as the oracle puts them (it skips the bad token here)."""
    k_new, v_new = make_new_tokens(5, 3, 2, 16)
    one = torch.ones(2, dtype=torch.float32)
    kc = torch.zeros((2, 16, 2, 16), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.tensor([0, 999, 3], dtype=torch.int64)
    pa.reshape_and_cache_fp8(k_new.cuda(), v_new.cuda(), kc, vc, slots.cuda(), one.cuda(), one.cuda(), status)
    torch.cuda.synchronize()
    assert status.item() & pa.PA_DEV_BAD_SLOT
    k_ref = np.zeros((2, 16, 2, 16), np.uint8)
    v_ref = np.zeros_like(k_ref)
    oracle_mod.reshape_and_cache_fp8(bits(k_new), bits(v_new), k_ref, v_ref, np.array([0, -1, 3], np.int64),
                                     one.numpy(), one.numpy())
    assert np.array_equal(kc.cpu().numpy(), k_ref) and np.array_equal(vc.cpu().numpy(), v_ref)


# -- decode over the fp8 cache ---------------------------------------------------------

@pytest.mark.parametrize("bs", [16, 784, 832])
def test_decode_fp8_ragged_tails_nan_poisoned(oracle_mod, bs):
    prob = hybrid(501 + bs, TAIL_LENGTHS, bs, poison_unused=True)
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_DECODE_MMA
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"fp8 tails bs={bs}")


@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_decode_fp8_forced_splits(oracle_mod, splits):
    prob = hybrid(511, [5000, 333, 1], 784, poison_unused=True)
    out, status, _ = run_attention(prob, num_splits=splits)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"fp8 splits={splits}")


@pytest.mark.parametrize("G,hkv", [(1, 4), (2, 4), (3, 4), (4, 2), (5, 4), (6, 4), (8, 4), (12, 4), (16, 2)])
def test_decode_fp8_group_sizes_d256(oracle_mod, G, hkv):
    prob = hybrid(521 + G, [700, 1500, 9], 16, num_q_heads=G * hkv, num_kv_heads=hkv)
    out, status, _ = run_attention(prob)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"fp8 G={G}")


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 8, 12, 16])
def test_decode_fp8_dense_d128(oracle_mod, G):
    prob = make_problem(531 + G, num_seqs=3, seq_lens=[1, 100, 2049], num_q_heads=8 * G, num_kv_heads=8,
                        head_dim=128, block_size=16, scale=1 / math.sqrt(128), poison_unused=True, kv_fp8=True)
    out, status, _ = run_attention(prob)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"fp8 dense G={G}")


@pytest.mark.parametrize("window", [2048, 17])
def test_decode_fp8_window(oracle_mod, window):
    prob = hybrid(541 + window, [5000, 2049, 100, 0], 784, poison_unused=True)
    out, status, _ = run_attention(prob, window=window)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=window), what=f"fp8 window={window}")


def test_decode_fp8_bf16_output(oracle_mod):
    prob = hybrid(551, [3000, 17], 832)
    out, status, _ = run_attention(prob, out_dtype=pa.PA_OUT_BF16)
    ref = oracle_out(oracle_mod, prob)
    ref_bf16 = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    err = np.abs(out.double().numpy() - ref_bf16)
    assert status == 0 and np.isfinite(out.numpy()).all()
    assert err.max() <= 2e-3 + 2 * 2.0 ** -8 * np.abs(ref).max()


@pytest.mark.parametrize("hq", [24, 16])  # 6 heads per KV head: one producer lane; 4: a lane per stream
def test_decode_fp8_early_kv_bitwise(hq):
    prob = hybrid(561, [1, 15, 17, 785, 5000, 0], 784, poison_unused=True, num_q_heads=hq)
    outs = []
    for flags in (0, pa.PA_FLAG_EARLY_KV_READ):
        out, status, _ = run_attention(prob, num_splits=5, flags=flags)
        assert status == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


def test_decode_fp8_after_quantising_reshape_on_one_stream(oracle_mod):
    """The serving order: the new token's K/V quantised into the fp8 cache,
    then decode, on one stream without a host sync; the decode must see the
    new codes (oracle run on the cache as the GPU left it, checked bit-exact
    against the oracle's own quantisation first)."""
    prob = hybrid(571, [32768, 900, 17], 784)
    k_new, v_new = make_new_tokens(17, prob.num_seqs, prob.num_kv_heads, prob.head_dim)
    q, kc, vc, bt, sl = to_dev(prob)
    ks, vs = scales_dev(prob)
    slots = prob.new_token_slots()
    k_ref, v_ref = prob.k_cache[0].numpy().copy(), prob.v_cache[0].numpy().copy()
    oracle_mod.reshape_and_cache_fp8(bits(k_new), bits(v_new), k_ref, v_ref, slots.numpy(),
                                     prob.k_scale[0].numpy(), prob.v_scale[0].numpy())
    desc = desc_for(prob)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device="cuda")
    out = torch.full((prob.num_seqs, prob.num_q_heads, prob.head_dim), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kn, vn, sd = k_new.cuda(), v_new.cuda(), slots.cuda()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(2_000_000)
        pa.reshape_and_cache_fp8(kn, vn, kc, vc, sd, ks, vs, status)
        pa.paged_attention_decode_fp8(q, kc, vc, ks, vs, bt, sl, desc, out, ws, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.array_equal(kc.cpu().numpy(), k_ref) and np.array_equal(vc.cpu().numpy(), v_ref)
    prob.k_cache[0], prob.v_cache[0] = torch.from_numpy(k_ref), torch.from_numpy(v_ref)
    assert_parity(out.cpu(), oracle_out(oracle_mod, prob), what="fp8 decode after reshape")


def test_decode_fp8_l32768_bs784_workload(oracle_mod):
    """The benchmarked fp8 layer (one of its 16 layers) in the benchmark's launch."""
    prob = make_problem(1009, **dict(WORKLOADS["decode_fp8_l32768_bs784"], num_layers=1))
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["num_splits"] > 1
    assert_parity(out, oracle_out(oracle_mod, prob), what="fp8 32K layer")


def test_decode_fp8_rejects_missing_scales():
    prob = hybrid(581, [100], 16)
    q, kc, vc, bt, sl = to_dev(prob)
    desc = desc_for(prob)
    out = torch.empty((1, 24, 256), device="cuda")
    with pytest.raises(ValueError, match="k_scale, v_scale"):  # the binding refuses before the call
        pa.paged_attention_decode_fp8(q, kc, vc, None, None, bt, sl, desc, out)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device="cuda")
    rc = pa.load_library().pa_paged_attention_decode_fp8(  # and so does the C entry point
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), None, None, bt.data_ptr(), sl.data_ptr(), ctypes.byref(desc),
        out.data_ptr(), ws.data_ptr(), ws.numel(), None, torch.cuda.current_stream().cuda_stream)
    assert rc == pa.PA_ERR_INVALID_ARG


# -- verify over the fp8 cache (tcgen05, f16 products) --------------------------------

@pytest.mark.parametrize("q_len,lens,bs", [(2, [2, 33, 900], 16), (5, [5, 64, 785], 784),
                                           (16, [16, 17, 831, 1700], 832), (16, [3000], 16)])
def test_verify_fp8_small(oracle_mod, q_len, lens, bs):
    prob = hybrid(601 + q_len, lens, bs, q_len=q_len, poison_unused=True)
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what=f"fp8 verify q_len={q_len}")


@pytest.mark.parametrize("splits", [2, 5, 13])
def test_verify_fp8_forced_splits(oracle_mod, splits):
    prob = hybrid(611 + splits, [1700, 900, 37], 784, q_len=16, poison_unused=True)
    out, status, plan = run_attention(prob, num_splits=splits)
    assert status == 0 and plan["num_splits"] > 1
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what=f"fp8 verify splits={splits}")


@pytest.mark.parametrize("q_len,lens,window", [(48, [1000, 48], 0), (200, [1500], 300), (16, [3000, 500], 1024)])
def test_verify_fp8_row_blocks_and_window(oracle_mod, q_len, lens, window):
    prob = hybrid(621 + q_len, lens, 784, q_len=q_len, poison_unused=True)
    out, status, _ = run_attention(prob, window=window)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=window), rel_l2=REL_L2_VERIFY,
                  what=f"fp8 verify q_len={q_len} W={window}")


@pytest.mark.parametrize("splits", [1, 3])
def test_verify_fp8_dense_d128(oracle_mod, splits):
    prob = make_problem(631, num_seqs=2, seq_lens=[300, 77], num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, q_len=8, scale=1 / math.sqrt(128), poison_unused=True, kv_fp8=True)
    out, status, _ = run_attention(prob, num_splits=splits)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what="fp8 verify d128")


def test_verify_fp8_early_kv_bitwise():
    prob = hybrid(641, [16, 17, 831, 1700], 832, q_len=16, poison_unused=True)
    outs = []
    for flags in (0, pa.PA_FLAG_EARLY_KV_READ):
        out, status, _ = run_attention(prob, flags=flags)
        assert status == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


def test_verify_fp8_b8_q16_l8192_bs832_workload(oracle_mod):
    prob = make_problem(1010, **dict(WORKLOADS["verify_b8_q16_l8192_bs832"], kv_fp8=True))
    out, status, _ = run_attention(prob)
    assert status == 0
    rows = [0, 3, 7]
    sel = torch.cat([torch.arange(b * 16, (b + 1) * 16) for b in rows])
    assert torch.isfinite(out).all()
    assert_parity(out[sel], oracle_out(oracle_mod, prob, rows=rows), rel_l2=REL_L2_VERIFY,
                  what="fp8 verify workload (sampled)")


def test_verify_fp8_wide_group_g12(oracle_mod):
    prob = hybrid(651, [5, 900, 2000], 784, q_len=5, num_q_heads=48, num_kv_heads=4, poison_unused=True)
    out, status, _ = run_attention(prob)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what="fp8 verify G=12")


# -- the range of q over an fp8 cache ---------------------------------------------------
# Over an fp8 cache the products run in f16, whose range (about 6e-8 .. 65504)
# is far narrower than bf16's.  Each q row (verify) or head (decode) enters f16
# scaled by a power of two that puts its largest element in [2^14, 2^15), so
# any finite bf16 q keeps its bits.  These problems give the query heads
# magnitudes from 1e-6 to 1e5: logits from ~1e-5 (a near-uniform softmax) to
# ~1e5 nats (a one-hot one).
#
# At 1e5 nats the fp32 logits themselves carry rounding errors of a fraction
# of a nat, so a row whose top keys tie to within that error has an output
# that any fp32 kernel gets only to within the softmax's sensitivity.  The
# tolerance is therefore derived per (row, head) from the inputs:
#   dx    = 2^-19 * max_t scale log2(e) sum_d |q_d K_td|   (the products are
#           exact; the tensor core rounds each 16-dim step's sum into the fp32
#           accumulator, D / 16 <= 16 roundings of at most 2 ulps each
#           (truncation allowed): below 2^-19 of the sum of the products'
#           magnitudes, in log2 units)
#   extra = 2 ln 2 * dx * sum_t p_t |V_t - o|_inf           (first-order change
#           of o = sum_t p_t V_t when every logit moves by up to dx)
# and every element must satisfy |gpu - oracle| <= 2e-3 + extra.  Rows with
# extra < 1e-6 -- the near-uniform rows of the small magnitudes and the
# one-hot rows of the large ones, all but the near-ties -- must also pass the
# full gate, relative L2 included.

Q_MAGNITUDES = [1e-6, 1e-4, 1e-2, 1.0, 30.0, 1e3, 2e4, 1e5]


def scale_q_heads(prob):
    hq = prob.num_q_heads
    mags = torch.tensor([Q_MAGNITUDES[h % len(Q_MAGNITUDES)] for h in range(hq)], dtype=torch.float32)
    prob.q[0] = (prob.q[0].float() * mags[None, :, None]).to(torch.bfloat16)
    assert torch.isfinite(prob.q[0].float()).all()
    return prob


def q_range_problem(seed, lens, bs, q_len=1, fp8=True):
    prob = hybrid(seed, lens, bs, q_len=q_len, num_q_heads=24, poison_unused=True, kv_fp8=fp8)
    return scale_q_heads(prob)


def rounding_sensitivity(prob):
    """extra[row, head] of the derivation above, from the inputs in float64
    (torch decodes the e4m3 codes exactly)."""
    def values(c, s):
        if prob.kv_fp8:
            return c.view(torch.float8_e4m3fn).double() * s.double()[None, None, :, None]
        return c.double()
    kc = values(prob.k_cache[0], prob.k_scale[0] if prob.kv_fp8 else None)
    vc = values(prob.v_cache[0], prob.v_scale[0] if prob.kv_fp8 else None)
    G = prob.num_q_heads // prob.num_kv_heads
    extra = np.zeros((prob.num_seqs * prob.q_len, prob.num_q_heads))
    for b in range(prob.num_seqs):
        L = int(prob.seq_lens[b])
        t = torch.arange(L)
        pages = prob.block_table[b, t // prob.block_size].long()
        K, V = kc[pages, t % prob.block_size], vc[pages, t % prob.block_size]  # [L, Hkv, D]
        for r in range(prob.q_len):
            n = L - prob.q_len + r + 1
            if n <= 0:
                continue
            q = prob.q[0][b * prob.q_len + r].double()  # [Hq, D]
            for h in range(prob.num_q_heads):
                Kh, Vh = K[:n, h // G], V[:n, h // G]
                s = prob.scale * (Kh @ q[h])
                dx = 2.0 ** -19 * (prob.scale * math.log2(math.e) * (Kh.abs() @ q[h].abs())).max()
                p = torch.softmax(s, 0)
                o = p @ Vh
                spread = (p * (Vh - o).abs().max(dim=1).values).sum()
                extra[b * prob.q_len + r, h] = float(2 * math.log(2) * dx * spread)
    return extra


def assert_q_range_parity(out, ref, extra, rel_l2, what):
    g = out.double().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref).max(axis=2)  # [rows, heads]
    assert (err <= 2e-3 + extra).all(), f"{what}: max excess {(err - 2e-3 - extra).max():.3g}"
    ok = extra < 1e-6
    assert ok.mean() > 0.4, f"{what}: too few well-conditioned rows ({ok.mean():.2f})"
    assert_parity(out[torch.from_numpy(ok)][:, None, :], ref[ok][:, None, :], rel_l2=rel_l2,
                  what=f"{what} (well-conditioned rows)")


@pytest.mark.parametrize("splits", [0, 1, 3])
def test_decode_fp8_q_range(oracle_mod, splits):
    prob = q_range_problem(581, [3000, 77], 784)
    out, status, _ = run_attention(prob, num_splits=splits)
    assert status == 0
    assert_q_range_parity(out, oracle_out(oracle_mod, prob), rounding_sensitivity(prob), REL_L2_DECODE,
                          f"fp8 decode q from 1e-6 to 1e5, splits={splits}")


@pytest.mark.parametrize("D", [256, 128])
def test_verify_fp8_q_range(oracle_mod, D):
    if D == 256:
        prob = q_range_problem(591, [2000, 40], 832, q_len=16)
    else:
        prob = scale_q_heads(make_problem(592, num_seqs=2, seq_lens=[2000, 40], num_q_heads=32, num_kv_heads=8,
                                          head_dim=128, block_size=16, q_len=16, scale=1 / math.sqrt(128),
                                          kv_fp8=True, poison_unused=True))
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05
    assert_q_range_parity(out, oracle_out(oracle_mod, prob), rounding_sensitivity(prob), REL_L2_VERIFY,
                          f"fp8 verify q range D={D}")


def test_decode_bf16_q_range(oracle_mod):
    """The same magnitudes over a bf16 cache (bf16 products, no pre-scale)."""
    prob = q_range_problem(601, [3000, 77], 784, fp8=False)
    out, status, _ = run_attention(prob, num_splits=3)
    assert status == 0
    assert_q_range_parity(out, oracle_out(oracle_mod, prob), rounding_sensitivity(prob), REL_L2_DECODE,
                          "bf16 decode q from 1e-6 to 1e5")
