"""Pins of the CPU oracle against facts fixed outside it.

Each test below would fail for a plausible mistake in the oracle: a dropped
scale, a wrong sign, a wrong page/offset split, a wrong GQA head mapping, an
off-by-one in the causal rule, a missing max-subtraction, a wrong split merge.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from tests.helpers import bits, dense_attention, place_in_pages, randn_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run(oracle_mod, q, k_cache, v_cache, bt, seq_lens, scale, q_len=1, threads=4, window=0):
    return oracle_mod.paged_attention(bits(q), bits(k_cache), bits(v_cache), bt.numpy(),
                                      np.asarray(seq_lens, dtype=np.int32), scale, q_len=q_len,
                                      num_threads=threads, window=window)


def _contig(gen, lens, hkv, d):
    ks = [randn_bf16((L, hkv, d), gen) for L in lens]
    vs = [randn_bf16((L, hkv, d), gen) for L in lens]
    return ks, vs


# -- golden fixtures -----------------------------------------------------------

def test_closed_form_golden(oracle_mod):
    """Hand-derivable softmax attention values (tests/golden/closed_form_attention.json)."""
    spec = json.load(open(os.path.join(GOLDEN, "closed_form_attention.json")))
    for case in spec["cases"]:
        d = case["head_dim"]
        k = torch.tensor(case["k"], dtype=torch.bfloat16).reshape(-1, 1, d)
        v = torch.tensor(case["v"], dtype=torch.bfloat16).reshape(-1, 1, d)
        q = torch.tensor(case["q"], dtype=torch.bfloat16).reshape(-1, 1, d)
        L = k.shape[0]
        kc, vc, bt = place_in_pages([k], [v], 16, 3, seed=5)
        out = _run(oracle_mod, q, kc, vc, bt, [L], case["scale"], q_len=case["q_len"])
        np.testing.assert_allclose(out[:, 0, :], np.array(case["expected"]), rtol=0, atol=1e-14,
                                   err_msg=case["name"])


def test_page_address_golden(oracle_mod):
    """The oracle reads token t at (block_table[t // BS], t % BS): a single
    marked slot is found exactly where the page's formula puts it."""
    spec = json.load(open(os.path.join(GOLDEN, "page_address.json")))
    for tiling in spec["page_tiling"]:
        bs = tiling["block_size"]
        assert bs == 64 * tiling["full_64_tiles"] + tiling["tail_tokens"]
    d, hkv = 8, 1
    for ex in spec["examples"]:
        bs, t = ex["block_size"], ex["token"]
        L = t + 1
        pages = math.ceil(L / bs)
        num_pages = pages + 2
        g = torch.Generator().manual_seed(bs * 7 + t)
        perm = torch.randperm(num_pages, generator=g)
        bt = perm[:pages].to(torch.int32).reshape(1, -1)
        kc = torch.zeros((num_pages, bs, hkv, d), dtype=torch.bfloat16)
        vc = torch.zeros_like(kc)
        phys = int(bt[0, ex["logical_page"]])
        vc[phys, ex["page_offset"], 0, :] = 1.0  # the mean over L tokens is then 1 / L
        q = torch.zeros((1, 1, d), dtype=torch.bfloat16)
        out = _run(oracle_mod, q, kc, vc, bt, [L], scale=0.0)
        np.testing.assert_allclose(out[0, 0], np.full(d, 1.0 / L), rtol=1e-14, atol=0,
                                   err_msg=f"bs={bs} t={t}")


# -- closed forms and special cases ---------------------------------------------

def test_constant_v_returns_v(oracle_mod):
    gen = torch.Generator().manual_seed(1)
    L, hkv, d, hq = 300, 2, 64, 6
    k = randn_bf16((L, hkv, d), gen)
    row = randn_bf16((hkv, d), gen)
    v = row.unsqueeze(0).expand(L, hkv, d).contiguous()
    kc, vc, bt = place_in_pages([k], [v], 16, 24, seed=2)
    q = randn_bf16((1, hq, d), gen)
    out = _run(oracle_mod, q, kc, vc, bt, [L], 0.125)
    for h in range(hq):
        np.testing.assert_allclose(out[0, h], row[h // 3].double().numpy(), rtol=1e-14, atol=1e-14)


def test_single_token_returns_its_v(oracle_mod):
    gen = torch.Generator().manual_seed(3)
    hkv, d, hq = 4, 32, 8
    k = randn_bf16((1, hkv, d), gen)
    v = randn_bf16((1, hkv, d), gen)
    kc, vc, bt = place_in_pages([k], [v], 16, 4, seed=4)
    q = randn_bf16((1, hq, d), gen)
    out = _run(oracle_mod, q, kc, vc, bt, [1], 0.3)
    for h in range(hq):
        assert np.array_equal(out[0, h], v[0, h // 2].double().numpy())


def test_zero_scale_is_mean_of_v(oracle_mod):
    gen = torch.Generator().manual_seed(5)
    L, hkv, d, hq = 777, 1, 16, 3
    k, v = _contig(gen, [L], hkv, d)
    kc, vc, bt = place_in_pages(k, v, 784, 3, seed=6)
    q = randn_bf16((1, hq, d), gen)
    out = _run(oracle_mod, q, kc, vc, bt, [L], 0.0)
    mean = v[0][:, 0, :].double().mean(dim=0).numpy()
    for h in range(hq):
        np.testing.assert_allclose(out[0, h], mean, rtol=1e-13, atol=1e-15)


def test_zero_query_is_mean_of_v(oracle_mod):
    gen = torch.Generator().manual_seed(7)
    L, hkv, d = 100, 2, 16
    k, v = _contig(gen, [L], hkv, d)
    kc, vc, bt = place_in_pages(k, v, 16, 10, seed=8)
    q = torch.zeros((1, 4, d), dtype=torch.bfloat16)
    out = _run(oracle_mod, q, kc, vc, bt, [L], 1 / 4)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], v[0][:, h // 2, :].double().mean(0).numpy(), rtol=1e-13)


def test_large_logits_pick_the_argmax(oracle_mod):
    """Scores of order 1e4: without the max subtraction exp() overflows."""
    gen = torch.Generator().manual_seed(9)
    L, d = 50, 8
    k = torch.zeros((L, 1, d), dtype=torch.bfloat16)
    k[:, 0, 0] = torch.arange(L, dtype=torch.float32).to(torch.bfloat16)  # token 49 is the largest
    v = randn_bf16((L, 1, d), gen)
    kc, vc, bt = place_in_pages([k], [v], 16, 5, seed=10)
    q = torch.zeros((1, 1, d), dtype=torch.bfloat16)
    q[0, 0, 0] = 256.0
    out = _run(oracle_mod, q, kc, vc, bt, [L], 1.0)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], v[L - 1, 0].double().numpy(), rtol=1e-12, atol=1e-12)


def test_empty_context_is_zero(oracle_mod):
    gen = torch.Generator().manual_seed(11)
    k, v = _contig(gen, [5], 1, 8)
    kc, vc, bt = place_in_pages(k, v, 16, 2, seed=1)
    q = randn_bf16((2, 2, 8), gen)
    out = _run(oracle_mod, q, kc, vc, torch.cat([bt, bt]), [0, 5], 0.5)
    assert np.all(out[0] == 0.0) and np.any(out[1] != 0.0)


# -- invariants --------------------------------------------------------------------

def test_page_permutation_invariance_bitwise(oracle_mod):
    gen = torch.Generator().manual_seed(12)
    lens = [1000, 37]
    k, v = _contig(gen, lens, 2, 64)
    q = randn_bf16((2, 6, 64), gen)
    outs = []
    for seed in (1, 2, 3):
        kc, vc, bt = place_in_pages(k, v, 16, 70, seed=seed)
        outs.append(_run(oracle_mod, q, kc, vc, bt, lens, 0.125))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_paging_invariance_784_832_16_bitwise(oracle_mod):
    gen = torch.Generator().manual_seed(13)
    lens = [2000, 785]
    k, v = _contig(gen, lens, 2, 32)
    q = randn_bf16((2, 4, 32), gen)
    outs = []
    for bs, pages in ((784, 6), (832, 5), (16, 180)):
        kc, vc, bt = place_in_pages(k, v, bs, pages, seed=bs)
        outs.append(_run(oracle_mod, q, kc, vc, bt, lens, 0.2))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_gqa_head_mapping_is_contiguous(oracle_mod):
    """Query head h reads KV head h // G: V constant per KV head identifies it.
    (An interleaved mapping h % Hkv would give a different pattern.)"""
    L, hkv, hq, d = 40, 4, 24, 8
    gen = torch.Generator().manual_seed(14)
    k = randn_bf16((L, hkv, d), gen)
    v = torch.zeros((L, hkv, d), dtype=torch.bfloat16)
    for j in range(hkv):
        v[:, j, :] = float(j + 1)
    kc, vc, bt = place_in_pages([k], [v], 16, 4, seed=3)
    q = randn_bf16((1, hq, d), gen)
    out = _run(oracle_mod, q, kc, vc, bt, [L], 1 / 16)
    for h in range(hq):
        np.testing.assert_allclose(out[0, h], np.full(d, float(h // 6 + 1)), rtol=1e-14)


def test_identical_queries_in_a_group_agree(oracle_mod):
    gen = torch.Generator().manual_seed(15)
    k, v = _contig(gen, [300], 2, 16)
    kc, vc, bt = place_in_pages(k, v, 16, 20, seed=1)
    q = randn_bf16((1, 4, 16), gen)
    q[0, 1] = q[0, 0]
    out = _run(oracle_mod, q, kc, vc, bt, [300], 0.25)
    assert np.array_equal(out[0, 0], out[0, 1]) and not np.array_equal(out[0, 0], out[0, 2])


def test_batch_independence(oracle_mod):
    gen = torch.Generator().manual_seed(16)
    lens = [129, 513, 64]
    k, v = _contig(gen, lens, 1, 16)
    q = randn_bf16((3, 2, 16), gen)
    kc, vc, bt = place_in_pages(k, v, 16, 48, seed=2)
    full = _run(oracle_mod, q, kc, vc, bt, lens, 0.25)
    for b in range(3):
        one = _run(oracle_mod, q[b:b + 1], kc, vc, bt[b:b + 1], lens[b:b + 1], 0.25)
        assert np.array_equal(one[0], full[b])


# -- against a library routine on tiny inputs ----------------------------------------

@pytest.mark.parametrize("lens,hq,hkv,d,bs,q_len", [
    ([1, 17, 50], 6, 1, 8, 16, 1),
    ([33], 24, 4, 16, 16, 1),
    ([70, 5], 4, 2, 32, 784, 1),
    ([20, 31], 6, 2, 8, 16, 4),
    ([16, 40], 12, 1, 16, 832, 5),
])
def test_bruteforce_dense_softmax(oracle_mod, lens, hq, hkv, d, bs, q_len):
    gen = torch.Generator().manual_seed(sum(lens) + hq + d)
    k, v = _contig(gen, lens, hkv, d)
    q = randn_bf16((len(lens) * q_len, hq, d), gen)
    pages = sum(math.ceil(L / bs) for L in lens) + 1
    kc, vc, bt = place_in_pages(k, v, bs, pages, seed=9)
    scale = 1 / math.sqrt(d)
    out = _run(oracle_mod, q, kc, vc, bt, lens, scale, q_len=q_len)
    ref = dense_attention(q, k, v, scale, q_len, hkv).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_verify_row_equals_decode_on_prefix(oracle_mod):
    gen = torch.Generator().manual_seed(17)
    q_len, L = 6, 100
    k, v = _contig(gen, [L], 2, 16)
    kc, vc, bt = place_in_pages(k, v, 16, 8, seed=3)
    q = randn_bf16((q_len, 4, 16), gen)
    ver = _run(oracle_mod, q, kc, vc, bt, [L], 0.25, q_len=q_len)
    for r in range(q_len):
        dec = _run(oracle_mod, q[r:r + 1], kc, vc, bt, [L - q_len + r + 1], 0.25)
        assert np.array_equal(ver[r], dec[0])


# -- the split method: partials and their log-sum-exp merge ----------------------

def test_lse_combine_closed_form(oracle_mod):
    o = np.array([[1.0, 0.0], [0.0, 2.0]])
    m = np.array([0.5, 1.5])
    l = np.array([2.0, 3.0])
    w = np.array([2.0 * math.exp(-1.0), 3.0])
    expect = (w[0] * o[0] + w[1] * o[1]) / w.sum()
    np.testing.assert_allclose(oracle_mod.lse_combine(o, m, l), expect, rtol=1e-15)
    # an empty split (l = 0, m = -inf) carries no weight
    o2 = np.vstack([o, np.full((1, 2), 7.0)])
    np.testing.assert_allclose(oracle_mod.lse_combine(o2, np.append(m, -np.inf), np.append(l, 0.0)),
                               expect, rtol=1e-15)
    assert np.all(oracle_mod.lse_combine(o[:1], np.array([-np.inf]), np.array([0.0])) == 0.0)


def test_split_then_reduce_equals_whole(oracle_mod):
    gen = torch.Generator().manual_seed(18)
    L, d = 2000, 32
    k, v = _contig(gen, [L], 1, d)
    kc, vc, bt = place_in_pages(k, v, 784, 4, seed=5)
    q = randn_bf16((1, 2, d), gen)
    full = _run(oracle_mod, q, kc, vc, bt, [L], 0.3)
    rng = np.random.default_rng(0)
    for trial in range(4):
        cuts = np.sort(rng.choice(np.arange(1, L), size=trial * 5 + 1, replace=False))
        edges = [0] + cuts.tolist() + [L + 64]  # the last split runs past the end
        parts = [oracle_mod.attention_partial(bits(q), bits(kc), bits(vc), bt.numpy(),
                                              np.array([L], np.int32), 0.3, 0, 1, a, b)
                 for a, b in zip(edges[:-1], edges[1:])]
        o = np.stack([p[0] for p in parts])
        merged = oracle_mod.lse_combine(o, np.array([p[1] for p in parts]), np.array([p[2] for p in parts]))
        np.testing.assert_allclose(merged, full[0, 1], rtol=1e-12, atol=1e-14)


# -- sliding window ("last 2048 positions" of the RTX 3090 page) ------------------------

def _window_problem(seed, lens, q_len, hq=6, hkv=2, d=16, bs=16):
    gen = torch.Generator().manual_seed(seed)
    k, v = _contig(gen, lens, hkv, d)
    q = randn_bf16((len(lens) * q_len, hq, d), gen)
    pages = sum(math.ceil(L / bs) for L in lens) + 1
    kc, vc, bt = place_in_pages(k, v, bs, pages, seed=seed + 1)
    return k, v, q, kc, vc, bt


@pytest.mark.parametrize("q_len", [1, 5])
def test_window_wider_than_context_is_full_attention_bitwise(oracle_mod, q_len):
    lens = [40, 77, 5]
    k, v, q, kc, vc, bt = _window_problem(31, lens, q_len)
    full = _run(oracle_mod, q, kc, vc, bt, lens, 0.25, q_len=q_len)
    for w in (77, 78, 10**6):
        assert np.array_equal(_run(oracle_mod, q, kc, vc, bt, lens, 0.25, q_len=q_len, window=w), full)


@pytest.mark.parametrize("q_len", [1, 5])
def test_window_of_one_returns_the_last_visible_v(oracle_mod, q_len):
    lens = [40, 77, 9]
    k, v, q, kc, vc, bt = _window_problem(32, lens, q_len)
    out = _run(oracle_mod, q, kc, vc, bt, lens, 0.25, q_len=q_len, window=1)
    for b, L in enumerate(lens):
        for r in range(q_len):
            t = L - q_len + r  # the row's own (last visible) key
            for h in range(6):
                np.testing.assert_array_equal(out[b * q_len + r, h], v[b][t, h // 3].double().numpy())


@pytest.mark.parametrize("lens,q_len,window", [([200, 37], 1, 16), ([200, 37], 1, 50), ([150], 7, 33),
                                               ([64, 90], 4, 17)])
def test_window_bruteforce_dense_softmax(oracle_mod, lens, q_len, window):
    k, v, q, kc, vc, bt = _window_problem(33 + window, lens, q_len)
    out = _run(oracle_mod, q, kc, vc, bt, lens, 0.25, q_len=q_len, window=window)
    ref = dense_attention(q, k, v, 0.25, q_len, 2, window=window).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
    # a wrong window edge (one key more or less) would be caught at this tolerance
    assert not np.allclose(out, dense_attention(q, k, v, 0.25, q_len, 2, window=window + 1).numpy(),
                           rtol=1e-9, atol=1e-9)


def test_window_equals_the_split_over_its_keys_bitwise(oracle_mod):
    lens, W = [500], 64
    k, v, q, kc, vc, bt = _window_problem(34, lens, 1)
    out = _run(oracle_mod, q, kc, vc, bt, lens, 0.3, window=W)
    for h in range(6):
        o, m, l = oracle_mod.attention_partial(bits(q), bits(kc), bits(vc), bt.numpy(), np.array(lens, np.int32),
                                               0.3, 0, h, lens[0] - W, lens[0])
        assert np.array_equal(out[0, h], o)


# -- reshape_and_cache --------------------------------------------------------------

def test_reshape_and_cache_scatter_bit_exact(oracle_mod):
    gen = torch.Generator().manual_seed(19)
    P, bs, hkv, d, n = 6, 16, 2, 8, 9
    kc = bits(randn_bf16((P, bs, hkv, d), gen)).copy()
    vc = bits(randn_bf16((P, bs, hkv, d), gen)).copy()
    k0, v0 = kc.copy(), vc.copy()
    kn = randn_bf16((n, hkv, d), gen)
    vn = randn_bf16((n, hkv, d), gen)
    slots = np.array([0, 15, 16, 95, -1, 40, 41, 17, 63], dtype=np.int64)
    oracle_mod.reshape_and_cache(bits(kn), bits(vn), kc, vc, slots)
    written = np.zeros((P, bs), dtype=bool)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(kc[s // bs, s % bs], bits(kn)[i])
        assert np.array_equal(vc[s // bs, s % bs], bits(vn)[i])
        written[s // bs, s % bs] = True
    assert np.array_equal(kc[~written], k0[~written]) and np.array_equal(vc[~written], v0[~written])
    with pytest.raises(ValueError):
        oracle_mod.reshape_and_cache(bits(kn[:1]), bits(vn[:1]), kc, vc, np.array([P * bs], np.int64))


# -- byte accounting ---------------------------------------------------------------------

def test_kv_bytes_per_token_closed_form():
    """2 (K and V) x Hkv x D x 2 bytes per context token per layer: 4096 B for
    both the hybrid (4 x 256) and the dense control (8 x 128) shapes; over the
    hybrid model's 16 full-attention layers that is the 64 KiB per token the
    Radeon decode-collapse page quotes."""
    assert 2 * 4 * 256 * 2 == 4096 and 2 * 8 * 128 * 2 == 4096
    assert 16 * 4096 == 64 * 1024


# -- hybrid page size -------------------------------------------------------------

def test_hybrid_page_golden(oracle_mod):
    """The article's example: a state page worth 769..784 attention tokens is a
    784-token page at 16-token alignment and an 832-token page at 64."""
    spec = json.load(open(os.path.join(GOLDEN, "hybrid_page.json")))
    lo, hi = spec["state_tokens_range"]
    for per_token in (4096, 2 * 4 * 256 * 2 * 16, 1):
        for n in (lo, (lo + hi) // 2, hi):
            for case in spec["cases"]:
                got = oracle_mod.hybrid_page_tokens(n * per_token, per_token, case["alignment"])
                assert got == case["page"], (n, per_token, case)
    for page, pct in spec["capacity_growth_pct"].items():
        assert abs(100.0 * (int(page) / 784 - 1) - pct) < 0.05


def test_hybrid_page_bruteforce(oracle_mod):
    """The smallest multiple of the alignment whose attention capacity covers
    the state page, found by walking the multiples."""
    for align in (1, 16, 64):
        for per_token in (1, 3, 4096):
            for state in (1, per_token * 5 - 1, per_token * 64, per_token * 64 + 1, per_token * 781 + 7):
                page = align
                while page * per_token < state:
                    page += align
                assert oracle_mod.hybrid_page_tokens(state, per_token, align) == page
    assert oracle_mod.hybrid_page_tokens(0, 4096, 16) == -1
    assert oracle_mod.hybrid_page_tokens(100, 0, 16) == -1
    assert oracle_mod.hybrid_page_tokens(100, 4096, 0) == -1


# -- fp8 e4m3 KV cache -------------------------------------------------------------

E4M3_NAN_CODES = (0x7F, 0xFF)


def _torch_e4m3_values():
    """Every code's value through torch's float8_e4m3fn type (a library routine)."""
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_decode_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle_mod.e4m3_decode(codes)
    ref = _torch_e4m3_values()
    nan = np.isnan(got)
    assert sorted(np.flatnonzero(nan).tolist()) == list(E4M3_NAN_CODES)
    assert np.array_equal(got[~nan], ref[~nan]) and np.isnan(ref[nan]).all()
    # points fixed by the format: 1 sign, 4 exponent (bias 7), 3 mantissa bits
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0      # largest finite
    assert got[0x08] == 2.0 ** -6 and got[0x07] == 7 * 2.0 ** -9  # smallest normal, largest subnormal
    assert got[0x01] == 2.0 ** -9                           # smallest subnormal
    assert got[0x38] == 1.0 and got[0x40] == 2.0 and got[0x39] == 1.125
    assert got[0x80] == 0.0 and math.copysign(1.0, got[0x80]) == -1.0


def test_e4m3_encode_round_trip_and_ties(oracle_mod):
    vals = oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = [c for c in range(256) if c not in E4M3_NAN_CODES]
    # every value encodes to its own code
    assert np.array_equal(oracle_mod.e4m3_encode(vals[finite].astype(np.float32)), np.array(finite, np.uint8))
    # midpoints between neighbours round to the even code; just off them, to the nearer one
    pos = sorted(v for v in vals[:0x7F] if v >= 0)
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = (lo + hi) / 2
        even = lo if int(oracle_mod.e4m3_encode(np.float32([lo]))[0]) % 2 == 0 else hi
        got = oracle_mod.e4m3_decode(oracle_mod.e4m3_encode(np.float32([mid, -mid])))
        assert got[0] == even and got[1] == -even, (lo, hi)
        below, above = np.nextafter(np.float32(mid), np.float32(0)), np.nextafter(np.float32(mid), np.float32(1e9))
        got = oracle_mod.e4m3_decode(oracle_mod.e4m3_encode(np.float32([below, above])))
        assert got[0] == lo and got[1] == hi


def test_e4m3_encode_matches_torch_in_range(oracle_mod):
    """Nearest-even rounding agrees with torch's float8_e4m3fn cast wherever the
    cast does not overflow (torch turns |x| >= 464 into NaN; the cache saturates)."""
    g = torch.Generator().manual_seed(5)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x[x.abs() < 464].float()
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle_mod.e4m3_encode(x.numpy()), ref)


def test_e4m3_encode_saturates(oracle_mod):
    x = np.float32([448.0, 448.5, 463.9, 464.0, 1e9, np.inf, -500.0, -np.inf, np.nan, -np.nan, 0.0, -0.0])
    got = oracle_mod.e4m3_encode(x)
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0xFF, 0x00, 0x80]


def _fp8_problem(gen, lens, hkv, d, bs, exact_scales):
    """Random finite e4m3 codes paged through a block table, with per-head scales
    (powers of two when exact_scales: decoded x scale is then a bf16 value)."""
    P = sum(math.ceil(L / bs) for L in lens) + 2
    kc = torch.randint(0, 256, (P, bs, hkv, d), generator=gen).to(torch.uint8)
    vc = torch.randint(0, 256, (P, bs, hkv, d), generator=gen).to(torch.uint8)
    for c in (kc, vc):
        c[(c & 0x7F) == 0x7F] = 0x3C  # no NaN codes
        c[(c & 0x78) >= 0x58] &= 0xC7  # |value| < 16: softmax stays well spread
    if exact_scales:
        ks = np.float32([2.0 ** -(3 + h) for h in range(hkv)])
        vs = np.float32([2.0 ** -(1 + 2 * h) for h in range(hkv)])
    else:
        ks = np.float32([0.0371 * (1 + h) for h in range(hkv)])
        vs = np.float32([0.113 / (1 + h) for h in range(hkv)])
    perm = torch.randperm(P, generator=gen)
    npg = max(math.ceil(L / bs) for L in lens)
    bt = torch.full((len(lens), npg), -1, dtype=torch.int32)
    cur = 0
    for b, L in enumerate(lens):
        for lp in range(math.ceil(L / bs)):
            bt[b, lp] = int(perm[cur])
            cur += 1
    return kc.numpy(), vc.numpy(), ks, vs, bt


def test_fp8_attention_equals_bf16_attention_on_the_decoded_values_bitwise(oracle_mod):
    """With power-of-two scales every dequantised element is a bf16 value: the
    fp8 path must then give exactly the bf16 path's result on that cache."""
    gen = torch.Generator().manual_seed(61)
    lens, hkv, d, bs, hq = [37, 1, 100, 16], 2, 16, 16, 6
    kc, vc, ks, vs, bt = _fp8_problem(gen, lens, hkv, d, bs, exact_scales=True)
    kd = oracle_mod.e4m3_decode(kc) * ks[None, None, :, None]
    vd = oracle_mod.e4m3_decode(vc) * vs[None, None, :, None]
    kb = torch.from_numpy(kd).to(torch.bfloat16)
    vb = torch.from_numpy(vd).to(torch.bfloat16)
    assert np.array_equal(kb.double().numpy(), kd) and np.array_equal(vb.double().numpy(), vd)
    for q_len, window in ((1, 0), (1, 20), (3, 0)):
        q = randn_bf16((len(lens) * q_len, hq, d), gen)
        sl = np.int32([max(L, q_len) for L in lens])
        ref = _run(oracle_mod, q, kb, vb, bt, sl, 0.25, q_len=q_len, window=window)
        got = oracle_mod.paged_attention_fp8(bits(q), kc, vc, ks, vs, bt.numpy(), sl, 0.25, q_len=q_len,
                                             window=window, num_threads=3)
        assert np.array_equal(got, ref), (q_len, window)


def test_fp8_attention_bruteforce_dense_softmax(oracle_mod):
    """Arbitrary per-head scales against torch fp64 softmax over the dequantised
    contiguous K/V (codes decoded by torch's float8 type)."""
    gen = torch.Generator().manual_seed(67)
    lens, hkv, d, bs, hq = [50, 7, 33], 3, 8, 16, 6
    kc, vc, ks, vs, bt = _fp8_problem(gen, lens, hkv, d, bs, exact_scales=False)
    kt = torch.from_numpy(kc).view(torch.float8_e4m3fn).double() * torch.from_numpy(ks).double()[None, None, :, None]
    vt = torch.from_numpy(vc).view(torch.float8_e4m3fn).double() * torch.from_numpy(vs).double()[None, None, :, None]
    k_list, v_list = [], []
    for b, L in enumerate(lens):
        k_list.append(torch.cat([kt[int(bt[b, t // bs])][t % bs: t % bs + 1] for t in range(L)]))
        v_list.append(torch.cat([vt[int(bt[b, t // bs])][t % bs: t % bs + 1] for t in range(L)]))
    q = randn_bf16((len(lens), hq, d), gen)
    ref = dense_attention(q, k_list, v_list, 0.3, 1, hkv).numpy()
    got = oracle_mod.paged_attention_fp8(bits(q), kc, vc, ks, vs, bt.numpy(), np.int32(lens), 0.3)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_reshape_and_cache_fp8_quantises_and_scatters(oracle_mod):
    """Codes equal torch's float8 cast of (bf16 value / head scale) in binary32
    (inputs kept inside +-448), written at (slot / BS, slot % BS); other slots untouched."""
    gen = torch.Generator().manual_seed(71)
    P, bs, hkv, d, n = 5, 16, 3, 32, 11
    kc = np.full((P, bs, hkv, d), 0x55, np.uint8)
    vc = np.full((P, bs, hkv, d), 0xAA, np.uint8)
    kn = randn_bf16((n, hkv, d), gen)
    vn = randn_bf16((n, hkv, d), gen)
    ks = np.float32([0.02, 0.05, 0.013])
    vs = np.float32([0.011, 0.3, 0.07])
    slots = np.array([0, 15, 16, 79, -1, 40, 41, 17, 63, 2, 3], dtype=np.int64)
    oracle_mod.reshape_and_cache_fp8(bits(kn), bits(vn), kc, vc, slots, ks, vs)
    kq = (kn.float() / torch.from_numpy(ks)[None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    vq = (vn.float() / torch.from_numpy(vs)[None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    written = np.zeros((P, bs), dtype=bool)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(kc[s // bs, s % bs], kq[i]) and np.array_equal(vc[s // bs, s % bs], vq[i])
        written[s // bs, s % bs] = True
    assert (kc[~written] == 0x55).all() and (vc[~written] == 0xAA).all()
    with pytest.raises(ValueError):
        oracle_mod.reshape_and_cache_fp8(bits(kn[:1]), bits(vn[:1]), kc, vc, np.array([P * bs], np.int64), ks, vs)
