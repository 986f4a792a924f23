"""GPU parity of the fused append + decode (pa_paged_attention_decode_append
and its fp8 form): each sequence's new token is written into the cache slot
of position seq_lens[b] - 1 and read by the same call.  The cache it leaves
must equal the oracle's scatter of the new rows bit for bit, the output must
match the oracle's attention over that cache, and both must equal, bit for
bit, reshape_and_cache followed by the ordinary decode."""
import math

import numpy as np
import pytest
import torch

import paged_attention_decode_split_gb300 as pa
from paged_attention_decode_split_gb300 import _build
from paged_attention_decode_split_gb300.inputs import make_new_tokens, make_problem
from tests.gpu_common import assert_cache_written, assert_parity, desc_for, oracle_out, to_dev
from tests.helpers import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    pa.load_library()


def problem(seed, lens, bs, fp8=False, hq=24, hkv=4, d=256):
    return make_problem(seed, num_seqs=len(lens), seq_lens=list(lens), num_q_heads=hq, num_kv_heads=hkv,
                        head_dim=d, block_size=bs, scale=1 / math.sqrt(d), poison_unused=True, kv_fp8=fp8)


def run_fused(prob, k_new, v_new, num_splits=0, flags=0, window=0):
    q, kc, vc, bt, sl = to_dev(prob)
    desc = desc_for(prob, num_splits=num_splits, flags=flags, window=window)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device="cuda")
    out = torch.full((prob.num_seqs, prob.num_q_heads, prob.head_dim), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if prob.kv_fp8:
        ks, vs = prob.k_scale[0].cuda(), prob.v_scale[0].cuda()
        pa.paged_attention_decode_append_fp8(q, k_new.cuda(), v_new.cuda(), kc, vc, ks, vs, bt, sl, desc, out, ws,
                                             status)
    else:
        pa.paged_attention_decode_append(q, k_new.cuda(), v_new.cuda(), kc, vc, bt, sl, desc, out, ws, status)
    torch.cuda.synchronize()
    return out.cpu(), kc.cpu(), vc.cpu(), int(status.item()), pa.last_plan()


def run_two_calls(prob, k_new, v_new, num_splits=0, flags=0, window=0):
    q, kc, vc, bt, sl = to_dev(prob)
    slots = prob.new_token_slots().cuda()
    desc = desc_for(prob, num_splits=num_splits, flags=flags, window=window)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device="cuda")
    out = torch.full((prob.num_seqs, prob.num_q_heads, prob.head_dim), float("nan"), device="cuda")
    if prob.kv_fp8:
        ks, vs = prob.k_scale[0].cuda(), prob.v_scale[0].cuda()
        pa.reshape_and_cache_fp8(k_new.cuda(), v_new.cuda(), kc, vc, slots, ks, vs)
        pa.paged_attention_decode_fp8(q, kc, vc, ks, vs, bt, sl, desc, out, ws)
    else:
        pa.reshape_and_cache(k_new.cuda(), v_new.cuda(), kc, vc, slots)
        pa.paged_attention_decode(q, kc, vc, bt, sl, desc, out, ws)
    torch.cuda.synchronize()
    return out.cpu(), kc.cpu(), vc.cpu()


def oracle_cache(oracle_mod, prob, k_new, v_new):
    """The caches after the oracle's scatter of the new rows (CPU copies)."""
    slots = prob.new_token_slots().numpy()
    if prob.kv_fp8:
        k_ref, v_ref = prob.k_cache[0].numpy().copy(), prob.v_cache[0].numpy().copy()
        oracle_mod.reshape_and_cache_fp8(k_new, v_new, k_ref, v_ref, slots, prob.k_scale[0].numpy(),
                                         prob.v_scale[0].numpy())
        return torch.from_numpy(k_ref), torch.from_numpy(v_ref)
    k_ref, v_ref = bits(prob.k_cache[0]).copy(), bits(prob.v_cache[0]).copy()
    oracle_mod.reshape_and_cache(bits(k_new), bits(v_new), k_ref, v_ref, slots)
    as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return as_bf16(k_ref), as_bf16(v_ref)


def check(oracle_mod, prob, seed, **kw):
    k_new, v_new = make_new_tokens(seed, prob.num_seqs, prob.num_kv_heads, prob.head_dim)
    out, kc, vc, status, plan = run_fused(prob, k_new, v_new, **kw)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_DECODE_MMA
    k_ref, v_ref = oracle_cache(oracle_mod, prob, k_new, v_new)
    if prob.kv_fp8:
        assert torch.equal(kc, k_ref) and torch.equal(vc, v_ref), "fused append wrote other codes than the oracle"
    else:
        assert np.array_equal(bits(kc), bits(k_ref)) and np.array_equal(bits(vc), bits(v_ref)), \
            "fused append wrote other rows than the oracle"
    prob.k_cache[0], prob.v_cache[0] = k_ref, v_ref
    assert_parity(out, oracle_out(oracle_mod, prob, window=kw.get("window", 0)), what=f"fused append {kw}")
    return prob, k_new, v_new, out, kc, vc


@pytest.mark.parametrize("bs", [16, 784, 832])
def test_append_ragged_tails(oracle_mod, bs):
    prob = problem(701 + bs, [1, 15, 16, 17, 783, 784, 785, 2000], bs)
    check(oracle_mod, prob, 7)


@pytest.mark.parametrize("splits", [1, 3, 64])
def test_append_forced_splits(oracle_mod, splits):
    check(oracle_mod, problem(711 + splits, [5000, 333, 1], 784), 9, num_splits=splits)


def test_append_equals_two_calls_bitwise(oracle_mod):
    """Same plan, same data: the fused call and reshape_and_cache + decode give
    identical outputs and caches."""
    base = problem(721, [32768, 900, 17], 784)
    k_new, v_new = make_new_tokens(11, 3, 4, 256)
    clone = lambda p: make_problem(721, num_seqs=3, seq_lens=[32768, 900, 17], num_q_heads=24, num_kv_heads=4,
                                   head_dim=256, block_size=784, scale=1 / 16, poison_unused=True)
    for flags in (0, pa.PA_FLAG_EARLY_KV_READ):
        o1, k1, v1, st, _ = run_fused(clone(base), k_new, v_new, flags=flags)
        o2, k2, v2 = run_two_calls(clone(base), k_new, v_new, flags=flags)
        assert st == 0
        # bit patterns: the unused slots hold NaN, which never compares equal
        assert torch.equal(o1, o2)
        assert np.array_equal(bits(k1), bits(k2)) and np.array_equal(bits(v1), bits(v2))


@pytest.mark.parametrize("G,hkv,d,bs", [(8, 4, 128, 16), (12, 4, 256, 784), (1, 8, 128, 16)])
def test_append_other_shapes(oracle_mod, G, hkv, d, bs):
    check(oracle_mod, problem(731 + G, [700, 4097], bs, hq=G * hkv, hkv=hkv, d=d), 13)


def test_append_window_and_early_kv(oracle_mod):
    check(oracle_mod, problem(741, [7000, 100], 784), 15, window=2048, flags=pa.PA_FLAG_EARLY_KV_READ)


@pytest.mark.parametrize("splits", [0, 2])
def test_append_fp8(oracle_mod, splits):
    check(oracle_mod, problem(751 + splits, [3000, 785, 1], 784, fp8=True), 17, num_splits=splits)


def test_append_fp8_equals_two_calls_bitwise():
    k_new, v_new = make_new_tokens(19, 2, 4, 256)
    mk = lambda: problem(761, [4000, 50], 784, fp8=True)
    o1, k1, v1, st, _ = run_fused(mk(), k_new, v_new)
    o2, k2, v2 = run_two_calls(mk(), k_new, v_new)
    assert st == 0 and torch.equal(o1, o2) and torch.equal(k1, k2) and torch.equal(v1, v2)


def test_append_empty_sequence_writes_nothing(oracle_mod):
    """seq_lens[b] == 0: no new token, nothing written, a zero row."""
    prob = problem(771, [0, 500], 16)
    k_new, v_new = make_new_tokens(21, 2, 4, 256)
    out, kc, vc, status, _ = run_fused(prob, k_new, v_new)
    assert status == 0 and torch.all(out[0] == 0)
    changed = (bits(kc) != bits(prob.k_cache[0])).any(axis=(2, 3))
    assert changed.sum() == 1  # only sequence 1's slot, position 499
    page = int(prob.block_table[1, 499 // 16])
    assert changed[page, 499 % 16]


def test_append_bad_page_flagged():
    """The new token's page index outside the pool: nothing written, the
    sequence's rows zeroed, PA_DEV_BAD_PAGE set."""
    prob = problem(781, [900, 900], 16)
    q, kc, vc, bt, sl = to_dev(prob)
    bt[1, 899 // 16] = prob.num_pages + 3
    k_new, v_new = make_new_tokens(23, 2, 4, 256)
    kc0 = kc.clone()
    desc = desc_for(prob)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device="cuda")
    out = torch.empty((2, 24, 256), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.paged_attention_decode_append(q, k_new.cuda(), v_new.cuda(), kc, vc, bt, sl, desc, out, ws, status)
    torch.cuda.synchronize()
    assert status.item() & pa.PA_DEV_BAD_PAGE
    assert torch.all(out[1] == 0) and torch.isfinite(out[0]).all()
    changed = np.argwhere((bits(kc) != bits(kc0)).reshape(kc.shape[0], kc.shape[1], -1).any(-1)).tolist()
    slot0 = int(prob.new_token_slots()[0])
    assert changed == [[slot0 // 16, slot0 % 16]]  # only the good sequence's row was written


def test_append_graph_of_layers_equals_eager():
    """Four layers of the fused call captured in a CUDA graph (each layer its
    own caches) leave the same outputs and caches as eager calls."""
    res = []
    for use_graph in (False, True):
        prob = make_problem(791, num_seqs=2, seq_lens=[3000, 777], num_q_heads=24, num_kv_heads=4, head_dim=256,
                            block_size=784, scale=1 / 16, num_layers=4, device="cuda")
        k_new, v_new = make_new_tokens(25, 8, 4, 256, device="cuda")
        k_new, v_new = k_new.view(4, 2, 4, 256), v_new.view(4, 2, 4, 256)
        bt, sl = prob.block_table.cuda(), prob.seq_lens.cuda()
        desc = desc_for(prob, flags=pa.PA_FLAG_EARLY_KV_READ)
        ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device="cuda")
        out = torch.zeros((4, 2, 24, 256), device="cuda")
        s = torch.cuda.Stream()

        def step():
            for l in range(4):
                pa.paged_attention_decode_append(prob.q[l], k_new[l], v_new[l], prob.k_cache[l], prob.v_cache[l],
                                                 bt, sl, desc, out[l], ws)
        if use_graph:
            with torch.cuda.stream(s):
                step()  # warm-up outside capture (writes the same rows)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                step()
            out.zero_()
            g.replay()
        else:
            with torch.cuda.stream(s):
                step()
        torch.cuda.synchronize()
        res.append((out.cpu(), [c.cpu() for c in prob.k_cache]))
    assert torch.equal(res[0][0], res[1][0])
    assert all(torch.equal(a, b) for a, b in zip(res[0][1], res[1][1]))


def test_append_hybrid_step_l32768_bs784_workload(oracle_mod):
    """The benchmark's step layer in its benchmark launch (automatic plan,
    PA_FLAG_EARLY_KV_READ): the 32K hybrid layer with its new token appended
    and read by the fused call, against the oracle on the oracle-written cache."""
    from paged_attention_decode_split_gb300.inputs import WORKLOADS
    prob = make_problem(1002, **dict(WORKLOADS["hybrid_step_l32768_bs784_x16"], num_layers=1))
    check(oracle_mod, prob, 77, flags=pa.PA_FLAG_EARLY_KV_READ)
    assert pa.last_plan()["num_splits"] == 38
