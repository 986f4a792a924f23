"""GPU checks of PA_FLAG_EARLY_KV_READ: decode and verify may stream the cached
context before the work ahead of them on the stream has finished, but must
read the rows that work writes (the new tokens from reshape_and_cache) only
afterwards.  The flag changes the order of the reads, not the arithmetic, so
its outputs must equal the default path bit for bit; chained after
reshape_and_cache on one stream without a host sync, the new rows must be
seen (parity with the oracle on the updated cache).
"""
import pytest
import torch

import paged_attention_decode_split_gb300 as pa
from paged_attention_decode_split_gb300 import _build
from paged_attention_decode_split_gb300.inputs import make_new_tokens, make_problem
from tests.gpu_common import (REL_L2_VERIFY, assert_cache_written, assert_parity, desc_for, oracle_out, run_attention,
                              to_dev)

pytestmark = pytest.mark.gpu

EARLY = pa.PA_FLAG_EARLY_KV_READ


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    pa.load_library()


def hybrid(seed, lens, bs, **kw):
    args = dict(num_seqs=len(lens), seq_lens=list(lens), num_q_heads=24, num_kv_heads=4, head_dim=256,
                block_size=bs, scale=1 / 16)
    args.update(kw)
    return make_problem(seed, **args)


def call(prob, tensors, flags, num_splits=0):
    q, kc, vc, bt, sl = tensors
    desc = desc_for(prob, num_splits=num_splits)
    desc.flags = flags
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device="cuda")
    out = torch.full((prob.num_seqs * prob.q_len, prob.num_q_heads, prob.head_dim), float("nan"),
                     dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if prob.kv_fp8:
        ks, vs = prob.k_scale[0].cuda(), prob.v_scale[0].cuda()
        fn = pa.paged_attention_decode_fp8 if prob.q_len == 1 else pa.paged_attention_verify_fp8
        fn(q, kc, vc, ks, vs, bt, sl, desc, out, ws, status)
    else:
        fn = pa.paged_attention_decode if prob.q_len == 1 else pa.paged_attention_verify
        fn(q, kc, vc, bt, sl, desc, out, ws, status)
    return out, status


# The dense shape (8 KV heads of 128 dims) runs the kernels whose chunk
# streams each have their own producer lane; the hybrid shape one lane for all.
DENSE = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, scale=128 ** -0.5)
SHAPES = {"hybrid": {}, "dense": DENSE}


@pytest.mark.parametrize("shape", ["hybrid", "dense"])
@pytest.mark.parametrize("splits", [0, 1, 5])
@pytest.mark.parametrize("bs", [16, 784])
def test_decode_early_equals_default_bitwise(bs, splits, shape):
    prob = hybrid(301 + bs, [1, 15, 16, 17, 785, 5000, 0], bs, poison_unused=True, **SHAPES[shape])
    t = to_dev(prob)
    ref, st0 = call(prob, t, 0, splits)
    got, st1 = call(prob, t, EARLY, splits)
    torch.cuda.synchronize()
    assert st0.item() == 0 and st1.item() == 0
    assert torch.equal(got.cpu(), ref.cpu())


@pytest.mark.parametrize("q_len,lens,bs", [(16, [16, 17, 831, 1700], 832), (5, [5, 64, 785], 784)])
def test_verify_early_equals_default_bitwise(q_len, lens, bs):
    prob = hybrid(311 + q_len, lens, bs, q_len=q_len, poison_unused=True)
    t = to_dev(prob)
    ref, _ = call(prob, t, 0)
    got, _ = call(prob, t, EARLY)
    torch.cuda.synchronize()
    assert torch.equal(got.cpu(), ref.cpu())


# Several 128-row blocks per KV head (40 rows x 6 heads = 240), one and three
# splits, the bf16 and the fp8 cache: with early K/V reads only the softmax and
# MMA warps synchronise on the tensor-memory address, the other warps stream on.
@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("splits", [1, 3])
def test_verify_row_blocks_early_equals_default_bitwise(fp8, splits):
    prob = hybrid(321 + splits, [40, 900, 2100], 784, q_len=40, poison_unused=True, kv_fp8=fp8)
    t = to_dev(prob)
    ref, st0 = call(prob, t, 0, splits)
    got, st1 = call(prob, t, EARLY, splits)
    torch.cuda.synchronize()
    assert st0.item() == 0 and st1.item() == 0
    assert torch.equal(got.cpu(), ref.cpu())


def chained(prob, seed, flags):
    """reshape_and_cache of the new rows, then the attention call, on one stream
    with no host synchronisation in between; returns (out, status, updated prob)."""
    k_new, v_new = make_new_tokens(seed, prob.num_seqs * prob.q_len, prob.num_kv_heads, prob.head_dim)
    q, kc, vc, bt, sl = to_dev(prob)
    kn, vn, slots = k_new.cuda(), v_new.cuda(), prob.new_token_slots().cuda()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(2_000_000)  # keeps the stream busy so the chain overlaps on the device
        pa.reshape_and_cache(kn, vn, kc, vc, slots)
        out, status = call(prob, (q, kc, vc, bt, sl), flags)
    torch.cuda.synchronize()
    import oracle
    assert_cache_written(oracle, prob.k_cache[0], prob.v_cache[0], k_new, v_new, slots, kc, vc)
    prob.k_cache[0], prob.v_cache[0] = kc.cpu(), vc.cpu()
    return out.cpu(), status.item(), prob


@pytest.mark.parametrize("lens,bs,shape", [([32768], 784, "hybrid"), ([17, 4000, 1], 16, "hybrid"),
                                           ([832, 833], 832, "hybrid"), ([17, 4000, 1], 16, "dense"),
                                           ([32768], 16, "dense")])
def test_decode_early_chain_reads_new_row(oracle_mod, lens, bs, shape):
    prob = hybrid(321, lens, bs, **SHAPES[shape])
    out, status, prob = chained(prob, 7, EARLY)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), what="early decode after reshape_and_cache")


def test_verify_early_chain_reads_new_rows(oracle_mod):
    prob = hybrid(331, [8208, 8208, 100], 832, q_len=16)
    out, status, prob = chained(prob, 9, EARLY)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY,
                  what="early verify after reshape_and_cache")


def test_early_step_graph_equals_default_bitwise():
    """Four layers of (reshape_and_cache, decode) captured in one graph, with
    and without the flag: identical outputs and caches."""
    outs = []
    for flags in (0, EARLY):
        prob = make_problem(341, num_seqs=2, seq_lens=[3000, 777], num_q_heads=24, num_kv_heads=4, head_dim=256,
                            block_size=784, scale=1 / 16, num_layers=4, device="cuda")
        k_new, v_new = make_new_tokens(13, 4 * 2, 4, 256, device="cuda")
        k_new, v_new = k_new.view(4, 2, 4, 256), v_new.view(4, 2, 4, 256)
        slots = prob.new_token_slots().cuda()
        bt, sl = prob.block_table.cuda(), prob.seq_lens.cuda()
        desc = desc_for(prob)
        desc.flags = flags
        ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device="cuda")
        out = torch.zeros((4, 2, 24, 256), dtype=torch.float32, device="cuda")
        s = torch.cuda.Stream()

        def step():
            for l in range(4):
                pa.reshape_and_cache(k_new[l], v_new[l], prob.k_cache[l], prob.v_cache[l], slots)
                pa.paged_attention_decode(prob.q[l], prob.k_cache[l], prob.v_cache[l], bt, sl, desc, out[l], ws)

        with torch.cuda.stream(s):
            step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        outs.append(out.cpu())
    assert torch.equal(outs[0], outs[1])
