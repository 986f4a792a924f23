"""GPU parity: the CUDA path through the C ABI against the CPU fp64 oracle.

Small problems are compared element by element; the full-size workloads run
in the launch configuration the benchmark times (automatic split plan) and
are compared on whole layers or sampled sequences.  Edge cases: ragged tails
around every chunk/page boundary, empty sequences, NaN-poisoned unused cache
slots, forced split counts, bad device inputs, bf16 output, graph capture.
"""
import math

import numpy as np
import pytest
import torch

import paged_attention_decode_split_gb300 as pa
from paged_attention_decode_split_gb300 import _build
from paged_attention_decode_split_gb300.inputs import (SWEEP_DEPTHS, WORKLOADS, make_new_tokens, make_problem,
                                                       sweep_workload)
from tests.gpu_common import (REL_L2_DECODE, REL_L2_VERIFY, assert_cache_written, assert_parity, oracle_out,
                               run_attention, to_dev)
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
                block_size=bs, scale=1 / 16)
    args.update(kw)
    return make_problem(seed, **args)


# -- decode ------------------------------------------------------------------------

def test_decode_l512_bs16_workload(oracle_mod):
    prob = make_problem(1001, **WORKLOADS["decode_l512_bs16"])
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_DECODE_MMA
    assert_parity(out, oracle_out(oracle_mod, prob), what="512-token decode")


@pytest.mark.parametrize("bs", [16, 784, 832])
def test_decode_ragged_tails_nan_poisoned(oracle_mod, bs):
    prob = hybrid(7 + bs, TAIL_LENGTHS, bs, poison_unused=True)
    out, status, _ = run_attention(prob)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"tails bs={bs}")


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64, 100, 313])  # > 64: the reduce loads its splits in several rounds
def test_decode_forced_split_counts(oracle_mod, splits):
    prob = hybrid(21, [5000, 333, 1], 784, poison_unused=True)
    out, status, plan = run_attention(prob, num_splits=splits)
    assert status == 0
    n_chunks = math.ceil(5000 / 16)
    per_split = math.ceil(n_chunks / min(splits, n_chunks))
    assert plan["num_splits"] == math.ceil(n_chunks / per_split)  # no empty trailing split
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"splits={splits}")


@pytest.mark.parametrize("splits", [100, 250])
def test_decode_dense_many_splits(oracle_mod, splits):
    """The dense shape (head_dim 128) merged from more than 64 splits."""
    prob = make_problem(23, num_seqs=2, seq_lens=[4000, 90], num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, scale=1 / math.sqrt(128), poison_unused=True)
    out, status, plan = run_attention(prob, num_splits=splits)
    assert status == 0 and plan["num_splits"] > 64
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"dense splits={splits}")


@pytest.mark.parametrize("G,hkv", [(1, 4), (2, 4), (3, 4), (4, 2), (5, 4), (6, 4), (8, 4), (12, 4), (12, 1), (16, 4),
                                   (16, 1)])
def test_decode_group_sizes_d256(oracle_mod, G, hkv):
    prob = hybrid(31 + G, [700, 1500], 16, num_q_heads=G * hkv, num_kv_heads=hkv)
    out, status, _ = run_attention(prob)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"G={G}")


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 8, 12, 16])
def test_decode_dense_control_d128(oracle_mod, G):
    prob = make_problem(41 + G, num_seqs=3, seq_lens=[1, 100, 2049], num_q_heads=8 * G, num_kv_heads=8,
                        head_dim=128, block_size=16, scale=1 / math.sqrt(128), poison_unused=True)
    out, status, _ = run_attention(prob)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"dense G={G}")


@pytest.mark.parametrize("splits", [0, 1, 3, 64])
def test_decode_wide_group_g12(oracle_mod, splits):
    """48 query heads on 4 KV heads: the 12 heads of a group are split over two
    warp groups of 6, which meet again in the CTA merge."""
    prob = hybrid(251 + splits, TAIL_LENGTHS[:7] + [5000], 784, num_q_heads=48, num_kv_heads=4,
                  poison_unused=True)
    out, status, plan = run_attention(prob, num_splits=splits)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_DECODE_MMA
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"G=12 splits={splits}")


def test_decode_empty_sequences_give_zero(oracle_mod):
    prob = hybrid(51, [0, 100, 0], 16)
    out, status, _ = run_attention(prob)
    assert status == 0
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert_parity(out, oracle_out(oracle_mod, prob), what="empty")


@pytest.mark.parametrize("splits", [0, 4, 1])  # the large-split merge, the few-split merge, no merge
def test_decode_bf16_output(oracle_mod, splits):
    prob = hybrid(61, [3000, 17], 832)
    out, status, plan = run_attention(prob, out_dtype=pa.PA_OUT_BF16, num_splits=splits)
    assert splits == 0 or plan["num_splits"] == splits
    ref = oracle_out(oracle_mod, prob)
    ref_bf16 = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    err = np.abs(out.double().numpy() - ref_bf16)
    # one bf16 rounding on each side of a <= 2e-3 difference
    assert status == 0 and err.max() <= 2e-3 + 2 * 2.0 ** -8 * np.abs(ref).max()


def test_decode_deterministic_and_page_size_invariant(oracle_mod):
    """Same tokens, same split plan: results are bitwise identical run to run
    and across 16-, 784- and 832-token pages (chunks never straddle pages)."""
    lens = [4000, 1234]
    outs = []
    base = hybrid(71, lens, 16)
    for bs in (16, 784, 832):
        prob = hybrid(72, lens, bs)
        # copy the logical K/V of `base` into this paging
        for b, L in enumerate(lens):
            for t in range(0, L, 16):
                n = min(16, L - t)
                src_p, src_o = int(base.block_table[b, t // 16]), t % 16
                dst_p, dst_o = int(prob.block_table[b, t // bs]), t % bs
                prob.k_cache[0][dst_p, dst_o:dst_o + n] = base.k_cache[0][src_p, src_o:src_o + n]
                prob.v_cache[0][dst_p, dst_o:dst_o + n] = base.v_cache[0][src_p, src_o:src_o + n]
        prob.q[0] = base.q[0].clone()
        o1, _, _ = run_attention(prob, num_splits=5)
        o2, _, _ = run_attention(prob, num_splits=5)
        assert torch.equal(o1, o2)
        outs.append(o1)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert_parity(outs[0], oracle_out(oracle_mod, base), what="paging invariance")


def test_decode_bad_seq_len_sets_status_and_zeroes(oracle_mod):
    prob = hybrid(81, [300, 200], 16)
    q, kc, vc, bt, sl = to_dev(prob)
    sl[1] = 10_000  # beyond max_seq_len (300)
    out, status, _ = run_attention(prob, tensors=(q, kc, vc, bt, sl), max_seq_len=300)
    assert status & pa.PA_DEV_BAD_SEQLEN
    assert torch.all(out[1] == 0)
    ref = oracle_out(oracle_mod, prob, rows=[0])
    assert_parity(out[:1], ref, what="good row next to a bad one")


@pytest.mark.parametrize("splits", [1, 4])
def test_decode_bad_page_sets_status_and_zeroes(oracle_mod, splits):
    prob = hybrid(91, [900, 900], 16)
    q, kc, vc, bt, sl = to_dev(prob)
    bt[1, 20] = prob.num_pages + 5  # out of range: read as zeros by the copy engine, flagged
    out, status, _ = run_attention(prob, tensors=(q, kc, vc, bt, sl), num_splits=splits)
    assert status & pa.PA_DEV_BAD_PAGE
    assert torch.all(out[1] == 0)
    assert_parity(out[:1], oracle_out(oracle_mod, prob, rows=[0]), what="good row next to a bad page")


def test_workspace_reused_across_descriptions(oracle_mod):
    """One workspace, sized for the largest call, serves calls of other batch
    sizes, split counts and shapes in turn without being cleared: every split
    writes its record, so nothing of an earlier call is read."""
    probs = [hybrid(181, [4000, 2500, 300], 784), hybrid(182, [5000], 784),
             make_problem(183, num_seqs=2, seq_lens=[3000, 40], num_q_heads=32, num_kv_heads=8, head_dim=128,
                          block_size=16, scale=1 / math.sqrt(128)),
             hybrid(184, [700, 20], 832, q_len=8), hybrid(185, [5000], 784), hybrid(186, [4000, 2500, 300], 784)]
    splits = [0, 37, 0, 3, 9, 0]
    from tests.gpu_common import desc_for
    need = max(pa.workspace_bytes(desc_for(p, num_splits=k)) for p, k in zip(probs, splits))
    ws = torch.full((need,), 0xff, dtype=torch.uint8, device="cuda")  # NaN in every fp32 slot
    for prob, k in zip(probs, splits):
        if prob.q_len > 1:
            write_new_rows(prob, 17)
        q, kc, vc, bt, sl = to_dev(prob)
        desc = desc_for(prob, num_splits=k)
        out = torch.empty((prob.num_seqs * prob.q_len, prob.num_q_heads, prob.head_dim), dtype=torch.float32,
                          device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        fn = pa.paged_attention_decode if prob.q_len == 1 else pa.paged_attention_verify
        fn(q, kc, vc, bt, sl, desc, out, ws, status)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert_parity(out.cpu(), oracle_out(oracle_mod, prob),
                      rel_l2=REL_L2_VERIFY if prob.q_len > 1 else REL_L2_DECODE, what=f"reused workspace q_len={prob.q_len}")


def test_decode_cuda_graph_replay_matches_eager():
    prob = hybrid(101, [2500], 784)
    q, kc, vc, bt, sl = to_dev(prob)
    eager, _, _ = run_attention(prob, tensors=(q, kc, vc, bt, sl))
    from tests.gpu_common import desc_for
    desc = desc_for(prob)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device="cuda")
    out = torch.zeros((1, 24, 256), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pa.paged_attention_decode(q, kc, vc, bt, sl, desc, out, ws)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.paged_attention_decode(q, kc, vc, bt, sl, desc, out, ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), eager)


# -- full-size workloads, benchmark launch configuration -------------------------

def test_hybrid_step_l32768_bs784_x16_layers(oracle_mod):
    spec = dict(WORKLOADS["hybrid_step_l32768_bs784_x16"])
    prob = make_problem(1002, **spec)
    for layer in (0, 15):
        out, status, plan = run_attention(prob, layer)
        assert status == 0 and plan["num_splits"] > 1
        assert_parity(out, oracle_out(oracle_mod, prob, layer), what=f"32K layer {layer}")


@pytest.mark.parametrize("depth", SWEEP_DEPTHS)
@pytest.mark.parametrize("dense", [False, True])
def test_context_sweep_depths(oracle_mod, depth, dense):
    """Every depth of the context sweep, both shapes, in the benchmark's plan."""
    prob = make_problem(1003 + depth + dense, **sweep_workload(depth, dense, num_layers=1))
    out, status, _ = run_attention(prob)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), what=f"sweep depth={depth} dense={dense}")


def test_batch32_uniform_bs784_sampled(oracle_mod):
    prob = make_problem(1004, **WORKLOADS["batch32_uniform_bs784"], device="cuda")
    out, status, _ = run_attention(prob)
    assert status == 0
    rows = [0, 5, 11, 17, 26, 31]
    ref = oracle_out(oracle_mod, prob, rows=rows)
    assert_parity(out[rows], ref, what="batch 32 sampled sequences")


# -- verify ----------------------------------------------------------------------

def write_new_rows(prob, seed):
    """reshape_and_cache of the q_len newest tokens of every sequence (GPU),
    checked bit for bit against the oracle's scatter before the oracle and
    the kernels read the cache."""
    import oracle
    k_new, v_new = make_new_tokens(seed, prob.num_seqs * prob.q_len, prob.num_kv_heads, prob.head_dim)
    slots = prob.new_token_slots()
    kc, vc = prob.k_cache[0].cuda(), prob.v_cache[0].cuda()
    pa.reshape_and_cache(k_new.cuda(), v_new.cuda(), kc, vc, slots.cuda())
    torch.cuda.synchronize()
    assert_cache_written(oracle, prob.k_cache[0], prob.v_cache[0], k_new, v_new, slots, kc, vc)
    prob.k_cache[0], prob.v_cache[0] = kc.cpu(), vc.cpu()


@pytest.mark.parametrize("q_len,lens,bs", [(2, [2, 33, 900], 16), (5, [5, 64, 785], 784),
                                           (16, [16, 17, 831, 1700], 832), (16, [3000], 16)])
def test_verify_small(oracle_mod, q_len, lens, bs):
    prob = hybrid(111 + q_len, lens, bs, q_len=q_len, poison_unused=True)
    write_new_rows(prob, 5)
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what=f"verify q_len={q_len}")


@pytest.mark.parametrize("splits", [2, 5, 13, 40])
def test_verify_forced_splits_tiles_cross_split_ends(oracle_mod, splits):
    """Split sizes that are not whole 64-token tiles: a tile reaches into the
    next split's tokens, which must be masked out (and the ends zero-filled)."""
    prob = hybrid(141 + splits, [1700, 900, 37], 784, q_len=16, poison_unused=True)
    write_new_rows(prob, 11)
    out, status, plan = run_attention(prob, num_splits=splits)
    assert status == 0 and plan["num_splits"] > 1
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what=f"verify splits={splits}")


@pytest.mark.parametrize("splits", [1, 3])
def test_verify_dense_shape_d128(oracle_mod, splits):
    prob = make_problem(121, num_seqs=2, seq_lens=[300, 77], num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, q_len=8, scale=1 / math.sqrt(128))
    out, status, _ = run_attention(prob, num_splits=splits)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what="verify d128")


@pytest.mark.parametrize("q_len,lens,bs,splits", [(48, [1000, 48], 784, 0), (48, [1000, 300], 16, 3),
                                                  (512, [2048], 832, 0), (200, [200, 1500], 784, 0)])
def test_verify_row_blocks(oracle_mod, q_len, lens, bs, splits):
    """More than 128 rows (q_len x 6 heads): blocks of 128 rows, the last one
    partial, each reading only the keys its rows can see (chunked prefill)."""
    prob = hybrid(151 + q_len, lens, bs, q_len=q_len, poison_unused=True)
    write_new_rows(prob, 13)
    out, status, plan = run_attention(prob, num_splits=splits)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what=f"verify rows q_len={q_len}")


@pytest.mark.parametrize("q_len", [5, 16])
def test_verify_wide_group_g12(oracle_mod, q_len):
    """12 query heads per KV head: 60 or 192 rows per (sequence, KV head)."""
    prob = hybrid(171 + q_len, [q_len, 900, 2000], 784, q_len=q_len, num_q_heads=48, num_kv_heads=4,
                  poison_unused=True)
    write_new_rows(prob, 19)
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what=f"verify G=12 q_len={q_len}")


def test_verify_row_blocks_d128(oracle_mod):
    prob = make_problem(161, num_seqs=1, seq_lens=[900], num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, q_len=300, scale=1 / math.sqrt(128), poison_unused=True)
    write_new_rows(prob, 17)
    out, status, _ = run_attention(prob)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what="verify rows d128")


def test_verify_short_context_sets_status():
    prob = hybrid(131, [40, 40], 16, q_len=16)
    q, kc, vc, bt, sl = to_dev(prob)
    sl[0] = 10  # fewer cached tokens than new rows
    out, status, _ = run_attention(prob, tensors=(q, kc, vc, bt, sl))
    assert status & pa.PA_DEV_BAD_SEQLEN
    assert torch.all(out[:16] == 0) and torch.all(torch.isfinite(out))


def test_verify_b8_q16_l8192_bs832_workload(oracle_mod):
    prob = make_problem(1005, **WORKLOADS["verify_b8_q16_l8192_bs832"])
    write_new_rows(prob, 9)
    out, status, plan = run_attention(prob)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob), rel_l2=REL_L2_VERIFY, what="verify workload")


def test_verify_g12_b32_q5_l2048_bs784_sampled(oracle_mod):
    """The wide-group verify workload in its benchmark launch: every sequence
    checked for finiteness and agreement with the dense reference on the
    first and last, the oracle on four sampled sequences."""
    prob = make_problem(1005, **WORKLOADS["verify_g12_b32_q5_l2048_bs784"])
    write_new_rows(prob, 23)
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05
    assert torch.isfinite(out).all()
    rows = [0, 9, 22, 31]
    sel = torch.cat([torch.arange(b * 5, (b + 1) * 5) for b in rows])
    assert_parity(out[sel], oracle_out(oracle_mod, prob, rows=rows), rel_l2=REL_L2_VERIFY,
                  what="verify G=12 workload")


# -- reshape_and_cache ----------------------------------------------------------------

def test_reshape_and_cache_bit_exact(oracle_mod):
    gen = torch.Generator().manual_seed(3)
    P, bs, hkv, d = 8, 784, 4, 256
    kc = torch.randn((P, bs, hkv, d), generator=gen).to(torch.bfloat16)
    vc = torch.randn((P, bs, hkv, d), generator=gen).to(torch.bfloat16)
    n = 300
    k_new, v_new = make_new_tokens(4, n, hkv, d)
    slots = torch.randperm(P * bs, generator=gen)[:n].to(torch.int64)
    slots[::17] = -1  # padding tokens
    kd, vd = kc.cuda(), vc.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.reshape_and_cache(k_new.cuda(), v_new.cuda(), kd, vd, slots.cuda(), status=status)
    torch.cuda.synchronize()
    k_ref, v_ref = bits(kc).copy(), bits(vc).copy()
    oracle_mod.reshape_and_cache(bits(k_new), bits(v_new), k_ref, v_ref, slots.numpy())
    assert status.item() == 0
    assert np.array_equal(bits(kd), k_ref) and np.array_equal(bits(vd), v_ref)


def test_reshape_and_cache_bad_slot_flagged():
    kc = torch.zeros((2, 16, 4, 256), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k_new, v_new = make_new_tokens(5, 2, 4, 256)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.reshape_and_cache(k_new.cuda(), v_new.cuda(), kc, vc, torch.tensor([3, 32], device="cuda"), status=status)
    torch.cuda.synchronize()
    assert status.item() & pa.PA_DEV_BAD_SLOT
    assert torch.equal(kc[0, 3].cpu(), k_new[0]) and torch.count_nonzero(kc[1]) == 0


# -- limits --------------------------------------------------------------------------

@pytest.mark.parametrize("splits,window", [(1, 0), (2, 0), (1, 7000)])
def test_decode_split_wider_than_staged_page_table(oracle_mod, splits, window):
    """A split spanning more than the 512 block-table entries a CTA stages in
    shared memory (16-token pages, 9000 tokens in one or two splits): the
    producer reads the table from global memory instead."""
    prob = hybrid(271 + splits, [9000, 100], 16, poison_unused=True)
    out, status, plan = run_attention(prob, num_splits=splits, window=window)
    assert status == 0 and plan["num_splits"] == splits
    assert_parity(out, oracle_out(oracle_mod, prob, window=window), what=f"unstaged splits={splits} W={window}")


def test_verify_maximum_rows_sampled(oracle_mod):
    """q_len x G = 8192 x 4 = 32768 rows per KV head, the largest verify block
    set (256 row blocks x 8 KV heads): sampled (row, head) outputs against the
    oracle's single-split attention, the rest checked finite."""
    q_len = 8192
    prob = make_problem(181, num_seqs=1, seq_lens=[q_len + 600], num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, q_len=q_len, scale=1 / math.sqrt(128), poison_unused=True)
    write_new_rows(prob, 29)
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05
    assert torch.isfinite(out).all()
    g = torch.Generator().manual_seed(3)
    rows = [0, 1, 127, 128, 4095, q_len - 1] + torch.randint(0, q_len, (10,), generator=g).tolist()
    heads = [0, 3, 4, 31]
    q, kc, vc = bits(prob.q[0]), bits(prob.k_cache[0]), bits(prob.v_cache[0])
    got, ref = [], []
    for r in rows:
        for h in heads:
            o, _, _ = oracle_mod.attention_partial(q, kc, vc, prob.block_table.numpy(), prob.seq_lens.numpy(),
                                                   prob.scale, r, h, 0, 1 << 40, q_len=q_len)
            got.append(out[r, h])
            ref.append(o)
    assert_parity(torch.stack(got)[:, None, :], np.stack(ref)[:, None, :], rel_l2=REL_L2_VERIFY,
                  what="verify 32768 rows (sampled)")



def test_verify_maximum_rows_sampled_d256(oracle_mod):
    """q_len x G = 4096 x 8 = 32768 rows per KV head at head_dim 256: the
    largest block set of the 128-key score tiles (256 row blocks x 4 KV
    heads), sampled against the oracle, the rest checked finite."""
    q_len = 4096
    prob = make_problem(191, num_seqs=1, seq_lens=[q_len + 700], num_q_heads=32, num_kv_heads=4, head_dim=256,
                        block_size=832, q_len=q_len, scale=1 / 16, poison_unused=True)
    write_new_rows(prob, 31)
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05
    assert torch.isfinite(out).all()
    g = torch.Generator().manual_seed(5)
    rows = [0, 1, 15, 16, 2047, q_len - 1] + torch.randint(0, q_len, (10,), generator=g).tolist()
    heads = [0, 7, 8, 31]
    q, kc, vc = bits(prob.q[0]), bits(prob.k_cache[0]), bits(prob.v_cache[0])
    got, ref = [], []
    for r in rows:
        for h in heads:
            o, _, _ = oracle_mod.attention_partial(q, kc, vc, prob.block_table.numpy(), prob.seq_lens.numpy(),
                                                   prob.scale, r, h, 0, 1 << 40, q_len=q_len)
            got.append(out[r, h])
            ref.append(o)
    assert_parity(torch.stack(got)[:, None, :], np.stack(ref)[:, None, :], rel_l2=REL_L2_VERIFY,
                  what="verify 32768 rows d256 (sampled)")

# -- the other benchmarked workloads at full size, in their benchmark launch ---------

def test_decode_window2048_l32768_bs784_workload(oracle_mod):
    """The 32K hybrid layer with a 2048-key window (the benchmark's window line)."""
    prob = make_problem(1007, **dict(WORKLOADS["hybrid_step_l32768_bs784_x16"], num_layers=1))
    out, status, plan = run_attention(prob, window=2048)
    assert status == 0
    assert_parity(out, oracle_out(oracle_mod, prob, window=2048), what="window 2048 at 32K")


def test_decode_g12_l32768_bs784_workload(oracle_mod):
    prob = make_problem(1008, **dict(WORKLOADS["decode_g12_l32768_bs784"], num_layers=1))
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["num_splits"] > 1
    assert_parity(out, oracle_out(oracle_mod, prob), what="G=12 at 32K")


def test_decode_dense_l32768_bs16_workload(oracle_mod):
    """The dense control at 32K (8 KV heads of 128 dims over 2048 pages of 16
    tokens), in its benchmark launch: a producer lane per chunk stream."""
    prob = make_problem(1011, **dict(WORKLOADS["decode_dense_l32768_bs16"], num_layers=1))
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["num_splits"] > 1
    assert_parity(out, oracle_out(oracle_mod, prob), what="dense 32/8/128 at 32K")


def test_prefill_q2048_l16384_bs832_workload_sampled(oracle_mod):
    """The chunked-prefill step (2048 new rows over 14336 cached tokens) in its
    benchmark launch: every output finite; sampled (row, head) outputs against
    the oracle's attention of that row, including the first and last rows of
    row blocks and of the step."""
    prob = make_problem(1006, **WORKLOADS["prefill_q2048_l16384_bs832"])
    out, status, plan = run_attention(prob)
    assert status == 0 and plan["path_id"] == pa.PA_PATH_VERIFY_TCGEN05
    assert torch.isfinite(out).all()
    q, kc, vc = bits(prob.q[0]), bits(prob.k_cache[0]), bits(prob.v_cache[0])
    g = torch.Generator().manual_seed(11)
    rows = [0, 20, 21, 1023, 2047] + torch.randint(0, 2048, (6,), generator=g).tolist()
    heads = [0, 5, 6, 23]
    got, ref = [], []
    for r in rows:
        for h in heads:
            o, _, _ = oracle_mod.attention_partial(q, kc, vc, prob.block_table.numpy(), prob.seq_lens.numpy(),
                                                   prob.scale, r, h, 0, 1 << 40, q_len=prob.q_len)
            got.append(out[r, h])
            ref.append(o)
    assert_parity(torch.stack(got)[:, None, :], np.stack(ref)[:, None, :], rel_l2=REL_L2_VERIFY,
                  what="prefill 2048 rows (sampled)")
