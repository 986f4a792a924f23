"""Randomised parity: many small problems drawn from one seed, each through the
C ABI against the oracle -- group sizes, head dims, page sizes, ragged and
empty lengths, q_len (decode and verify), sliding windows, forced split
counts, the early-K/V flag and the fp8 cache all vary together, so that
combinations the targeted tests do not name are covered too."""
import math
import random

import pytest
import torch

import paged_attention_decode_split_gb300 as pa
from paged_attention_decode_split_gb300 import _build
from paged_attention_decode_split_gb300.inputs import make_problem
from tests.gpu_common import REL_L2_VERIFY, assert_parity, oracle_out, run_attention

pytestmark = pytest.mark.gpu

DECODE_GROUPS = {256: [1, 2, 3, 4, 5, 6, 8, 12, 16], 128: [1, 2, 3, 4, 5, 6, 8, 12, 16]}
N_CASES = 120


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    pa.load_library()


def draw_case(i):
    r = random.Random(7000 + i)
    d = r.choice([128, 256])
    g = r.choice(DECODE_GROUPS[d])
    hkv = r.choice([1, 2, 4]) if g * 4 <= 64 else r.choice([1, 2])
    bs = r.choice([16, 32, 48, 64, 784, 832])
    q_len = 1 if r.random() < 0.55 else r.choice([2, 3, 5, 8, 16, 23])
    b = r.randint(1, 4)
    lens = []
    for _ in range(b):
        kind = r.random()
        if kind < 0.1 and q_len == 1:
            lens.append(0)
        elif kind < 0.3:
            lens.append(max(q_len, r.randint(1, 40)))
        else:
            lens.append(max(q_len, r.randint(1, 3000)))
    window = 0 if r.random() < 0.6 else r.randint(1, 1500)
    splits = 0 if r.random() < 0.5 else r.randint(1, 20)
    flags = pa.PA_FLAG_EARLY_KV_READ if r.random() < 0.3 else 0
    fp8 = r.random() < 0.3
    return dict(d=d, g=g, hkv=hkv, bs=bs, q_len=q_len, lens=lens, window=window, splits=splits, flags=flags, fp8=fp8)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(oracle_mod, i):
    c = draw_case(i)
    prob = make_problem(8000 + i, num_seqs=len(c["lens"]), seq_lens=c["lens"], num_q_heads=c["g"] * c["hkv"],
                        num_kv_heads=c["hkv"], head_dim=c["d"], block_size=c["bs"], q_len=c["q_len"],
                        scale=1 / math.sqrt(c["d"]), poison_unused=True, kv_fp8=c["fp8"])
    out, status, plan = run_attention(prob, num_splits=c["splits"], window=c["window"], flags=c["flags"])
    assert status == 0, c
    want = pa.PA_PATH_DECODE_MMA if c["q_len"] == 1 else pa.PA_PATH_VERIFY_TCGEN05
    assert plan["path_id"] == want, c
    assert_parity(out, oracle_out(oracle_mod, prob, window=c["window"]), rel_l2=REL_L2_VERIFY, what=str(c))
