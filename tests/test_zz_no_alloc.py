"""The decode entry point for callers that cannot allocate device memory.

pa_paged_attention_decode_noalloc serves callers -- such as a plugin inside a
serving engine that has claimed almost all of HBM for its own KV-cache pool --
that have no workspace buffer to pass.  It keeps the split partials in a fixed
scratch array inside the library.  These tests call it through the C ABI and
check its output against the ordinary pa_paged_attention_decode (which is
checked against the CPU oracle elsewhere) on two calls in a row, the second on a
different problem, so stale scratch contents from the first call would show up.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_attention_decode_split_gb300 as pa
from paged_attention_decode_split_gb300 import _build
from paged_attention_decode_split_gb300.inputs import make_problem
from tests.gpu_common import ATOL, REL_L2_DECODE, desc_for, run_attention, to_dev

pytestmark = pytest.mark.gpu

_vp = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    lib = pa.load_library()
    fn = lib.pa_paged_attention_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.POINTER(pa.AttnDesc), _vp, _vp, _vp]
    return lib


def run_noalloc(lib, prob):
    q, kc, vc, bt, sl = to_dev(prob)
    desc = desc_for(prob)
    out = torch.full((prob.num_seqs, prob.num_q_heads, prob.head_dim), float("nan"), dtype=torch.float32,
                     device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.pa_paged_attention_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
                                               sl.data_ptr(), ctypes.byref(desc), out.data_ptr(), status.data_ptr(),
                                               stream)
    torch.cuda.synchronize()
    return rc, out.cpu(), int(status.item())


def assert_close(got, ref, what):
    g, r = got.double().numpy(), ref.double().numpy()
    assert np.isfinite(g).all(), what
    assert np.abs(g - r).max() <= ATOL, what
    num = np.linalg.norm((g - r).reshape(-1, g.shape[-1]), axis=1)
    den = np.linalg.norm(r.reshape(-1, g.shape[-1]), axis=1)
    nz = den > 0
    assert (num[nz] / den[nz]).max(initial=0.0) <= REL_L2_DECODE, what
    assert np.all(g.reshape(-1, g.shape[-1])[~nz] == 0.0), what


def hybrid(seed, lens, bs):
    return make_problem(seed, num_seqs=len(lens), seq_lens=list(lens), num_q_heads=24, num_kv_heads=4,
                        head_dim=256, block_size=bs, scale=1 / 16, poison_unused=True)


def test_noalloc_matches_decode_on_two_calls_in_a_row(lib):
    first = hybrid(201, [32768], 784)          # 38 splits: the scratch is used
    second = hybrid(202, [5000, 333, 1, 0], 832)  # a different plan over the same scratch
    for prob in (first, second):
        ref, st_ref, _ = run_attention(prob)
        assert st_ref == 0
        rc, out, status = run_noalloc(lib, prob)
        assert rc == pa.PA_OK, pa.status_string(rc)
        assert status == 0
        assert_close(out, ref, f"no-alloc vs decode, lengths {prob.seq_lens.tolist()}")


def test_noalloc_rejects_plans_beyond_its_scratch(lib):
    # 64 sequences of 32K tokens forced into 64 splits need ~100 MB of partials
    desc = pa.make_desc(num_seqs=64, num_q_heads=24, num_kv_heads=4, head_dim=256, block_size=784,
                        max_pages_per_seq=42, max_seq_len=32768, num_pages=64 * 42, scale=1 / 16, num_splits=64)
    assert pa.workspace_bytes(desc) > 8 << 20
    fake = 0x10000  # never dereferenced: the size check comes first
    rc = lib.pa_paged_attention_decode_noalloc(fake, fake, fake, fake, fake, ctypes.byref(desc), fake, None, None)
    assert rc == pa.PA_ERR_WORKSPACE


def test_noalloc_through_the_binding(lib):
    prob = hybrid(97, [3000, 17], 784)
    rc, ref, status = run_noalloc(lib, prob)
    assert rc == pa.PA_OK and status == 0
    q, kc, vc, bt, sl = to_dev(prob)
    out = torch.full((prob.num_seqs, prob.num_q_heads, prob.head_dim), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.paged_attention_decode_noalloc(q, kc, vc, bt, sl, desc_for(prob), out, st)
    torch.cuda.synchronize()
    assert st.item() == 0 and torch.equal(out.cpu(), ref)
