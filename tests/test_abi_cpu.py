"""Host-only checks of the C ABI: the library loads, exports what the header
declares, plans deterministically, and rejects bad arguments before touching
a GPU.  No test here launches a kernel or passes a pointer that could be
dereferenced."""
import ctypes
import os
import re

import pytest

import paged_attention_decode_split_gb300 as pa
from paged_attention_decode_split_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pagedattn.h")
FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pa.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(pa_\w+)\s*\(", text, flags=re.M)))


def test_header_symbols_exported(lib):
    names = declared_functions()
    assert {"pa_reshape_and_cache", "pa_paged_attention_decode", "pa_paged_attention_verify",
            "pa_workspace_bytes", "pa_status_string", "pa_last_plan"} <= set(names)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in pagedattn.h but not exported"


def test_header_is_plain_c_and_links(lib, tmp_path):
    """The header compiles as C99 with warnings as errors, and a C program that
    takes the address of every declared entry point links against the library
    and runs (no entry point is called)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "abi.c"
    src.write_text('#include "pagedattn.h"\n#include <stdio.h>\n'
                   "int main(void) {\n"
                   "    void (*const fns[])(void) = {" + ", ".join(f"(void (*)(void)){n}" for n in names) + "};\n"
                   '    printf("%d\\n", (int)(sizeof(fns) / sizeof(fns[0])));\n'
                   "    return 0;\n}\n")
    exe = tmp_path / "abi"
    build_dir = os.path.dirname(_build.LIB)
    res = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.dirname(HEADER), str(src),
                          "-L", build_dir, "-lpagedattn", f"-Wl,-rpath,{build_dir}", "-o", str(exe)],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0 and run.stdout.strip() == str(len(names)), run.stderr


def test_status_strings(lib):
    for code in range(5):
        assert pa.status_string(code).startswith("PA_")
    assert "unknown" in pa.status_string(99)


def hybrid_desc(**kw):
    base = dict(num_seqs=1, num_q_heads=24, num_kv_heads=4, head_dim=256, block_size=784,
                max_pages_per_seq=42, max_seq_len=32768, num_pages=46, scale=1 / 16, num_sms=152)
    base.update(kw)
    return pa.make_desc(**base)


def test_workspace_plan_hybrid_32k(lib):
    # 2048 chunks of 16 tokens, 4 (seq, kv-head) units, 152 SMs -> 38 splits of 54 chunks
    ws = pa.workspace_bytes(hybrid_desc())
    splits, rows = 38, 24
    part_o = (rows * splits * 256 * 4 + 255) // 256 * 256
    assert ws == part_o + rows * splits * 8


def test_workspace_plan_rules(lib):
    assert pa.workspace_bytes(hybrid_desc(num_splits=1)) == 0
    assert pa.workspace_bytes(hybrid_desc(num_splits=5)) == 24 * 5 * 256 * 4 + 24 * 5 * 8
    # a 512-token context (32 chunks) never splits below 4 chunks per split: 8 splits
    small = hybrid_desc(block_size=16, max_pages_per_seq=32, max_seq_len=512, num_pages=64)
    assert pa.workspace_bytes(small) == 24 * 8 * 256 * 4 + 24 * 8 * 8
    # the plan depends only on the description
    assert pa.workspace_bytes(hybrid_desc()) == pa.workspace_bytes(hybrid_desc())
    # empty context / empty batch: nothing to split
    assert pa.workspace_bytes(hybrid_desc(max_seq_len=0)) == 0
    assert pa.workspace_bytes(hybrid_desc(num_seqs=0)) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(num_q_heads=25), pa.PA_ERR_INVALID_ARG),       # Hq % Hkv != 0
    (dict(head_dim=64), pa.PA_ERR_UNSUPPORTED),
    (dict(block_size=20, max_pages_per_seq=2000), pa.PA_ERR_UNSUPPORTED),  # not a multiple of 16
    (dict(block_size=0), pa.PA_ERR_INVALID_ARG),
    (dict(max_pages_per_seq=10), pa.PA_ERR_INVALID_ARG),   # table too narrow for max_seq_len
    (dict(num_pages=0), pa.PA_ERR_INVALID_ARG),
    (dict(num_seqs=-1), pa.PA_ERR_INVALID_ARG),
    (dict(out_dtype=7), pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), pa.PA_ERR_INVALID_ARG),
    (dict(q_len=2), pa.PA_ERR_INVALID_ARG),              # decode takes one row per sequence
    (dict(num_q_heads=40, num_kv_heads=4), pa.PA_ERR_UNSUPPORTED),  # G = 10 not compiled
    (dict(flags=2), pa.PA_ERR_INVALID_ARG),               # unknown flag bit
])
def test_decode_rejects_bad_descriptions(lib, kw, code):
    desc = hybrid_desc(**kw)
    rc = lib.pa_paged_attention_decode(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(desc), FAKE, FAKE, 1 << 30,
                                       None, None)
    assert rc == code


def test_decode_rejects_bad_pointers_and_workspace(lib):
    desc = hybrid_desc()
    call = lib.pa_paged_attention_decode
    assert call(None, FAKE, FAKE, FAKE, FAKE, ctypes.byref(desc), FAKE, FAKE, 1 << 30, None, None) == pa.PA_ERR_INVALID_ARG
    assert call(FAKE + 8, FAKE, FAKE, FAKE, FAKE, ctypes.byref(desc), FAKE, FAKE, 1 << 30, None, None) == pa.PA_ERR_INVALID_ARG
    assert call(FAKE, FAKE, FAKE, FAKE + 2, FAKE, ctypes.byref(desc), FAKE, FAKE, 1 << 30, None, None) == pa.PA_ERR_INVALID_ARG
    need = pa.workspace_bytes(desc)
    assert call(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(desc), FAKE, FAKE, need - 1, None, None) == pa.PA_ERR_WORKSPACE
    assert call(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(desc), FAKE, None, need, None, None) == pa.PA_ERR_WORKSPACE
    assert call(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, need, None, None) == pa.PA_ERR_INVALID_ARG


def test_plan_info_layout_matches_header(lib):
    text = open(HEADER).read()
    body = text[text.index("typedef struct {", text.index("What the last successful")):text.index("} pa_plan_info;")]
    fields = re.findall(r"^\s*int32_t\s+(\w+);", body, flags=re.M)
    assert fields == [name for name, _ in pa.PlanInfo._fields_]


def test_desc_layout_matches_header(lib):
    # the binding's mirror of pa_attn_desc: same fields, same order, 64 bytes
    text = open(HEADER).read()
    body = text[text.index("typedef struct {", text.index("Shape and launch description")):text.index("} pa_attn_desc;")]
    fields = re.findall(r"^\s*(?:int32_t|int64_t|float)\s+(\w+);", body, flags=re.M)
    assert fields == [name for name, _ in pa.AttnDesc._fields_]
    assert ctypes.sizeof(pa.AttnDesc) == 64


def test_early_kv_flag_accepted(lib):
    desc = hybrid_desc(flags=pa.PA_FLAG_EARLY_KV_READ)
    assert pa.workspace_bytes(desc) == pa.workspace_bytes(hybrid_desc())


def test_empty_batch_is_a_noop(lib):
    desc = hybrid_desc(num_seqs=0)
    assert lib.pa_paged_attention_decode(None, None, None, None, None, ctypes.byref(desc), None, None, 0,
                                         None, None) == pa.PA_OK


def test_verify_row_blocks_plan(lib):
    # 2048 rows x 6 heads = 96 blocks of 128 rows per KV head: 384 CTAs fill the
    # SMs without splitting the context, so no workspace is needed
    prefill = hybrid_desc(q_len=2048, block_size=832, max_pages_per_seq=20, max_seq_len=16384, num_pages=22)
    assert pa.workspace_bytes(prefill) == 0
    # a 16-row verify of 8 sequences splits each (sequence, KV head) context 4 ways
    small = hybrid_desc(num_seqs=8, q_len=16, block_size=832, max_pages_per_seq=10, max_seq_len=8208, num_pages=88)
    assert pa.workspace_bytes(small) == ((8 * 16 * 24 * 4 * 256 * 4 + 255) // 256 * 256) + 8 * 16 * 24 * 4 * 8


def test_verify_rejects_bad_descriptions(lib):
    call = lib.pa_paged_attention_verify
    too_many_rows = hybrid_desc(q_len=8192, max_seq_len=16384, max_pages_per_seq=21, num_pages=22)  # 49152 rows
    assert call(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(too_many_rows), FAKE, FAKE, 1 << 30, None,
                None) == pa.PA_ERR_UNSUPPORTED
    bad_dim = hybrid_desc(q_len=16, head_dim=96)
    assert call(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(bad_dim), FAKE, FAKE, 1 << 30, None,
                None) == pa.PA_ERR_UNSUPPORTED


def test_reshape_and_cache_rejects_bad_arguments(lib):
    call = lib.pa_reshape_and_cache
    assert call(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 4, 256, 16, 10, None, None) == pa.PA_ERR_INVALID_ARG
    assert call(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 256, 16, 10, None, None) == pa.PA_ERR_INVALID_ARG
    assert call(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 4, 16, 10, None, None) == pa.PA_ERR_UNSUPPORTED  # 8-byte rows
    assert call(FAKE + 4, FAKE, FAKE, FAKE, FAKE, 1, 4, 256, 16, 10, None, None) == pa.PA_ERR_INVALID_ARG
    assert call(None, None, None, None, None, 0, 4, 256, 16, 10, None, None) == pa.PA_OK  # nothing to copy


def test_last_plan_before_any_call(lib):
    info = pa.PlanInfo()
    # this process has made no successful attention call on this thread
    assert lib.pa_last_plan(ctypes.byref(info)) == pa.PA_ERR_INVALID_ARG


def test_hybrid_page_tokens_matches_oracle(lib, oracle_mod):
    """Host page-size helper against the oracle's rule on a grid of shapes."""
    for align in (1, 16, 64, 128):
        for per_token in (1, 3, 4096, 2 * 8 * 128 * 2):
            for state in (1, per_token - 1, per_token, 64 * per_token + 1, 781 * per_token, 3 << 20, (1 << 40) + 5):
                if state <= 0:
                    continue
                assert lib.pa_hybrid_page_tokens(state, per_token, align) == \
                    oracle_mod.hybrid_page_tokens(state, per_token, align), (state, per_token, align)
    assert pa.hybrid_page_tokens(780 * 4096, 4096, 16) == 784
    assert pa.hybrid_page_tokens(780 * 4096, 4096, 64) == 832
    for bad in ((0, 4096, 16), (100, -1, 16), (100, 4096, 0)):
        assert lib.pa_hybrid_page_tokens(*bad) == -1
        with pytest.raises(pa.PagedAttnError):
            pa.hybrid_page_tokens(*bad)
    # a group larger than any state page: one group; a page past int64: -1
    assert lib.pa_hybrid_page_tokens(5, 1 << 62, 64) == 64
    assert lib.pa_hybrid_page_tokens((1 << 63) - 1, 1, 1 << 30) == -1


def test_fp8_entries_reject_bad_arguments(lib):
    dec = lib.pa_paged_attention_decode_fp8
    desc = hybrid_desc()
    args = lambda ks, vs, d: (FAKE, FAKE, FAKE, ks, vs, FAKE, FAKE, ctypes.byref(d), FAKE, FAKE, 1 << 30, None, None)
    assert dec(*args(None, FAKE, desc)) == pa.PA_ERR_INVALID_ARG       # scales are required
    assert dec(*args(FAKE, None, desc)) == pa.PA_ERR_INVALID_ARG
    assert dec(*args(FAKE + 2, FAKE, desc)) == pa.PA_ERR_INVALID_ARG   # misaligned float
    assert dec(*args(FAKE, FAKE, hybrid_desc(num_q_heads=40))) == pa.PA_ERR_UNSUPPORTED  # G = 10
    assert dec(*args(FAKE, FAKE, hybrid_desc(flags=2))) == pa.PA_ERR_INVALID_ARG
    rc = lib.pa_reshape_and_cache_fp8
    assert rc(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1, 4, 256, 16, 10, None, None) == pa.PA_ERR_INVALID_ARG
    assert rc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 12, 16, 10, None, None) == pa.PA_ERR_UNSUPPORTED
    assert rc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1, 4, 256, 16, 10, None, None) == pa.PA_ERR_INVALID_ARG
    assert rc(None, None, None, None, None, None, None, 0, 4, 256, 16, 10, None, None) == pa.PA_OK


def test_verify_plan_stays_at_whole_waves(lib):
    """Verify grids stay within whole waves of 152 CTAs even for long contexts
    (the decode-only rule that cuts splits to at most 256 chunks is not applied):
    8 x 8 units of the 32/8/128 shape at 8208 tokens take 2 splits (128 CTAs)."""
    dense = hybrid_desc(num_seqs=8, q_len=16, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=784,
                        max_pages_per_seq=11, max_seq_len=8208, num_pages=100)
    rows = 8 * 16 * 32
    assert pa.workspace_bytes(dense) == ((rows * 2 * 128 * 4 + 255) // 256 * 256) + rows * 2 * 8
    # decode of the same context keeps the rule: 8 x 8 units, 513 chunks -> 3 splits
    dec = hybrid_desc(num_seqs=8, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=784,
                      max_pages_per_seq=11, max_seq_len=8208, num_pages=100)
    assert pa.workspace_bytes(dec) == ((8 * 32 * 3 * 128 * 4 + 255) // 256 * 256) + 8 * 32 * 3 * 8


def test_noalloc_rejects_on_the_host(lib):
    """The no-allocation decode answers like the ordinary decode for a
    description that decode rejects (a verify-shaped q_len among them), and
    rejects a plan larger than its built-in scratch, before touching a device."""
    fn = lib.pa_paged_attention_decode_noalloc
    fn.restype = ctypes.c_int
    vp = ctypes.c_void_p
    fn.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(pa.AttnDesc), vp, vp, vp]
    verify_shaped = hybrid_desc(q_len=16)
    # its verify plan alone would be larger than the scratch; q_len is still what decides
    assert pa.workspace_bytes(verify_shaped) > pa.PA_NOALLOC_SCRATCH_BYTES
    assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(verify_shaped), FAKE, None, None) == pa.PA_ERR_INVALID_ARG
    bad = hybrid_desc(num_q_heads=25)
    assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(bad), FAKE, None, None) == pa.PA_ERR_INVALID_ARG
    big = pa.make_desc(num_seqs=64, num_q_heads=24, num_kv_heads=4, head_dim=256, block_size=784,
                       max_pages_per_seq=42, max_seq_len=32768, num_pages=64 * 42, scale=1 / 16, num_splits=64,
                       num_sms=152)
    assert pa.workspace_bytes(big) > pa.PA_NOALLOC_SCRATCH_BYTES
    assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(big), FAKE, None, None) == pa.PA_ERR_WORKSPACE


def test_binding_checks_tensors_before_calling(lib):
    """The C ABI cannot see a buffer's size, so the binding checks element
    types and shapes against the description first: a uint8 (e4m3) cache handed
    to a bf16 entry point, a cache of another geometry, or a host tensor is
    refused with ValueError before anything is launched."""
    import torch
    desc = hybrid_desc(block_size=16, max_pages_per_seq=4, max_seq_len=64, num_pages=8)
    q = torch.zeros((1, 24, 256), dtype=torch.bfloat16)
    cache = torch.zeros((8, 16, 4, 256), dtype=torch.bfloat16)
    codes = torch.zeros((8, 16, 4, 256), dtype=torch.uint8)
    bt = torch.zeros((1, 4), dtype=torch.int32)
    sl = torch.zeros((1,), dtype=torch.int32)
    out = torch.zeros((1, 24, 256), dtype=torch.float32)
    cases = [
        (dict(k_cache=codes, v_cache=codes), "k_cache: dtype"),  # fp8 codes in a bf16 call
        (dict(k_cache=torch.zeros((8, 16, 4, 128), dtype=torch.bfloat16)), "k_cache: shape"),  # another head_dim
        (dict(q=torch.zeros((2, 24, 256), dtype=torch.bfloat16)), "q: shape"),  # more rows than the description
        (dict(out=torch.zeros((1, 24, 256), dtype=torch.bfloat16)), "out: dtype"),  # bf16 out, fp32 description
        (dict(block_table=torch.zeros((1, 4), dtype=torch.int64)), "block_table: dtype"),
        (dict(seq_lens=torch.zeros((2,), dtype=torch.int32)), "seq_lens: shape"),
        (dict(status=torch.zeros((1,), dtype=torch.int64)), "status: dtype"),
        (dict(), "q: a CUDA tensor is required"),  # right types and shapes, but host tensors
    ]
    for bad, msg in cases:
        args = dict(q=q, k_cache=cache, v_cache=cache, block_table=bt, seq_lens=sl, out=out, status=None)
        args.update(bad)
        with pytest.raises(ValueError, match=msg):
            pa.paged_attention_decode(args["q"], args["k_cache"], args["v_cache"], args["block_table"],
                                      args["seq_lens"], desc, args["out"], status=args["status"])
    # every entry point checks before it calls
    k_new = torch.zeros((1, 4, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="k_new: shape"):
        pa.paged_attention_decode_append(q, k_new[:, :2], k_new, cache, cache, bt, sl, desc, out)
    with pytest.raises(ValueError, match="v_cache: dtype"):
        pa.paged_attention_verify(q, cache, codes, bt, sl, desc, out)
    with pytest.raises(ValueError, match="out: shape"):
        pa.paged_attention_decode_noalloc(q, cache, cache, bt, sl, desc, out[:, :12])
    # the fp8 entry points refuse a bf16 cache and wrongly shaped or missing scales
    scales = torch.ones((4,), dtype=torch.float32)
    with pytest.raises(ValueError, match="k_cache: dtype"):
        pa.paged_attention_decode_fp8(q, cache, cache, scales, scales, bt, sl, desc, out)
    with pytest.raises(ValueError, match="k_scale: shape"):
        pa.paged_attention_decode_fp8(q, codes, codes, torch.ones((3,)), scales, bt, sl, desc, out)
    with pytest.raises(ValueError, match="v_scale"):
        pa.paged_attention_verify_fp8(q, codes, codes, scales, None, bt, sl, desc, out)
    with pytest.raises(ValueError, match="k_new: dtype"):
        pa.paged_attention_decode_append_fp8(q, k_new.float(), k_new, codes, codes, scales, scales, bt, sl, desc, out)
    # reshape_and_cache: the new rows must match the cache's heads and dims
    slots = torch.zeros((2,), dtype=torch.int64)
    with pytest.raises(ValueError, match="k_new: shape"):
        pa.reshape_and_cache(torch.zeros((2, 4, 128), dtype=torch.bfloat16),
                             torch.zeros((2, 4, 128), dtype=torch.bfloat16), cache, cache, slots)
    rows = torch.zeros((2, 4, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="slot_mapping: dtype"):
        pa.reshape_and_cache(rows, rows, cache, cache, slots.int())
    with pytest.raises(ValueError, match="k_cache: dtype"):
        pa.reshape_and_cache_fp8(rows, rows, cache, cache, slots, scales, scales)
    with pytest.raises(ValueError, match="k_new: a CUDA tensor is required"):
        pa.reshape_and_cache_fp8(rows, rows, codes, codes, slots, scales, scales)


def test_compiled_binding_knows_its_entry_points(lib):
    """The compiled module takes the C entry points by name from the loaded
    library; an unknown name is refused."""
    import paged_attention_decode_split_gb300 as pkg
    assert pkg._bind is not None
    with pytest.raises(ValueError):
        pkg._bind.set_entry("pa_no_such_entry", 0)
