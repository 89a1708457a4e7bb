"""The C ABI: libgqa.so loads, exports every entry point include/gqa.h
declares, and rejects bad arguments on the host before any CUDA call.
(No GPU needed: every call here fails validation before touching CUDA.)"""
import ctypes
import os
import re

import pytest

import gqa_attention_kv_split_gb300 as gqa
from gqa_attention_kv_split_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa.h")

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return gqa.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^(?:const\s+char\s*\*|gqa_status|int)\s+(\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"gqa_decode", "nvfp4_paged_ctx_attn", "gqa_debug_dequant_pages", "gqa_last_error",
            "gqa_check_device_errors", "gqa_release_workspace", "gqa_version", "gqa_decode_plan",
            "gqa_ctx_plan", "gqa_decode_paged"} <= names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"libgqa.so does not export {name}"
    assert L.gqa_version() >= 100


P = ctypes.c_void_p


def fake(addr=0x10000):
    return P(addr)


def test_decode_rejects_bad_sizes_and_nulls(L):
    s = P(0)
    assert L.gqa_decode(fake(), fake(), fake(), fake(), 0, 16, 1.0, s) == UNSUPPORTED
    assert b"batch" in L.gqa_last_error()
    assert L.gqa_decode(fake(), fake(), fake(), fake(), 70000, 16, 1.0, s) == UNSUPPORTED
    assert L.gqa_decode(fake(), fake(), fake(), fake(), 1, 0, 1.0, s) == UNSUPPORTED
    assert L.gqa_decode(fake(), fake(), fake(), fake(), 1, 16, float("nan"), s) == INVALID
    assert L.gqa_decode(fake(), fake(), fake(), fake(), 1, 16, float("inf"), s) == INVALID
    assert L.gqa_decode(P(0), fake(), fake(), fake(), 1, 16, 1.0, s) == INVALID
    assert b"q is a null pointer" in L.gqa_last_error()
    assert L.gqa_decode(fake(), fake(), P(0), fake(), 1, 16, 1.0, s) == INVALID
    assert b"seq_lens" in L.gqa_last_error()


def test_ctx_rejects_bad_sizes_and_nulls(L):
    s = P(0)
    f = fake()
    args = [f, 1.0, f, f, f, f, f, f, f, f, 1.0]
    assert L.nvfp4_paged_ctx_attn(*args, 0, 16, 4, 2, s) == UNSUPPORTED
    assert L.nvfp4_paged_ctx_attn(*args, 1, -1, 4, 2, s) == INVALID
    assert L.nvfp4_paged_ctx_attn(*args, 1, 16, 0, 2, s) == INVALID
    assert L.nvfp4_paged_ctx_attn(*args, 1, 16, 4, 0, s) == INVALID
    bad_out = [f, 1.0, f, f, f, f, f, f, f, f, 0.0]
    assert L.nvfp4_paged_ctx_attn(*bad_out, 1, 16, 4, 2, s) == INVALID
    assert b"out_scale" in L.gqa_last_error()
    nan_q = [f, float("nan"), f, f, f, f, f, f, f, f, 1.0]
    assert L.nvfp4_paged_ctx_attn(*nan_q, 1, 16, 4, 2, s) == INVALID
    null_kv = [f, 1.0, f, f, f, f, f, f, P(0), f, 1.0]
    assert L.nvfp4_paged_ctx_attn(*null_kv, 1, 16, 4, 2, s) == INVALID
    assert b"kv_lens" in L.gqa_last_error()


def test_paged_decode_rejects_bad_sizes_and_nulls(L):
    s = P(0)
    f = fake()
    # q, k_pages, v_pages, block_table, seq_lens, out, batch, num_pages, max_pages_per_seq, q_scale
    assert L.gqa_decode_paged(f, f, f, f, f, f, 0, 4, 2, 1.0, s) == UNSUPPORTED
    assert b"batch" in L.gqa_last_error()
    assert L.gqa_decode_paged(f, f, f, f, f, f, 70000, 4, 2, 1.0, s) == UNSUPPORTED
    assert L.gqa_decode_paged(f, f, f, f, f, f, 1, 0, 2, 1.0, s) == INVALID
    assert b"num_pages" in L.gqa_last_error()
    assert L.gqa_decode_paged(f, f, f, f, f, f, 1, 4, 0, 1.0, s) == INVALID
    assert L.gqa_decode_paged(f, f, f, f, f, f, 1, 4, 1 << 26, 1.0, s) == INVALID  # capacity past 2^31 - 1
    assert L.gqa_decode_paged(f, f, f, f, f, f, 1, 4, 2, float("nan"), s) == INVALID
    assert L.gqa_decode_paged(f, P(0), f, f, f, f, 1, 4, 2, 1.0, s) == INVALID
    assert b"k_pages is a null pointer" in L.gqa_last_error()
    assert L.gqa_decode_paged(f, f, f, P(0), f, f, 1, 4, 2, 1.0, s) == INVALID
    assert b"block_table" in L.gqa_last_error()


def test_dequant_rejects_bad_sizes(L):
    s = P(0)
    f = fake()
    assert L.gqa_debug_dequant_pages(f, f, f, f, f, 1, 4, 2, 129, s) == INVALID  # max_kv > 64 * pages
    assert L.gqa_debug_dequant_pages(f, f, f, f, f, 0, 4, 2, 64, s) == UNSUPPORTED
    assert L.gqa_debug_dequant_pages(f, f, P(0), f, f, 1, 4, 2, 64, s) == INVALID


def test_python_binding_raises_without_library(monkeypatch):
    monkeypatch.setattr(gqa, "_lib", None)
    monkeypatch.setattr(gqa, "LIB_PATH", "/nonexistent/libgqa.so")
    import torch
    with pytest.raises(RuntimeError, match="not built"):
        gqa.gqa_decode(torch.zeros(1, 32, 128, dtype=torch.float16),
                       torch.zeros(1, 2, 8, 4, 128, dtype=torch.float16),
                       torch.ones(1, dtype=torch.int32))


def test_descriptor_checks_shapes_dtypes_and_strides():
    """The *_t entry points check every descriptor in C before any CUDA call
    (so this runs without a GPU); the binding only marshals."""
    import torch
    with pytest.raises(gqa.GqaError, match="q has dtype f32; expected f16"):
        gqa.gqa_decode(torch.zeros(1, 32, 128), torch.zeros(1, 2, 8, 4, 128, dtype=torch.float16),
                       torch.ones(1, dtype=torch.int32))
    with pytest.raises(gqa.GqaError, match="UNSUPPORTED.*kv has extent 4 in dimension 2; expected 8"):
        gqa.gqa_decode(torch.zeros(1, 32, 128, dtype=torch.float16),
                       torch.zeros(1, 2, 4, 4, 128, dtype=torch.float16), torch.ones(1, dtype=torch.int32))
    with pytest.raises(gqa.GqaError, match="seq_lens has extent 2 in dimension 0; expected 1"):
        gqa.gqa_decode(torch.zeros(1, 32, 128, dtype=torch.float16),
                       torch.zeros(1, 2, 8, 4, 128, dtype=torch.float16), torch.ones(2, dtype=torch.int32))
    with pytest.raises(gqa.GqaError, match="kv is not dense row-major"):
        gqa.gqa_decode(torch.zeros(1, 32, 128, dtype=torch.float16),
                       torch.zeros(1, 2, 8, 8, 128, dtype=torch.float16)[:, :, :, ::2], torch.ones(1, dtype=torch.int32))


def test_descriptor_checks_paged_decode_arguments():
    import torch
    q = torch.zeros(1, 32, 128, dtype=torch.float16)
    pages = torch.zeros(3, 8, 64, 128, dtype=torch.float16)
    bt = torch.zeros(1, 2, dtype=torch.int32)
    lens = torch.ones(1, dtype=torch.int32)
    with pytest.raises(gqa.GqaError, match="k_pages has dtype f32"):   # pages must be fp16
        gqa.gqa_decode_paged(q, pages.float(), pages, bt, lens)
    with pytest.raises(gqa.GqaError, match="UNSUPPORTED"):  # 64-token pages of 8 heads
        gqa.gqa_decode_paged(q, torch.zeros(3, 8, 32, 128, dtype=torch.float16), pages, bt, lens)
    with pytest.raises(gqa.GqaError, match="v_pages has extent 2"):  # K and V pages alike
        gqa.gqa_decode_paged(q, pages, torch.zeros(2, 8, 64, 128, dtype=torch.float16), bt, lens)
    with pytest.raises(gqa.GqaError, match="block_table has extent 2 in dimension 0"):  # one row per sequence
        gqa.gqa_decode_paged(q, pages, pages, torch.zeros(2, 2, dtype=torch.int32), lens)
    with pytest.raises(gqa.GqaError, match="block_table has dtype unknown"):   # int32 table
        gqa.gqa_decode_paged(q, pages, pages, bt.long(), lens)
    with pytest.raises(gqa.GqaError, match="not dense row-major"):  # contiguous
        gqa.gqa_decode_paged(q, pages, pages, torch.zeros(1, 4, dtype=torch.int32)[:, ::2], lens)


def test_descriptor_checks_context_arguments():
    import torch
    T, P, B = 5, 3, 2
    q = torch.zeros(T, 32, 128, dtype=torch.uint8)
    fp4 = torch.zeros(P, 8, 64, 64, dtype=torch.uint8)
    sf = torch.zeros(P, 8, 64, 8, dtype=torch.uint8)
    bt = torch.zeros(B, 2, dtype=torch.int32)
    qi = torch.tensor([0, 2, 5], dtype=torch.int32)
    kl = torch.tensor([3, 3], dtype=torch.int32)
    call = lambda **kw: gqa.nvfp4_paged_ctx_attn(*[kw.get(n, v) for n, v in (
        ("q", q), ("kf", fp4), ("ks", sf), ("vf", fp4), ("vs", sf), ("bt", bt), ("qi", qi), ("kl", kl))])
    with pytest.raises(gqa.GqaError, match="UNSUPPORTED.*q_fp8 has extent 16 in dimension 1"):
        call(q=torch.zeros(T, 16, 128, dtype=torch.uint8))
    with pytest.raises(gqa.GqaError, match="k_fp4 has dtype f16"):
        call(kf=fp4.half())
    with pytest.raises(gqa.GqaError, match="v_sf has extent 2 in dimension 0; expected 3"):
        call(vs=torch.zeros(2, 8, 64, 8, dtype=torch.uint8))
    with pytest.raises(gqa.GqaError, match="qo_indptr has extent 2 in dimension 0; expected 3"):
        call(qi=torch.tensor([0, 5], dtype=torch.int32))
    with pytest.raises(gqa.GqaError, match="block_table has extent 3 in dimension 0"):
        call(bt=torch.zeros(3, 2, dtype=torch.int32))
    with pytest.raises(gqa.GqaError, match="out_fp8 has extent 4 in dimension 0"):
        gqa.nvfp4_paged_ctx_attn(q, fp4, sf, fp4, sf, bt, qi, kl, out=torch.zeros(4, 32, 128, dtype=torch.uint8))


def test_descriptor_checks_in_c(L):
    """The same checks reached from C with hand-made descriptors: a null
    descriptor, a null data pointer, more dimensions than declared, and
    device fields that disagree -- all before any CUDA call."""
    import torch
    q = torch.zeros(1, 32, 128, dtype=torch.float16)
    kv = torch.zeros(1, 2, 8, 4, 128, dtype=torch.float16)
    lens = torch.ones(1, dtype=torch.int32)
    d = [gqa._desc(t, n) for t, n in ((q, "q"), (kv, "kv"), (lens, "lens"), (q, "out"))]
    r = lambda: [ctypes.byref(x) for x in d]
    assert L.gqa_decode_t(None, *r()[1:], 1.0, P(0)) == INVALID
    assert b"null descriptor" in L.gqa_last_error()
    d[0].data = None
    assert L.gqa_decode_t(*r(), 1.0, P(0)) == INVALID
    assert b"q is a null pointer" in L.gqa_last_error()
    d[0].data = q.data_ptr()
    d[2].ndim = 2
    assert L.gqa_decode_t(*r(), 1.0, P(0)) == INVALID
    assert b"seq_lens has 2 dimensions; expected 1" in L.gqa_last_error()
    d[2].ndim = 1
    d[3].device = 0  # out claims device 0, the others host
    assert L.gqa_decode_t(*r(), 1.0, P(0)) == 3  # GQA_ERR_DEVICE_MISMATCH
    assert b"out is on device 0" in L.gqa_last_error()


def test_decode_plan_covers_capacity():
    for B, cap in [(2, 256), (64, 8192), (8, 131072), (1, 1), (3, 1000)]:
        p = gqa.gqa_decode_plan(B, cap)
        assert p["tokens_per_split"] % 64 == 0
        assert p["num_splits"] * p["tokens_per_split"] >= cap
        assert (p["num_splits"] - 1) * p["tokens_per_split"] < cap
        assert p["num_launches"] == (1 if p["num_splits"] == 1 else 2)
    with pytest.raises(gqa.GqaError):
        gqa.gqa_decode_plan(0, 16)


def test_ctx_plan_splits_only_small_calls():
    """The prefill kernel splits each unit's KV range only when its units
    (8 KV heads x floor((total_q + 63 batch) / 64), a bound on the sequences'
    64-query blocks) leave the 152 SMs idle, into at most 152 / units ranges
    of at least 8 tiles that cover the table.  Calls of at most one query per
    sequence over at least 16 pages take the decode-shaped kernel instead:
    always ranges of 128-key tiles (at least 4 each, at most 32 ranges) that
    cover the table, and a merge."""
    for B, tq, mp in [(2, 2, 64), (1, 32, 512), (4, 8192, 32), (2, 8192, 1024), (1, 1, 4), (1, 1, 16),
                      (64, 64, 128), (8, 8, 2048), (1, 500, 100), (3, 5, 5), (1, 64, 16), (9, 9, 4096)]:
        p = gqa.gqa_ctx_plan(B, tq, mp)
        units = 8 * ((tq + 63 * B) // 64)
        if p["decode_shaped"]:
            assert tq <= B and mp >= 16 and p["persistent"] == 0 and p["num_launches"] == 2
            tiles = (mp + 1) // 2
            assert 1 <= p["num_splits"] <= 32
            assert p["num_splits"] * p["tiles_per_split"] >= tiles > (p["num_splits"] - 1) * p["tiles_per_split"]
            assert p["tiles_per_split"] >= min(4, tiles)
        elif p["num_splits"] == 1:
            assert p["tiles_per_split"] == 0 and p["num_launches"] == 1
            assert units > 76 or mp < 16
        else:
            assert p["num_launches"] == 2
            assert units * p["num_splits"] <= 152
            assert p["tiles_per_split"] >= 8
            assert p["num_splits"] * p["tiles_per_split"] >= mp        # the ranges cover every tile
            assert (p["num_splits"] - 1) * p["tiles_per_split"] < mp   # and none lies past the table
    assert gqa.gqa_ctx_plan(2, 2, 64) == {"tiles_per_split": 4, "num_splits": 8, "num_launches": 2, "persistent": 0,
                                          "decode_shaped": 1}
    assert gqa.gqa_ctx_plan(1, 32, 512) == {"tiles_per_split": 27, "num_splits": 19, "num_launches": 2,
                                            "persistent": 0, "decode_shaped": 0}
    assert gqa.gqa_ctx_plan(64, 64, 128)["decode_shaped"] == 1   # ctx_b64_q1_kv8192
    assert gqa.gqa_ctx_plan(64, 512, 128)["decode_shaped"] == 0  # ctx_b64_q8_kv8192: 8 queries per sequence
    assert gqa.gqa_ctx_plan(1, 1, 15)["decode_shaped"] == 0      # short KV
    assert gqa.gqa_ctx_plan(1, 0, 16)["num_launches"] == 0
    with pytest.raises(gqa.GqaError):
        gqa.gqa_ctx_plan(0, 1, 16)


def test_ctx_plan_takes_persistent_grid_only_for_many_short_units():
    """Unsplit calls with at least two units per SM (8 x floor((total_q + 63
    batch) / 64) >= 304) and short units (max_pages_per_seq <= 48) run the
    persistent grid; long units, few units and split calls do not."""
    assert gqa.gqa_ctx_plan(4, 8192, 32)["persistent"] == 1     # ctx_b4_q2048_kv2048
    assert gqa.gqa_ctx_plan(2, 8192, 1024)["persistent"] == 0   # ctx_b2_q4096_kv65536: long units
    assert gqa.gqa_ctx_plan(64, 64, 128)["persistent"] == 0     # decode-shaped, 128 tiles per unit
    assert gqa.gqa_ctx_plan(1, 2369, 48)["persistent"] == 1  # 8 x floor(2432 / 64) = 304 units, 48 pages
    assert gqa.gqa_ctx_plan(1, 2369, 49)["persistent"] == 0
    assert gqa.gqa_ctx_plan(1, 2368, 48)["persistent"] == 0  # 296 units
    assert gqa.gqa_ctx_plan(1, 0, 16)["persistent"] == 0
    for B, tq, mp in [(2, 2, 64), (1, 32, 512), (1, 1, 4), (3, 5, 5)]:
        p = gqa.gqa_ctx_plan(B, tq, mp)
        assert not (p["persistent"] and p["num_splits"] > 1)


def test_ctx_grid_switch_validates(L):
    for mode in (3, 2, 1, 0):
        assert L.gqa_set_ctx_grid(mode) == OK
    assert L.gqa_set_ctx_grid(4) == INVALID
    assert L.gqa_set_ctx_grid(-1) == INVALID
    assert b"grid mode" in L.gqa_last_error()
    assert L.gqa_set_ctx_grid(0) == OK


def test_starvation_switch_toggles(L):
    assert L.gqa_debug_starve_producers(1) == OK
    assert L.gqa_debug_starve_producers(0) == OK  # off again (the default)


def test_schedule_switch_accepts_only_instantiated_depths(L):
    for st, sl in gqa.CTX_SCHEDULES:
        assert L.gqa_set_schedule(st, sl, 0) == OK
    for d in gqa.DECODE_SCHEDULES:
        assert L.gqa_set_schedule(0, 0, d) == OK
    assert L.gqa_set_schedule(7, 4, 0) == UNSUPPORTED
    assert b"not instantiated" in L.gqa_last_error()
    assert L.gqa_set_schedule(0, 0, 6) == UNSUPPORTED  # not a multiple of the 4 consumer warps
    assert L.gqa_set_schedule(0, 0, 0) == OK  # production depths again


def test_sources_compile_for_sm100a():
    """The same sources build for B200's sm_100a (compile check only: the
    library is tuned for and run on sm_103a; no sm_100a GPU here)."""
    report = build_lib.build_other_arch("sm_100a")
    for kernel in ("ctx_nvfp4_kernel", "decode_split_kernel", "decode_merge_kernel", "ctx_merge_kernel"):
        assert kernel in report and "for 'sm_100a'" in report, kernel
    assert os.path.exists(os.path.join(ROOT, "gqa_attention_kv_split_gb300", "libgqa_sm100a.so"))
