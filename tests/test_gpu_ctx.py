"""GPU parity of nvfp4_paged_ctx_attn (through the C ABI) against the fp64
oracle.  Tolerance (tests/parity.py): >= 99.9 % of output elements within 2
E4M3 ulps of E4M3(exact) and rel-L2 <= 3e-2 after dequantisation.  Cases:
small ragged shapes spanning several 64-query units and 128-key tiles,
decode-like rows, rows that see no key, q_scale / out_scale != 1, the
split-KV path (few units: each unit's KV range divided and merged, with
empty ranges, ragged tails and the idle second M-tile), the
ctx_b4_q2048_kv2048, ctx_b2_q1_kv4096 and ctx_b1_q32_kv32768 workloads in
full, and ctx_b2_q4096_kv65536 on sampled rows in the benchmark's launch
configuration."""
import numpy as np
import pytest
import torch

import gqa_attention_kv_split_gb300 as gqa
import gqa_workloads as W
import oracle
from parity import check_ctx

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    gqa.build()
    yield
    assert gqa.gqa_check_device_errors(0) == 0


def args_of(x: W.CtxInputs, dev=DEV):
    return [t.to(dev) for t in (x.q_fp8, x.k_fp4, x.k_sf, x.v_fp4, x.v_sf, x.block_table, x.qo_indptr, x.kv_lens)]


def run(x: W.CtxInputs):
    out = gqa.nvfp4_paged_ctx_attn(*args_of(x), q_scale=x.q_scale, out_scale=x.out_scale)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def ref(x: W.CtxInputs, items=None):
    h = [t.cpu().numpy() for t in (x.q_fp8, x.k_fp4, x.k_sf, x.v_fp4, x.v_sf, x.block_table, x.qo_indptr, x.kv_lens)]
    return oracle.nvfp4_paged_ctx_attn(h[0], x.q_scale, *h[1:], x.out_scale, items=items)


@pytest.mark.parametrize("q_lens,kv_lens", [
    ([16], [16]),                 # one tile, one unit, square causal
    ([40, 130], [100, 130]),      # ragged units and tiles
    ([1, 1, 3], [300, 64, 129]),  # decode-like rows
    ([200], [200]),               # several units, diagonal tiles
    ([64], [1000]),               # long prefix, one unit
    ([129, 70], [257, 70]),
])
def test_small_shapes(q_lens, kv_lens):
    x = W.make_ctx_inputs(q_lens, kv_lens, seed=51 + sum(q_lens))
    check_ctx(run(x), ref(x), f"q{q_lens} kv{kv_lens}")


def test_rows_without_keys_are_zero():
    x = W.make_ctx_inputs([70], [3], seed=52)  # queries 0..66 see no key
    got = run(x)
    assert np.all(got[:67] == 0)
    check_ctx(got, ref(x), "q_len > kv_len")


@pytest.mark.parametrize("q_scale,out_scale", [(0.5, 1.0), (1.0, 2.0), (1.7, 0.25)])
def test_scales(q_scale, out_scale):
    x = W.make_ctx_inputs([100, 33], [300, 33], seed=53, q_scale=q_scale, out_scale=out_scale)
    check_ctx(run(x), ref(x), f"q_scale {q_scale} out_scale {out_scale}")


def test_constant_v_returns_v():
    x = W.make_ctx_inputs([90], [400], seed=54)
    x.v_fp4[:] = 0x22  # E2M1 1.0 in both nibbles
    x.v_sf[:] = 0x30   # E4M3 0.5
    got = oracle.e4m3_table()[run(x)]
    assert np.all(got == 0.5)


def test_deterministic_and_host_path():
    x = W.make_ctx_inputs([150, 20], [150, 500], seed=55)
    a = run(x)
    b = run(x)
    assert np.array_equal(a, b)
    host = gqa.nvfp4_paged_ctx_attn(x.q_fp8, x.k_fp4, x.k_sf, x.v_fp4, x.v_sf, x.block_table, x.qo_indptr,
                                    x.kv_lens, q_scale=x.q_scale, out_scale=x.out_scale)
    assert np.array_equal(a, host.numpy())


def test_many_sequences_and_empty_queries():
    """40 sequences (the unit lookup walks two groups of 32), some with no
    query rows, ragged query and KV lengths."""
    rng = np.random.default_rng(64)
    q_lens = [int(v) for v in rng.choice([0, 1, 7, 33, 64, 70], size=40)]
    kv_lens = [q + int(k) for q, k in zip(q_lens, rng.integers(0, 150, size=40))]
    x = W.make_ctx_inputs(q_lens, kv_lens, seed=64)
    check_ctx(run(x), ref(x), "40 sequences")


def plan_of(x: W.CtxInputs):
    return gqa.gqa_ctx_plan(x.block_table.shape[0], x.q_fp8.shape[0], x.block_table.shape[1])


# Split-KV: units too few to fill the GPU, so each unit's KV range is divided
# and the ranges merged.  Every case asserts that the split is really taken.
@pytest.mark.parametrize("q_lens,kv_lens", [
    ([1], [4096]),               # decode-like: 8 ranges of 8 tiles
    ([5, 1], [3000, 700]),       # ragged tails; the short sequence's later ranges are empty
    ([32], [8192]),              # a single block of 32 queries: M-tile 1 is skipped
    ([40], [2000]),              # M-tile 1 holds queries 32..39 only
    ([33, 64], [1100, 1500]),    # several units, range boundaries inside the causal diagonal's reach
])
def test_split_kv_shapes(q_lens, kv_lens):
    x = W.make_ctx_inputs(q_lens, kv_lens, seed=61 + sum(kv_lens))
    assert plan_of(x)["num_splits"] > 1
    check_ctx(run(x), ref(x), f"split q{q_lens} kv{kv_lens}")


def test_split_kv_rows_without_keys_and_empty_ranges():
    # sequence 0: 100 queries over 60 keys (queries 0..39 see none) and a single
    # tile, so all its ranges but the first are empty; sequence 1 forces the split
    x = W.make_ctx_inputs([100, 1], [60, 2048], seed=62)
    assert plan_of(x)["num_splits"] > 1
    got = run(x)
    assert np.all(got[:40] == 0)
    check_ctx(got, ref(x), "split, rows without keys")


def test_split_kv_scales_and_host_path():
    x = W.make_ctx_inputs([3], [1500], seed=63, q_scale=1.7, out_scale=0.25)
    assert plan_of(x)["num_splits"] > 1
    a = run(x)
    check_ctx(a, ref(x), "split, q_scale 1.7 out_scale 0.25")
    assert np.array_equal(a, run(x))
    host = gqa.nvfp4_paged_ctx_attn(x.q_fp8, x.k_fp4, x.k_sf, x.v_fp4, x.v_sf, x.block_table, x.qo_indptr,
                                    x.kv_lens, q_scale=x.q_scale, out_scale=x.out_scale)
    assert np.array_equal(a, host.numpy())


@pytest.mark.parametrize("name", ["ctx_b2_q1_kv4096", "ctx_b1_q32_kv32768"])
def test_workload_split_rows_full(name):
    x = W.ctx_workload(name)
    assert plan_of(x)["num_splits"] > 1
    check_ctx(run(x), ref(x), name)


def test_workload_b4_q2048_kv2048_full():
    x = W.ctx_workload("ctx_b4_q2048_kv2048")
    frac, rl, mx = check_ctx(run(x), ref(x), "ctx_b4_q2048_kv2048")
    assert rl <= 3e-2  # attainable here: the plain bound applies


def test_workload_b2_q4096_kv65536_sampled():
    x = W.ctx_workload("ctx_b2_q4096_kv65536")
    got = run(x)
    rng = np.random.default_rng(5)
    rows = np.concatenate([[0, 1, 4095, 4096, 4097, 8191], rng.integers(0, 8192, 58)])
    heads = rng.integers(0, 32, rows.size)
    items = np.stack([rows, heads], axis=1)
    r = ref(x, items=items)
    g = np.stack([got[rr, hh] for rr, hh in items])
    check_ctx(g, r, "ctx_b2_q4096_kv65536 sampled")
