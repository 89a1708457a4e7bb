"""The persistent grid of the context attention (one CTA per SM walks a
snake over the longest-first unit order, with the descriptor ring, the
double-buffered Q and ring counters that run on across units) against the
one-CTA-per-unit grid: byte for byte on shapes where every CTA takes many
units -- ragged query and KV lengths, empty sequences, sequences without
keys, blocks whose second M-tile is idle, rows that see no key -- and on
ctx_b4_q2048_kv2048 (the workload the launch plan gives it), plus the fp64
oracle on the persistent outputs, invalid qo_indptr and the bounded waits
under starvation."""
import numpy as np
import pytest
import torch

import gqa_attention_kv_split_gb300 as gqa
import gqa_workloads as W
import test_gpu_ctx as C
from parity import check_ctx

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def planned_grid_afterwards():
    yield
    gqa.gqa_set_ctx_grid(gqa.CTX_GRID_PLANNED)
    assert gqa.gqa_check_device_errors(0) == 0


def both_grids(x: W.CtxInputs):
    gqa.gqa_set_ctx_grid(gqa.CTX_GRID_PER_UNIT)
    per_unit = C.run(x)
    gqa.gqa_set_ctx_grid(gqa.CTX_GRID_PERSISTENT)
    persistent = C.run(x)
    assert gqa.gqa_check_device_errors(0) == 0
    return per_unit, persistent


def _ragged(seed, n, q_choices, extra_kv):
    rng = np.random.default_rng(seed)
    q_lens = [int(v) for v in rng.choice(q_choices, size=n)]
    kv_lens = [max(0, q + int(k)) for q, k in zip(q_lens, rng.integers(extra_kv[0], extra_kv[1], size=n))]
    return q_lens, kv_lens


CASES = {
    # 60 sequences: empty ones, single rows, blocks of <= 32 queries (M-tile 1 idle), ragged tails
    "ragged_60": _ragged(81, 60, [0, 1, 7, 32, 33, 64, 70, 129, 200], (0, 300)),
    # KV shorter than the queries (rows that see no key) and sequences without keys at all
    "short_kv_48": _ragged(82, 48, [5, 40, 64, 100, 150], (-160, 20)),
    # 80 equal sequences of 200: 2560 units, ~17 per CTA
    "uniform_80x200": ([200] * 80, [200] * 80),
    # one long sequence among many short ones: unequal unit lengths in one snake
    "mixed_long_short": ([1500] + [16] * 40 + [64] * 20, [3000] + [16] * 40 + [700] * 20),
}


@pytest.mark.parametrize("name", list(CASES))
def test_persistent_grid_matches_per_unit_grid_and_oracle(name):
    q_lens, kv_lens = CASES[name]
    x = W.make_ctx_inputs(q_lens, kv_lens, seed=90 + len(q_lens))
    units = 8 * sum((q + 63) // 64 for q in q_lens)
    assert units > 2 * 152, "every CTA of the persistent grid should take several units"
    per_unit, persistent = both_grids(x)
    assert np.array_equal(persistent, per_unit), name
    check_ctx(persistent, C.ref(x), f"persistent grid, {name}")


def test_plan_takes_persistent_grid_for_short_units_and_matches_at_full_size():
    xd = W.ctx_workload("ctx_b4_q2048_kv2048", device=DEV)
    plan = gqa.gqa_ctx_plan(xd.batch, xd.total_q, xd.block_table.shape[1])
    assert plan["persistent"] == 1 and plan["num_splits"] == 1
    a = [xd.q_fp8, xd.k_fp4, xd.k_sf, xd.v_fp4, xd.v_sf, xd.block_table, xd.qo_indptr, xd.kv_lens]
    outs = []
    for mode in (gqa.CTX_GRID_PER_UNIT, gqa.CTX_GRID_PERSISTENT, gqa.CTX_GRID_PLANNED):
        gqa.gqa_set_ctx_grid(mode)
        outs.append(gqa.nvfp4_paged_ctx_attn(*a, q_scale=xd.q_scale, out_scale=xd.out_scale).cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert gqa.gqa_ctx_plan(2, 8192, 1024)["persistent"] == 0  # ctx_b2_q4096_kv65536: long units, one CTA each


@pytest.mark.parametrize("q_lens,kv_lens", [([100, 60] * 30, [200, 60] * 30)])
def test_persistent_grid_flags_short_qo_indptr(q_lens, kv_lens):
    gqa.gqa_set_ctx_grid(gqa.CTX_GRID_PERSISTENT)
    C.test_short_qo_indptr_is_flagged_and_uncovered_rows_zeroed(q_lens, kv_lens)


def test_persistent_grid_writes_nothing_past_total_q():
    gqa.gqa_set_ctx_grid(gqa.CTX_GRID_PERSISTENT)
    C.test_overlong_qo_indptr_writes_nothing_past_total_q()


def test_persistent_grid_bounded_waits_expire():
    """Producers starved under the persistent grid: every role's wait
    expires, each CTA drains and frees its tensor memory, the host reads
    GQA_ERR_TIMEOUT, and the next normal call is correct."""
    import time
    x = W.make_ctx_inputs([100, 40] * 20, [300, 40] * 20, seed=93)  # 480 units: ~3 per CTA
    assert gqa.gqa_check_device_errors(0) == 0
    gqa.gqa_set_ctx_grid(gqa.CTX_GRID_PERSISTENT)
    gqa.gqa_debug_starve_producers(True)
    try:
        t0 = time.perf_counter()
        gqa.nvfp4_paged_ctx_attn(*C.args_of(x), q_scale=x.q_scale, out_scale=x.out_scale)
        word = gqa.gqa_check_device_errors(0)
        took = time.perf_counter() - t0
    finally:
        gqa.gqa_debug_starve_producers(False)
    assert word & 1, word
    assert took < 60
    check_ctx(C.run(x), C.ref(x), "persistent grid, after expired waits")
