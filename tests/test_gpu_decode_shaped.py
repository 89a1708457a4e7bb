"""The decode-shaped context kernel (S and P V computed transposed: keys on
the MMA's M dimension, 4 queries x 4 heads on N; KV ranges merged) against
the fp64 oracle, forced onto calls of every shape: one query per sequence,
several (chunks of 4 queries), ragged and single-page KV, sequences without
queries or keys, rows that see no key, q_scale / out_scale != 1; invalid
qo_indptr; its bounded waits under starvation; deterministic results.  The
planned choice of the kernel (calls of at most one query per sequence over
at least 16 pages) and its full-size workloads are covered in
test_abi.py and test_gpu_ctx.py."""
import time

import numpy as np
import pytest
import torch

import gqa_attention_kv_split_gb300 as gqa
import gqa_workloads as W
import test_gpu_ctx as C
from parity import check_ctx

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def decode_shaped_kernel():
    gqa.gqa_set_ctx_grid(gqa.CTX_GRID_DECODE_SHAPED)
    yield
    gqa.gqa_set_ctx_grid(gqa.CTX_GRID_PLANNED)
    assert gqa.gqa_check_device_errors(0) == 0


def _ragged_q1(n, seed):
    rng = np.random.default_rng(seed)
    return [1] * n, [int(v) for v in rng.integers(1, 5000, size=n)]


@pytest.mark.parametrize("q_lens,kv_lens", [
    ([1], [64]),                           # one page: the tile's second page is absent
    ([1, 1, 3], [300, 64, 129]),           # ragged pages, keys past kv_len in the last page
    ([2], [1000]),
    ([5, 1], [3000, 700]),                 # 5 queries: two chunks of the sequence
    ([4, 4], [100, 3]),                    # KV shorter than the queries: rows that see no key
    ([1, 0, 2, 1], [0, 500, 64, 129]),     # a sequence without keys, one without queries
    ([7, 2, 1, 9], [900, 130, 5000, 257]),
    _ragged_q1(40, 7),                     # 40 sequences (the unit lookup's prefix sums span two warps' worth)
])
def test_decode_shaped_shapes(q_lens, kv_lens):
    x = W.make_ctx_inputs(q_lens, kv_lens, seed=300 + sum(kv_lens), out_scale=2.0 ** -4)
    assert C.plan_of(x)["decode_shaped"] == 1
    got = C.run(x)
    check_ctx(got, C.ref(x), f"decode-shaped q{q_lens[:8]} kv{kv_lens[:8]}")
    if 0 in kv_lens:
        b = kv_lens.index(0)
        r0 = sum(q_lens[:b])
        assert np.all(got[r0:r0 + q_lens[b]] == 0)


def test_decode_shaped_scales_and_determinism():
    x = W.make_ctx_inputs([1, 1], [2000, 300], seed=311, q_scale=1.7, out_scale=0.25)
    a = C.run(x)
    check_ctx(a, C.ref(x), "decode-shaped, q_scale 1.7 out_scale 0.25")
    assert np.array_equal(a, C.run(x))


# (the last sequence keeps one of its rows, so it needs more than one)
@pytest.mark.parametrize("q_lens,kv_lens", [([1, 1] * 20 + [3], [200, 60] * 20 + [500]), ([1, 2], [3000, 2000])])
def test_decode_shaped_short_qo_indptr(q_lens, kv_lens):
    C.test_short_qo_indptr_is_flagged_and_uncovered_rows_zeroed(q_lens, kv_lens)


def test_decode_shaped_overlong_qo_indptr():
    C.test_overlong_qo_indptr_writes_nothing_past_total_q()


def test_decode_shaped_bounded_waits_expire():
    """Producers starved: every role's wait expires (the softmax warps keep
    meeting at their named barriers and finish their loops), each CTA drains
    and frees its tensor memory, the host reads GQA_ERR_TIMEOUT, and the next
    normal call is correct."""
    x = W.make_ctx_inputs([1] * 24, [900] * 24, seed=312)
    assert gqa.gqa_check_device_errors(0) == 0
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
    check_ctx(C.run(x), C.ref(x), "decode-shaped, after expired waits")
    torch.cuda.synchronize()
