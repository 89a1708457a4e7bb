"""Ring-depth study: every instantiated schedule computes the same result,
bit for bit (the invariant "GB300 NVFP4 Context Attention: scale slot 조기
반납과 8단 packed K/V ring" checks for its ring changes), so a schedule changes
only speed.  Context attention at every (packed stages, K/V slots) pair,
decode at every ring depth, each against the production depths, byte for
byte, on shapes with ragged tails, diagonal tiles and one or many splits."""
import numpy as np
import pytest
import torch

import gqa_attention_kv_split_gb300 as gqa
import gqa_workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def production_depths_afterwards():
    yield
    gqa.gqa_set_schedule(0, 0, 0)
    assert gqa.gqa_check_device_errors(0) == 0


def _ctx(x):
    a = [t.to(DEV) for t in (x.q_fp8, x.k_fp4, x.k_sf, x.v_fp4, x.v_sf, x.block_table, x.qo_indptr, x.kv_lens)]
    out = gqa.nvfp4_paged_ctx_attn(*a, q_scale=x.q_scale, out_scale=x.out_scale)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("q_lens,kv_lens", [([200, 70], [700, 70]), ([129, 1, 64, 300], [2000, 500, 64, 300])])
def test_ctx_schedules_are_bit_identical(q_lens, kv_lens):
    x = W.make_ctx_inputs(q_lens, kv_lens, seed=71 + sum(kv_lens))
    assert gqa.gqa_ctx_plan(x.batch, x.total_q, x.block_table.shape[1])["num_splits"] == 1
    gqa.gqa_set_schedule(0, 0, 0)
    ref = _ctx(x)
    for st, sl in gqa.CTX_SCHEDULES[1:]:
        gqa.gqa_set_schedule(st, sl, 0)
        got = _ctx(x)
        assert torch.equal(got, ref), f"schedule ({st}, {sl}) differs from the production depths"


def test_ctx_schedules_bit_identical_at_full_size():
    xd = W.ctx_workload("ctx_b4_q2048_kv2048", device=DEV)
    gqa.gqa_set_schedule(0, 0, 0)
    ref = _ctx(xd)
    for st, sl in gqa.CTX_SCHEDULES[1:]:
        gqa.gqa_set_schedule(st, sl, 0)
        assert torch.equal(_ctx(xd), ref), f"schedule ({st}, {sl})"


@pytest.mark.parametrize("batch,cap,lens", [(3, 256, [1, 200, 256]), (5, 5000, [5000, 17, 2500, 0, 4999])])
def test_decode_schedules_are_bit_identical(batch, cap, lens):
    x = W.make_decode_inputs(batch, cap, lens, seed=72 + cap)
    q, kv, sl = x.q.to(DEV), x.kv.to(DEV), x.seq_lens.to(DEV)
    gqa.gqa_set_schedule(0, 0, 0)
    ref = gqa.gqa_decode(q, kv, sl, q_scale=x.q_scale).cpu()
    for d in gqa.DECODE_SCHEDULES[1:]:
        gqa.gqa_set_schedule(0, 0, d)
        got = gqa.gqa_decode(q, kv, sl, q_scale=x.q_scale).cpu()
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"decode ring depth {d} differs"
