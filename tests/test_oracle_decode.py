"""Pins for the fp64 decode oracle (CPU only).

The oracle is checked against torch's scaled_dot_product_attention in fp64
with enable_gqa=True and a boolean length mask -- the comparator named on
"NVIDIA SM110 GPU를 위한 실험적인 FP16 GQA 디코드 커널 추가", section 3 --
and against closed forms: one visible token returns that token's V, a
constant V returns V, and an empty sequence returns zeros.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import gqa_workloads as W
import oracle


def sdpa_decode_ref(q, kv, lens, q_scale):
    """torch SDPA (fp64, CPU) with enable_gqa -- a library routine."""
    B, Hq, D = q.shape
    cap = kv.shape[3]
    qq = q.double().view(B, Hq, 1, D)
    k = kv[:, 0].double()
    v = kv[:, 1].double()
    mask = (torch.arange(cap)[None, :] < lens.long()[:, None]).view(B, 1, 1, cap)
    out = F.scaled_dot_product_attention(qq, k, v, attn_mask=mask, scale=q_scale / np.sqrt(128.0),
                                         enable_gqa=True)
    return out.view(B, Hq, D).numpy()


@pytest.mark.parametrize("lens,cap,q_scale,seed", [
    ([1, 200], 256, 1.0, 0),
    ([64, 127, 191, 256], 256, 1.0, 5),   # the B4 / capacity 256 shape of the decode page's tables
    ([3, 17, 64], 80, 0.5, 6),
    ([40], 64, 2.0, 7),
])
def test_decode_matches_sdpa_fp64(lens, cap, q_scale, seed):
    x = W.make_decode_inputs(len(lens), cap, lens, seed=seed, q_scale=q_scale)
    ours = oracle.gqa_decode(x.q.numpy(), x.kv.numpy(), x.seq_lens.numpy(), q_scale)
    ref = sdpa_decode_ref(x.q, x.kv, x.seq_lens, q_scale)
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)


def test_head_mapping_is_contiguous_groups():
    """Query head h must read KV head h // 4: give each KV head a constant V
    equal to its index and check every query head's output."""
    x = W.make_decode_inputs(1, 16, [16], seed=1)
    kv = x.kv.clone()
    for g in range(8):
        kv[0, 1, g] = float(g)
    out = oracle.gqa_decode(x.q.numpy(), kv.numpy(), x.seq_lens.numpy())
    for h in range(32):
        np.testing.assert_allclose(out[0, h], h // 4, rtol=1e-14, atol=0)


def test_single_token_returns_v0_exactly():
    x = W.make_decode_inputs(2, 256, [1, 200], seed=0)
    out = oracle.gqa_decode(x.q.numpy(), x.kv.numpy(), x.seq_lens.numpy())
    v0 = x.kv[0, 1, :, 0, :].double().numpy()  # [8,128]
    for h in range(32):
        assert np.array_equal(out[0, h], v0[h // 4])


def test_constant_v_returns_v():
    x = W.make_decode_inputs(2, 64, [37, 64], seed=3)
    kv = x.kv.clone()
    kv[:, 1] = 0.375
    out = oracle.gqa_decode(x.q.numpy(), kv.numpy(), x.seq_lens.numpy())
    np.testing.assert_allclose(out, 0.375, rtol=1e-14, atol=0)


def test_zero_length_and_clamp():
    x = W.make_decode_inputs(3, 32, [0, 40, -5], seed=4)
    out = oracle.gqa_decode(x.q.numpy(), x.kv.numpy(), x.seq_lens.numpy())
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    full = oracle.gqa_decode(x.q.numpy(), x.kv.numpy(), np.array([0, 32, 0], dtype=np.int32))
    np.testing.assert_array_equal(out[1], full[1])  # 40 > capacity 32 -> clamped


def test_item_subset_equals_full():
    x = W.make_decode_inputs(3, 96, [5, 96, 50], seed=8, q_scale=0.7)
    full = oracle.gqa_decode(x.q.numpy(), x.kv.numpy(), x.seq_lens.numpy(), 0.7)
    items = np.array([[2, 31], [0, 0], [1, 17]])
    sub = oracle.gqa_decode(x.q.numpy(), x.kv.numpy(), x.seq_lens.numpy(), 0.7, items=items)
    for k, (b, h) in enumerate(items):
        np.testing.assert_array_equal(sub[k], full[b, h])


def test_token_permutation_invariance():
    """Softmax attention ignores token order: shuffling K and V rows together
    leaves every output unchanged (up to fp64 rounding order)."""
    x = W.make_decode_inputs(1, 50, [50], seed=9)
    perm = torch.randperm(50, generator=torch.Generator().manual_seed(1))
    kv2 = x.kv[:, :, :, perm, :].contiguous()
    a = oracle.gqa_decode(x.q.numpy(), x.kv.numpy(), x.seq_lens.numpy())
    b = oracle.gqa_decode(x.q.numpy(), kv2.numpy(), x.seq_lens.numpy())
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


# ---- paged decode: the gather through the block table -------------------

def test_paged_identity_table_equals_stacked():
    """With pages laid out in order (block table = 0, 1, 2, ...), the paged
    oracle sees exactly the stacked cache: bit-identical fp64 results."""
    x = W.make_decode_inputs(3, 256, [1, 200, 256], seed=71)
    p = W.page_decode_inputs(x, seed=71, shuffle=False)
    assert np.array_equal(p.block_table.numpy().ravel(), np.arange(12))
    d = oracle.gqa_decode(x.q.numpy(), x.kv.numpy(), x.seq_lens.numpy(), x.q_scale)
    g = oracle.gqa_decode_paged(p.q.numpy(), p.k_pages.numpy(), p.v_pages.numpy(), p.block_table.numpy(),
                                p.seq_lens.numpy(), p.q_scale)
    assert np.array_equal(d, g)


def test_paged_result_is_independent_of_page_placement():
    """Shuffling the physical pages (and the table with them) changes nothing."""
    x = W.make_decode_inputs(2, 320, [320, 77], seed=72)
    a = W.page_decode_inputs(x, seed=72, shuffle=False)
    b = W.page_decode_inputs(x, seed=72, shuffle=True)
    assert not np.array_equal(a.block_table.numpy(), b.block_table.numpy())
    ra = oracle.gqa_decode_paged(a.q.numpy(), a.k_pages.numpy(), a.v_pages.numpy(), a.block_table.numpy(),
                                 a.seq_lens.numpy(), a.q_scale)
    rb = oracle.gqa_decode_paged(b.q.numpy(), b.k_pages.numpy(), b.v_pages.numpy(), b.block_table.numpy(),
                                 b.seq_lens.numpy(), b.q_scale)
    assert np.array_equal(ra, rb)


def test_paged_ignores_slots_past_the_length_and_unused_pages():
    """Slots of the last page past the length, pages the table does not reach
    and table entries past the last page do not enter the result; a page used
    by a token does (the gather reads the right slot)."""
    x = W.make_decode_inputs(2, 256, [70, 130], seed=73)
    p = W.page_decode_inputs(x, seed=73)
    ref = oracle.gqa_decode_paged(p.q.numpy(), p.k_pages.numpy(), p.v_pages.numpy(), p.block_table.numpy(),
                                  p.seq_lens.numpy(), p.q_scale)
    kp, vp, bt = p.k_pages.numpy().copy(), p.v_pages.numpy().copy(), p.block_table.numpy().copy()
    kp[bt[0, 1], :, 6:] = np.float16(300.0)   # sequence 0 holds 70 tokens: page 1, slots 6.. unused
    vp[bt[0, 1], :, 6:] = np.float16(-300.0)
    kp[bt[0, 2]] = np.float16(123.0)          # page 2 of sequence 0 is never reached
    bt[1, 3] = 10 ** 6                        # entry past sequence 1's last page (130 tokens: pages 0..2)
    got = oracle.gqa_decode_paged(p.q.numpy(), kp, vp, bt, p.seq_lens.numpy(), p.q_scale)
    assert np.array_equal(ref, got)
    vp[bt[0, 1], :, 5] = np.float16(50.0)     # token 69 = page 1, slot 5: it is read
    moved = oracle.gqa_decode_paged(p.q.numpy(), kp, vp, bt, p.seq_lens.numpy(), p.q_scale)
    assert not np.allclose(moved[0], ref[0]) and np.array_equal(moved[1], ref[1])
