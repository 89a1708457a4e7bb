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
