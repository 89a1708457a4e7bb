"""Pins for the NVFP4 paged context-attention oracle (CPU only).

* Dequantisation is checked against an independent route through library
  routines: torch's float8_e4m3fn decode of the scales, the printed E2M1 value
  table (tests/golden/e2m1_values.txt), a float32 product (exact) and torch's
  float32 -> float8_e4m3fn cast.
* Attention is checked against torch's scaled_dot_product_attention in fp64
  with enable_gqa=True and torch's own bottom-right causal bias
  (torch.nn.attention.bias.causal_lower_right) on the decoded tensors.
* Closed forms: q_len = kv_len = 1 returns v[0]; a constant V returns V;
  out_scale divides the result; a shuffled block table changes nothing.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import gqa_workloads as W
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_table():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_values.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split()
                vals[int(c)] = float(v)
    return torch.tensor([vals[i] for i in range(16)], dtype=torch.float32)


def torch_dequant(fp4, sf, block_table, kv_lens):
    """[B, max_kv, 8, 128] E4M3 codes via library casts (independent of the oracle)."""
    e2m1 = _e2m1_table()
    B = kv_lens.shape[0]
    max_kv = int(kv_lens.max())
    out = torch.zeros(B, max_kv, 8, 128, dtype=torch.uint8)
    for b in range(B):
        n = int(kv_lens[b])
        t = torch.arange(n)
        pages = block_table[b, t // 64].long()
        slots = t % 64
        packed = fp4[pages, :, slots, :]               # [n, 8, 64]
        codes = torch.stack([packed & 0xF, packed >> 4], dim=-1).reshape(n, 8, 128)
        vals = e2m1[codes.long()]
        scales = sf[pages, :, slots, :].view(torch.float8_e4m3fn).to(torch.float32)  # [n,8,8]
        prod = vals * scales.repeat_interleave(16, dim=-1)
        out[b, :n] = prod.to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def sdpa_ctx_ref(x: W.CtxInputs):
    """fp64 SDPA with bottom-right causal bias over torch-decoded tensors."""
    kq = torch_dequant(x.k_fp4, x.k_sf, x.block_table, x.kv_lens)
    vq = torch_dequant(x.v_fp4, x.v_sf, x.block_table, x.kv_lens)
    out = torch.zeros(x.total_q, 32, 128, dtype=torch.float64)
    qi = x.qo_indptr.tolist()
    for b in range(x.batch):
        ql, kl = qi[b + 1] - qi[b], int(x.kv_lens[b])
        q = x.q_fp8[qi[b]:qi[b + 1]].view(torch.float8_e4m3fn).double().permute(1, 0, 2)[None]
        k = kq[b, :kl].view(torch.float8_e4m3fn).double().permute(1, 0, 2)[None]
        v = vq[b, :kl].view(torch.float8_e4m3fn).double().permute(1, 0, 2)[None]
        mask = causal_lower_right(ql, kl)._materialize()
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=x.q_scale / np.sqrt(128.0),
                                           enable_gqa=True)
        o = torch.nan_to_num(o, nan=0.0)  # rows with no visible key: zero by the library's reading
        out[qi[b]:qi[b + 1]] = o[0].permute(1, 0, 2) / x.out_scale
    return out.numpy()


def run_oracle(x: W.CtxInputs, **kw):
    return oracle.nvfp4_paged_ctx_attn(
        x.q_fp8.numpy(), x.q_scale, x.k_fp4.numpy(), x.k_sf.numpy(), x.v_fp4.numpy(), x.v_sf.numpy(),
        x.block_table.numpy(), x.qo_indptr.numpy(), x.kv_lens.numpy(), x.out_scale, **kw)


def test_bottom_right_causal_golden_matches_library_bias():
    rows = []
    with open(os.path.join(GOLDEN, "bottom_right_causal_q3_kv5.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    assert torch.equal(causal_lower_right(3, 5)._materialize().int(), torch.tensor(rows, dtype=torch.int32))


@pytest.mark.parametrize("shuffle", [False, True])
def test_dequant_matches_library_casts(shuffle):
    x = W.make_ctx_inputs([5, 70], [130, 70], seed=11, shuffle=shuffle)
    for fp4, sf in ((x.k_fp4, x.k_sf), (x.v_fp4, x.v_sf)):
        ours = oracle.dequant_pages(fp4.numpy(), sf.numpy(), x.block_table.numpy(), x.kv_lens.numpy())
        ref = torch_dequant(fp4, sf, x.block_table, x.kv_lens).numpy()
        assert np.array_equal(ours, ref)


def test_dequant_independent_of_page_placement():
    a = W.make_ctx_inputs([1, 1], [150, 64], seed=12, shuffle=False)
    b = W.make_ctx_inputs([1, 1], [150, 64], seed=12, shuffle=True)
    assert not torch.equal(a.block_table, b.block_table)
    da = oracle.dequant_pages(a.k_fp4.numpy(), a.k_sf.numpy(), a.block_table.numpy(), a.kv_lens.numpy())
    db = oracle.dequant_pages(b.k_fp4.numpy(), b.k_sf.numpy(), b.block_table.numpy(), b.kv_lens.numpy())
    assert np.array_equal(da, db)


@pytest.mark.parametrize("q_lens,kv_lens,q_scale,out_scale", [
    ([16, 16], [16, 16], 1.0, 1.0),
    ([7, 33], [100, 33], 1.0, 1.0),
    ([64], [200], 0.5, 2.0),
    ([1, 3], [129, 3], 1.3, 1.0),
])
def test_ctx_matches_sdpa_fp64(q_lens, kv_lens, q_scale, out_scale):
    x = W.make_ctx_inputs(q_lens, kv_lens, seed=13, q_scale=q_scale, out_scale=out_scale)
    np.testing.assert_allclose(run_oracle(x), sdpa_ctx_ref(x), rtol=1e-11, atol=1e-12)


def test_ctx_single_key_returns_v0():
    x = W.make_ctx_inputs([1], [1], seed=14)
    out = run_oracle(x)
    vq = oracle.dequant_pages(x.v_fp4.numpy(), x.v_sf.numpy(), x.block_table.numpy(), x.kv_lens.numpy())
    v0 = oracle.e4m3_table()[vq[0, 0]]  # [8,128]
    for h in range(32):
        assert np.array_equal(out[0, h], v0[h // 4])


def test_ctx_constant_v_returns_v():
    x = W.make_ctx_inputs([20], [90], seed=15)
    # every V element = E2M1 1.0 (code 2) with scale 0.5 (E4M3 0x30): value 0.5
    x.v_fp4[:] = 0x22
    x.v_sf[:] = 0x30
    np.testing.assert_allclose(run_oracle(x), 0.5, rtol=1e-14, atol=0)


def test_ctx_out_scale_divides():
    x1 = W.make_ctx_inputs([9], [40], seed=16, out_scale=1.0)
    x2 = W.make_ctx_inputs([9], [40], seed=16, out_scale=4.0)
    np.testing.assert_allclose(run_oracle(x1) / 4.0, run_oracle(x2), rtol=1e-15, atol=0)


def test_ctx_rows_without_keys_are_zero():
    # q_len 5 > kv_len 3: queries 0 and 1 see no key under the bottom-right rule
    x = W.make_ctx_inputs([5], [3], seed=17)
    out = run_oracle(x)
    assert np.all(out[0] == 0) and np.all(out[1] == 0)
    assert np.any(out[2] != 0)


def test_ctx_item_subset_equals_full():
    x = W.make_ctx_inputs([10, 4], [30, 70], seed=18)
    full = run_oracle(x)
    items = np.array([[13, 5], [0, 31], [9, 8]])
    sub = run_oracle(x, items=items)
    for k, (r, h) in enumerate(items):
        np.testing.assert_array_equal(sub[k], full[r, h])
