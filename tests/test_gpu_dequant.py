"""The context kernel's NVFP4 -> E4M3 dequantisation, bit-exact against the
oracle's decoded E4M3 tiles, through gqa_debug_dequant_pages.  The export
writes the K path's E4M3 bytes and checks on the device that the V path's
f16 values are the same numbers (bit 3 of the error word otherwise), so a
clean error word after the bit-exact comparison covers both paths."""
import numpy as np
import pytest
import torch

import gqa_attention_kv_split_gb300 as gqa
import gqa_workloads as W
import oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def gpu_dequant(fp4, sf, bt, kl, max_kv):
    out = gqa.gqa_debug_dequant_pages(fp4.to(DEV), sf.to(DEV), bt.to(DEV), kl.to(DEV), max_kv)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("shuffle", [False, True])
def test_random_pages_bit_exact(shuffle):
    x = W.make_ctx_inputs([1, 1, 1], [200, 64, 3], seed=31, shuffle=shuffle)
    for fp4, sf in ((x.k_fp4, x.k_sf), (x.v_fp4, x.v_sf)):
        got = gpu_dequant(fp4, sf, x.block_table, x.kv_lens, 200)
        exp = oracle.dequant_pages(fp4.numpy(), sf.numpy(), x.block_table.numpy(), x.kv_lens.numpy(), 200)
        assert np.array_equal(got, exp)
    assert gqa.gqa_check_device_errors(0) == 0


def test_every_code_and_scale_bit_exact():
    """All 16 E2M1 codes against all 254 non-NaN E4M3 scale codes (both signs,
    subnormal products, ties, saturation)."""
    scales = [c for c in range(256) if (c & 0x7F) != 0x7F]
    n_tok = len(scales)  # one token per scale code; all 8 blocks of a token share it
    pages = (n_tok + 63) // 64
    fp4 = torch.zeros(pages, 8, 64, 64, dtype=torch.uint8)
    sf = torch.zeros(pages, 8, 64, 8, dtype=torch.uint8)
    codes = torch.arange(16, dtype=torch.uint8)
    byte_pattern = (codes[0::2] | (codes[1::2] << 4))  # 8 bytes: codes 0..15 in element order
    for t, s in enumerate(scales):
        p, slot = divmod(t, 64)
        fp4[p, :, slot, :] = byte_pattern.repeat(8)
        sf[p, :, slot, :] = s
    bt = torch.arange(pages, dtype=torch.int32).view(1, pages)
    kl = torch.tensor([n_tok], dtype=torch.int32)
    got = gpu_dequant(fp4, sf, bt, kl, n_tok)
    exp = oracle.dequant_pages(fp4.numpy(), sf.numpy(), bt.numpy(), kl.numpy(), n_tok)
    bad = np.argwhere(got != exp)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"
    assert gqa.gqa_check_device_errors(0) == 0  # the V path's f16 values agreed with every E4M3 byte
