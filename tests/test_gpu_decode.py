"""GPU parity of gqa_decode (through the C ABI) against the fp64 oracle.

Tolerance: max |err| <= 1e-2 and rel-L2 <= 2e-3 (tests/parity.py).  Cases
span one and many splits, ragged tails, empty and clamped lengths, the
shapes of the decode page's benchmark tables, and the full-size workloads
in the launch configuration the benchmark times (sampled rows)."""
import numpy as np
import pytest
import torch

import gqa_attention_kv_split_gb300 as gqa
import gqa_workloads as W
import oracle
from parity import check_decode

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    gqa.build()
    yield
    assert gqa.gqa_check_device_errors(0) == 0


def run(x: W.DecodeInputs, **kw):
    out = gqa.gqa_decode(x.q.to(DEV), x.kv.to(DEV), x.seq_lens.to(DEV), q_scale=x.q_scale, **kw)
    torch.cuda.synchronize()
    return out.cpu()


def ref(x: W.DecodeInputs, items=None):
    return oracle.gqa_decode(x.q.cpu().numpy(), x.kv.cpu().numpy(), x.seq_lens.cpu().numpy(), x.q_scale,
                             items=items)


def test_workload_b2_cap256_full():
    x = W.decode_workload("decode_b2_cap256")
    got = run(x)
    check_decode(got.double().numpy(), ref(x), "decode_b2_cap256")
    # one visible token returns V[0] (fp16-exact: the kernel's weights are 1)
    v0 = x.kv[0, 1, :, 0, :]
    for h in range(32):
        assert torch.equal(got[0, h], v0[h // 4])


@pytest.mark.parametrize("batch,cap,lens", [
    (1, 64, [1]), (4, 256, [64, 127, 191, 256]), (1, 1024, [1024]), (1, 4096, [3968]),
])
def test_decode_page_table_shapes(batch, cap, lens):
    x = W.make_decode_inputs(batch, cap, lens, seed=100 + cap)
    check_decode(run(x).double().numpy(), ref(x), f"B{batch} cap{cap}")


@pytest.mark.parametrize("cap", [1000, 4100])
def test_ragged_and_degenerate_lengths(cap):
    lens = [0, 1, 2, 15, 16, 17, 63, 64, 65, 511, 512, 513, cap - 1, cap, cap + 7, -3]
    x = W.make_decode_inputs(len(lens), cap, lens, seed=7)
    got = run(x)
    check_decode(got.double().numpy(), ref(x), f"ragged cap{cap}")
    assert torch.count_nonzero(got[0]) == 0 and torch.count_nonzero(got[-1]) == 0


@pytest.mark.parametrize("q_scale", [0.5, 2.0, -1.0])
def test_q_scale(q_scale):
    x = W.make_decode_inputs(3, 2048, [700, 2048, 1], seed=9, q_scale=q_scale)
    check_decode(run(x).double().numpy(), ref(x), f"q_scale {q_scale}")


def test_constant_v_returns_v():
    x = W.make_decode_inputs(2, 3000, [2999, 1500], seed=10)
    x.kv[:, 1] = 0.625
    got = run(x).double().numpy()
    np.testing.assert_allclose(got, 0.625, rtol=0, atol=1e-3)


def test_deterministic_and_stream_ordered():
    x = W.make_decode_inputs(8, 5000, [5000, 4321, 17, 2500, 1, 4999, 3000, 64], seed=11)
    q, kv, sl = x.q.to(DEV), x.kv.to(DEV), x.seq_lens.to(DEV)
    a = gqa.gqa_decode(q, kv, sl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = gqa.gqa_decode(q, kv, sl)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_host_buffers_match_device_path():
    x = W.make_decode_inputs(3, 1500, [1500, 700, 0], seed=12)
    dev = run(x)
    host = gqa.gqa_decode(x.q.pin_memory(), x.kv.pin_memory(), x.seq_lens.pin_memory())
    assert torch.equal(dev, host)
    pageable = gqa.gqa_decode(x.q, x.kv, x.seq_lens)
    assert torch.equal(dev, pageable)


def test_device_mismatch_rejected():
    x = W.make_decode_inputs(1, 64, [5], seed=13)
    with pytest.raises(gqa.GqaError, match="DEVICE_MISMATCH"):
        gqa.gqa_decode(x.q.to(DEV), x.kv, x.seq_lens.to(DEV))


def _sampled_check(x: W.DecodeInputs, batches, what):
    """Oracle on every head of a subset of sequences of a device-resident workload."""
    out = gqa.gqa_decode(x.q, x.kv, x.seq_lens, q_scale=x.q_scale)
    torch.cuda.synchronize()
    bs = torch.tensor(batches, device=x.q.device)
    sub = W.DecodeInputs(x.q[bs].cpu(), x.kv[bs].cpu(), x.seq_lens[bs].cpu(), x.q_scale)
    check_decode(out[bs].double().cpu().numpy(), ref(sub), what)


def test_workload_b64_cap8192_sampled():
    x = W.decode_workload("decode_b64_cap8192", device=DEV)
    lens = x.seq_lens.cpu()
    pick = sorted({int(lens.argmax()), int(lens.argmin()), 0, 17, 40, 63})
    _sampled_check(x, pick, "decode_b64_cap8192")


def test_workload_b8_cap131072_sampled():
    x = W.decode_workload("decode_b8_cap131072", device=DEV)
    assert x.kv.numel() == 2 ** 31  # 64-bit offsets exercised
    _sampled_check(x, [0, 7], "decode_b8_cap131072")
