"""GPU parity of gqa_decode (through the C ABI) against the fp64 oracle.

Tolerance: max |err| <= 1e-2 and rel-L2 <= 2e-3 (tests/parity.py).  Cases
span one and many splits, ragged tails, empty and clamped lengths, the
shapes of the decode page's benchmark tables, and the full-size workloads
in the launch configuration the benchmark times (every sequence); and the
paged decode (gqa_decode_paged): against the oracle, bit-identical to the
stacked decode of the same draws, host buffers, a flagged bad page index."""
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


def _full_check(x: W.DecodeInputs, what):
    """Oracle on every (sequence, head) of a device-resident workload, called
    as the benchmark calls it."""
    out = gqa.gqa_decode(x.q, x.kv, x.seq_lens, q_scale=x.q_scale)
    torch.cuda.synchronize()
    host = W.DecodeInputs(x.q.cpu(), x.kv.cpu(), x.seq_lens.cpu(), x.q_scale)
    check_decode(out.double().cpu().numpy(), ref(host), what)


def test_workload_b64_cap8192_full():
    x = W.decode_workload("decode_b64_cap8192", device=DEV)
    assert gqa.gqa_decode_plan(x.batch, x.capacity)["num_launches"] == 2
    _full_check(x, "decode_b64_cap8192, all 64 sequences")


def test_workload_b8_cap131072_full():
    x = W.decode_workload("decode_b8_cap131072", device=DEV)
    assert x.kv.numel() == 2 ** 31  # 64-bit offsets exercised
    _full_check(x, "decode_b8_cap131072, all 8 sequences")
    del x
    torch.cuda.empty_cache()


# ---- paged decode ---------------------------------------------------------

def run_paged(p: W.PagedDecodeInputs, dev=DEV):
    out = gqa.gqa_decode_paged(*[t.to(dev) for t in (p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens)],
                               q_scale=p.q_scale)
    if dev is not None and dev.type == "cuda":
        torch.cuda.synchronize()
    return out.cpu()


def ref_paged(p: W.PagedDecodeInputs):
    return oracle.gqa_decode_paged(p.q.numpy(), p.k_pages.numpy(), p.v_pages.numpy(), p.block_table.numpy(),
                                   p.seq_lens.numpy(), p.q_scale)


@pytest.mark.parametrize("batch,cap,lens,seed", [
    (3, 256, [1, 200, 256], 81),                                    # one split
    (4, 4096, [4096, 1, 2999, 0], 82),                              # split + merge, empty sequence
    (6, 1000 // 64 * 64 + 64, [0, 1, 64, 65, 1000, 1024], 83),      # ragged page tails
])
def test_paged_matches_oracle(batch, cap, lens, seed):
    p = W.page_decode_inputs(W.make_decode_inputs(batch, cap, lens, seed=seed), seed=seed)
    check_decode(run_paged(p).double().numpy(), ref_paged(p), f"paged B{batch} cap{cap}")


def test_paged_is_bit_identical_to_stacked():
    """The paged kernel reads the same 16-token tiles in the same order as the
    stacked one, so the two agree bit for bit on a re-laid-out workload."""
    x = W.make_decode_inputs(5, 2048, [2048, 1, 700, 1999, 64], seed=84)
    p = W.page_decode_inputs(x, seed=84)
    assert torch.equal(run(x), run_paged(p))


def test_paged_host_buffers_match_device_path():
    p = W.page_decode_inputs(W.make_decode_inputs(2, 512, [500, 33], seed=85), seed=85)
    host = gqa.gqa_decode_paged(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, q_scale=p.q_scale)
    assert torch.equal(host, run_paged(p))


def test_paged_bad_page_index_is_flagged_not_read():
    """A table entry outside [0, num_pages) met on the device: page 0 is read
    instead and bit 1 of the error word is set (no out-of-bounds access)."""
    p = W.page_decode_inputs(W.make_decode_inputs(1, 128, [100], seed=86), seed=86)
    bt = p.block_table.clone()
    bt[0, 1] = 1 << 20
    gqa.gqa_decode_paged(p.q.to(DEV), p.k_pages.to(DEV), p.v_pages.to(DEV), bt.to(DEV), p.seq_lens.to(DEV),
                         q_scale=p.q_scale)
    assert gqa.gqa_check_device_errors(0) & 2


def test_workload_paged_b64_cap8192_bit_identical_and_sampled():
    """The benchmark's paged workload: bit-identical to the stacked decode of
    the same draws, and sampled rows against the oracle."""
    x = W.decode_workload("decode_b64_cap8192", device="cuda")
    p = W.decode_workload("decode_paged_b64_cap8192", device="cuda")
    a = gqa.gqa_decode(x.q, x.kv, x.seq_lens, q_scale=x.q_scale)
    b = gqa.gqa_decode_paged(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, q_scale=p.q_scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    seqs = [0, 17, 63]
    sub = W.PagedDecodeInputs(p.q[seqs].cpu(), p.k_pages.cpu(), p.v_pages.cpu(), p.block_table[seqs].cpu(),
                              p.seq_lens[seqs].cpu(), p.q_scale)
    check_decode(b[seqs].cpu().double().numpy(), ref_paged(sub), "decode_paged_b64_cap8192 sampled")


def test_paged_decode_host_path_checks_the_table():
    """With host buffers the library reads the lengths and the table: a used
    entry outside [0, num_pages) is rejected before anything is staged."""
    import torch
    q = torch.zeros(1, 32, 128, dtype=torch.float16)
    pages = torch.zeros(2, 8, 64, 128, dtype=torch.float16)
    bt = torch.tensor([[0, 5]], dtype=torch.int32)       # page 5 does not exist
    with pytest.raises(gqa.GqaError, match="block_table"):
        gqa.gqa_decode_paged(q, pages, pages, bt, torch.tensor([100], dtype=torch.int32))


def test_bounded_waits_expire_in_the_decode_kernels():
    """Failure detection in the real kernels: producers starved (each wait
    expires after ~2 s); the stacked and the paged decode (split + merge, and a single
    split) report GQA_ERR_TIMEOUT, and the next normal calls are correct."""
    import time
    x = W.make_decode_inputs(4, 4096, [4096, 100, 0, 3000], seed=14)
    x1 = W.make_decode_inputs(2, 256, [1, 200], seed=15)
    p = W.page_decode_inputs(x, seed=14)
    assert gqa.gqa_decode_plan(4, 4096)["num_launches"] == 2 and gqa.gqa_decode_plan(2, 256)["num_launches"] == 1
    assert gqa.gqa_check_device_errors(0) == 0
    words = []
    gqa.gqa_debug_starve_producers(True)
    try:
        t0 = time.perf_counter()
        for case in (x, x1):
            gqa.gqa_decode(case.q.to(DEV), case.kv.to(DEV), case.seq_lens.to(DEV), q_scale=case.q_scale)
            words.append(gqa.gqa_check_device_errors(0))
        run_paged(p)
        words.append(gqa.gqa_check_device_errors(0))
        took = time.perf_counter() - t0
    finally:
        gqa.gqa_debug_starve_producers(False)
    assert all(w & 1 for w in words), words
    assert took < 60
    check_decode(run(x).double().numpy(), ref(x), "decode after expired waits")
    check_decode(run(x1).double().numpy(), ref(x1), "single split after expired waits")
    check_decode(run_paged(p).double().numpy(), ref_paged(p), "paged decode after expired waits")
    assert gqa.gqa_check_device_errors(0) == 0


def test_bounded_wait_expires_and_is_reported():
    """Failure detection without a fault: a wait that nothing completes gives
    up after ~2 s, the host reads GQA_ERR_TIMEOUT (bit 0), and the context is
    still usable afterwards."""
    import time
    assert gqa.gqa_check_device_errors(0) == 0
    t0 = time.perf_counter()
    gqa.gqa_debug_wait_expiry(0)
    word = gqa.gqa_check_device_errors(0)   # synchronises; returns and clears the word
    took = time.perf_counter() - t0
    assert word & 1 and 1.5 < took < 30
    assert gqa.gqa_check_device_errors(0) == 0
    x = W.decode_workload("decode_b2_cap256")
    check_decode(run(x).double().numpy(), ref(x), "decode after an expired wait")
