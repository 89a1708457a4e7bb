"""gqa_decode_noalloc: the decode entry point that allocates no device memory.

Some callers cannot allocate at call time -- an inference engine that has
reserved nearly all of HBM for its own KV cache and owns every byte through
its allocator, or a latency-critical loop that must not block in
cudaMalloc/cudaFree (both can synchronise the device).  For them the library
keeps the split partials in a fixed 16 MiB device array.  This test calls the
entry point through the C ABI and checks it against gqa_decode, on two calls
in a row with different shapes (the second call reuses the array the first
one left behind), and checks the size limit and the device-only rule.

Collected last on purpose, so that a stop-at-first-failure run has already
run every other test; it is also self-contained for a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import gqa_attention_kv_split_gb300 as gqa
import gqa_workloads as W
from parity import DECODE_MAX_ABS, DECODE_REL_L2, rel_l2

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
UNSUPPORTED = 2


@pytest.fixture(scope="module")
def L():
    gqa.build()
    return gqa.lib()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(L, x, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return L.gqa_decode_noalloc(_ptr(x.q), _ptr(x.kv), _ptr(x.seq_lens), _ptr(out), x.batch, x.capacity,
                                x.q_scale, stream)


def test_matches_gqa_decode_on_two_calls_in_a_row(L):
    cases = [
        W.make_decode_inputs(16, 3000, None, seed=41, random_lens=(1, 3000), device=DEV),
        W.make_decode_inputs(4, 20000, [20000, 1, 9999, 15000], seed=42, q_scale=0.5, device=DEV),
    ]
    for x in cases:
        assert gqa.gqa_decode_plan(x.batch, x.capacity)["num_splits"] > 1  # the partials are used
        out = torch.empty_like(x.q)
        assert _noalloc(L, x, out) == 0, L.gqa_last_error()
        ref = gqa.gqa_decode(x.q, x.kv, x.seq_lens, q_scale=x.q_scale)
        torch.cuda.synchronize()
        a = out.double().cpu().numpy()
        b = ref.double().cpu().numpy()
        assert np.isfinite(a).all()
        assert np.abs(a - b).max() <= DECODE_MAX_ABS
        assert rel_l2(a, b) <= DECODE_REL_L2


def test_rejects_sizes_beyond_the_static_scratch(L):
    # 64 x 65536 needs 64 * 32 * 16 splits * 520 B = 17.0 MB of partials > 16 MiB.
    B, cap = 64, 65536
    assert B * 32 * gqa.gqa_decode_plan(B, cap)["num_splits"] * 520 > (16 << 20)
    q = torch.zeros(B, 32, 128, dtype=torch.float16, device=DEV)
    kv = torch.empty(B, 2, 8, cap, 128, dtype=torch.float16, device=DEV)  # never read
    lens = torch.zeros(B, dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    x = W.DecodeInputs(q, kv, lens, 1.0)
    assert _noalloc(L, x, out) == UNSUPPORTED
    assert b"static scratch" in L.gqa_last_error()
    del kv
    torch.cuda.empty_cache()


def test_rejects_host_buffers(L):
    x = W.make_decode_inputs(2, 64, [3, 64], seed=43)
    out = torch.empty_like(x.q)
    assert _noalloc(L, x, out) == UNSUPPORTED
    assert b"device pointers only" in L.gqa_last_error()
