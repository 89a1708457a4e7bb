"""fp64 CPU oracle for GQA decode and NVFP4 paged context attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference legs of ``bench.py`` may import this package.  The
product library never loads it, and it shares no code with the CUDA path: the
arithmetic lives in ``gqa_oracle.c`` (plain C, fp64), compiled here with gcc
and called through ctypes on numpy arrays.

What each function computes, and the passage it follows, is stated in the C
source beside it.  In short:

* ``f16_to_f64`` / ``e4m3_to_f64`` / ``e2m1_to_f64`` / ``f64_to_e4m3`` -- the
  number formats from their bit definitions.
* ``gqa_decode`` -- softmax(q K^T * q_scale / sqrt(128)) V per query head,
  KV head = query head // 4 ("NVIDIA SM110 GPU를 위한 실험적인 FP16 GQA 디코드
  커널 추가", sections 1 and 3).
* ``dequant_pages`` -- NVFP4 page -> E4M3 tiles through the block table
  ("GB300 NVFP4 Context Attention ...", introduction).
* ``nvfp4_paged_ctx_attn`` -- bottom-right causal attention over the
  dequantised pages, result O / out_scale (same page, introduction).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgqa_oracle.so")
_lock = threading.Lock()
_lib = None

HQ, HKV, D, PAGE = 32, 8, 128, 64


def build(force: bool = False) -> str:
    """Compile gqa_oracle.c into libgqa_oracle.so (gcc, no GPU needed)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            c = ctypes
            lib.oracle_f16_to_f64.argtypes = [c.c_uint16]
            lib.oracle_f16_to_f64.restype = c.c_double
            lib.oracle_e4m3_to_f64.argtypes = [c.c_uint8]
            lib.oracle_e4m3_to_f64.restype = c.c_double
            lib.oracle_e2m1_to_f64.argtypes = [c.c_uint8]
            lib.oracle_e2m1_to_f64.restype = c.c_double
            lib.oracle_f64_to_e4m3_rne_sat.argtypes = [c.c_double]
            lib.oracle_f64_to_e4m3_rne_sat.restype = c.c_uint8
            p = c.c_void_p
            i64 = c.c_int64
            lib.oracle_gqa_decode.argtypes = [p, p, p, i64, i64, c.c_double, p, i64, p, c.c_int]
            lib.oracle_gqa_decode.restype = c.c_int
            lib.oracle_dequant_pages.argtypes = [p, p, p, i64, p, i64, i64, p]
            lib.oracle_dequant_pages.restype = c.c_int
            lib.oracle_nvfp4_paged_ctx_attn.argtypes = [
                p, c.c_double, p, p, p, p, p, i64, p, p, i64, c.c_double, p, i64, p, c.c_int]
            lib.oracle_nvfp4_paged_ctx_attn.restype = c.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    """Host cores available to this process."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


# ---------------------------------------------------------------- formats ---

def f16_to_f64(codes) -> np.ndarray:
    lib = _load()
    codes = np.asarray(codes, dtype=np.uint16)
    return np.array([lib.oracle_f16_to_f64(int(c)) for c in codes.ravel()]).reshape(codes.shape)


def e4m3_to_f64(codes) -> np.ndarray:
    lib = _load()
    codes = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_to_f64(int(c)) for c in codes.ravel()]).reshape(codes.shape)


def e2m1_to_f64(nibbles) -> np.ndarray:
    lib = _load()
    nibbles = np.asarray(nibbles, dtype=np.uint8)
    return np.array([lib.oracle_e2m1_to_f64(int(c)) for c in nibbles.ravel()]).reshape(nibbles.shape)


def f64_to_e4m3(values) -> np.ndarray:
    """E4M3 code of each value: round to nearest even, saturate to +-448."""
    lib = _load()
    values = np.asarray(values, dtype=np.float64)
    return np.array([lib.oracle_f64_to_e4m3_rne_sat(float(v)) for v in values.ravel()],
                    dtype=np.uint8).reshape(values.shape)


_E4M3_TABLE = None


def e4m3_table() -> np.ndarray:
    """fp64 value of each of the 256 E4M3 codes (from the oracle's decoder)."""
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        _E4M3_TABLE = e4m3_to_f64(np.arange(256, dtype=np.uint8))
    return _E4M3_TABLE


# ----------------------------------------------------------------- decode ---

def gqa_decode(q_f16, kv_f16, seq_lens, q_scale: float = 1.0, items=None, threads: int | None = None):
    """fp64 decode attention.

    q_f16: [B,32,128] float16 (or its uint16 bits); kv_f16: [B,2,8,cap,128];
    seq_lens: [B] int32.  items: None (returns [B,32,128]) or an [n,2] array of
    (b, h) pairs (returns [n,128]).
    """
    lib = _load()
    q = _c(np.asarray(q_f16).view(np.uint16) if np.asarray(q_f16).dtype == np.float16 else q_f16, np.uint16)
    kv = _c(np.asarray(kv_f16).view(np.uint16) if np.asarray(kv_f16).dtype == np.float16 else kv_f16, np.uint16)
    sl = _c(seq_lens, np.int32)
    B = q.shape[0]
    assert q.shape == (B, HQ, D) and kv.shape[:3] == (B, 2, HKV) and kv.shape[4] == D and sl.shape == (B,)
    cap = kv.shape[3]
    if items is None:
        out = np.zeros((B, HQ, D), dtype=np.float64)
        it, n = None, 0
    else:
        it = _c(items, np.int64).reshape(-1, 2)
        n = it.shape[0]
        out = np.zeros((n, D), dtype=np.float64)
    rc = lib.oracle_gqa_decode(_ptr(q), _ptr(kv), _ptr(sl), B, cap, float(q_scale),
                               None if it is None else _ptr(it), n, _ptr(out),
                               threads or default_threads())
    assert rc == 0
    return out


def gqa_decode_paged(q_f16, k_pages, v_pages, block_table, seq_lens, q_scale: float = 1.0, items=None,
                     threads: int | None = None):
    """fp64 decode attention over a paged K/V cache: the decode of the SM110
    FP16 GQA decode page (section 1) with K/V held in 64-token HND pages
    ("GB300 NVFP4 Context Attention ...", introduction, for the layout).
    Token t of sequence b is slot t % 64 of page block_table[b, t // 64],
    KV head g of that page; the sequence's tokens are gathered into the
    stacked [B, 2, 8, cap, 128] cache (cap = 64 * table width) and go through
    gqa_decode above.

    k_pages, v_pages: [num_pages, 8, 64, 128] float16 (or uint16 bits);
    block_table: [B, max_pages] int32; seq_lens: [B] int32.
    """
    kp = np.asarray(k_pages)
    vp = np.asarray(v_pages)
    kp = kp.view(np.uint16) if kp.dtype == np.float16 else kp
    vp = vp.view(np.uint16) if vp.dtype == np.float16 else vp
    bt = np.asarray(block_table).astype(np.int64)
    sl = np.asarray(seq_lens).astype(np.int32)
    B, mp = bt.shape
    cap = mp * 64
    kv = np.zeros((B, 2, HKV, cap, D), dtype=np.uint16)
    for b in range(B):
        n = min(max(int(sl[b]), 0), cap)
        for p in range((n + 63) // 64):
            pg = bt[b, p]
            kv[b, 0, :, 64 * p:64 * p + 64, :] = kp[pg]  # [8, 64, 128]: head, slot, d
            kv[b, 1, :, 64 * p:64 * p + 64, :] = vp[pg]
    return gqa_decode(q_f16, kv, sl, q_scale, items=items, threads=threads)


# ------------------------------------------------------------------- ctx ---

def dequant_pages(fp4_pages, sf_pages, block_table, kv_lens, max_kv: int | None = None) -> np.ndarray:
    """E4M3 codes [B, max_kv, 8, 128] of each sequence's dequantised tokens."""
    lib = _load()
    fp4 = _c(fp4_pages, np.uint8)
    sf = _c(sf_pages, np.uint8)
    bt = _c(block_table, np.int32)
    kl = _c(kv_lens, np.int32)
    B = kl.shape[0]
    if max_kv is None:
        max_kv = int(kl.max()) if B else 0
    out = np.zeros((B, max_kv, HKV, D), dtype=np.uint8)
    rc = lib.oracle_dequant_pages(_ptr(fp4), _ptr(sf), _ptr(bt), bt.shape[1], _ptr(kl), B, max_kv, _ptr(out))
    assert rc == 0
    return out


def nvfp4_paged_ctx_attn(q_fp8, q_scale, k_fp4, k_sf, v_fp4, v_sf, block_table, qo_indptr, kv_lens,
                         out_scale: float = 1.0, items=None, threads: int | None = None) -> np.ndarray:
    """fp64 O / out_scale.  q_fp8: [total_q,32,128] E4M3 codes (uint8).

    items: None (returns [total_q,32,128]) or an [n,2] array of (row, head)
    pairs (returns [n,128]).
    """
    lib = _load()
    q = _c(q_fp8, np.uint8)
    kf, ks, vf, vs = (_c(a, np.uint8) for a in (k_fp4, k_sf, v_fp4, v_sf))
    bt = _c(block_table, np.int32)
    qi = _c(qo_indptr, np.int32)
    kl = _c(kv_lens, np.int32)
    B = kl.shape[0]
    total_q = int(qi[-1])
    if items is None:
        out = np.zeros((total_q, HQ, D), dtype=np.float64)
        it, n = None, 0
    else:
        it = _c(items, np.int64).reshape(-1, 2)
        n = it.shape[0]
        out = np.zeros((n, D), dtype=np.float64)
    rc = lib.oracle_nvfp4_paged_ctx_attn(
        _ptr(q), float(q_scale), _ptr(kf), _ptr(ks), _ptr(vf), _ptr(vs), _ptr(bt), bt.shape[1],
        _ptr(qi), _ptr(kl), B, float(out_scale), None if it is None else _ptr(it), n, _ptr(out),
        threads or default_threads())
    if rc != 0:
        raise MemoryError("oracle could not hold the dequantised pages")
    return out
