"""Python binding of libgqa -- GB300 (sm_103a) grouped-query attention kernels.

Thin ctypes marshalling over the C ABI declared in ``include/gqa.h``; the
functions carry the C entry points' names.  Tensors are passed as gqa_tensor
descriptors (data pointer, dtype, device, shape, strides) to the *_t entry
points, which check dtype, shape, strides and placement in C; a rejected
call raises GqaError with the library's message.  PyTorch is used only for
device memory and the current stream: every step of the computation runs in
the library's CUDA kernels.  There is no fallback: if ``libgqa.so`` is
missing or fails to load, every call raises.

    gqa_decode(q, kv, seq_lens, *, out=None, q_scale=1.0)
    nvfp4_paged_ctx_attn(q_fp8, k_fp4, k_sf, v_fp4, v_sf, block_table, qo_indptr, kv_lens,
                         *, q_scale=1.0, out_scale=1.0, out=None)
    gqa_debug_dequant_pages(fp4, sf, block_table, kv_lens, max_kv)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "GqaError", "lib", "gqa_decode", "nvfp4_paged_ctx_attn", "gqa_debug_dequant_pages",
    "gqa_check_device_errors", "gqa_release_workspace", "gqa_decode_plan", "gqa_ctx_plan", "gqa_decode_paged", "gqa_debug_wait_expiry", "gqa_decode_noalloc", "gqa_debug_starve_producers", "gqa_set_schedule", "gqa_set_ctx_grid", "LIB_PATH",
    "build",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa.so")
HQ, HKV, D, PAGE = 32, 8, 128, 64

_STATUS = {0: "GQA_OK", 1: "GQA_ERR_INVALID_ARG", 2: "GQA_ERR_UNSUPPORTED", 3: "GQA_ERR_DEVICE_MISMATCH",
           4: "GQA_ERR_CUDA", 5: "GQA_ERR_OOM", 6: "GQA_ERR_TIMEOUT"}


class GqaTensor(ctypes.Structure):
    """gqa_tensor of include/gqa.h."""
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("device", ctypes.c_int32),
                ("ndim", ctypes.c_int32), ("shape", ctypes.c_int64 * 6), ("strides", ctypes.c_int64 * 6)]


_DTYPES = {torch.float16: 1, torch.float8_e4m3fn: 2, torch.uint8: 3, torch.int32: 4, torch.float32: 5}


def _desc(t: torch.Tensor, name: str) -> GqaTensor:
    """Descriptor of a tensor (the library checks it)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dim() > 6:
        raise ValueError(f"{name} has more than 6 dimensions")
    d = GqaTensor()
    d.data = t.data_ptr()
    d.dtype = _DTYPES.get(t.dtype, 0)
    d.device = t.device.index if t.is_cuda else -1
    d.ndim = t.dim()
    for i, (n, st) in enumerate(zip(t.shape, t.stride())):
        d.shape[i] = n
        d.strides[i] = st
    return d


class GqaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libgqa.so in-tree for sm_103a."""
    from .build_lib import build as _build
    return _build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded libgqa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libgqa.so is not built ({LIB_PATH}); call "
                                   "gqa_attention_kv_split_gb300.build() first")
            L = ctypes.CDLL(LIB_PATH)
            c = ctypes
            vp, i32p, i64, f32 = c.c_void_p, c.c_void_p, c.c_int64, c.c_float
            L.gqa_last_error.restype = c.c_char_p
            L.gqa_version.restype = c.c_int
            tp = c.POINTER(GqaTensor)
            L.gqa_decode_t.argtypes = [tp, tp, tp, tp, f32, vp]
            L.gqa_decode_t.restype = c.c_int
            L.gqa_decode_paged_t.argtypes = [tp, tp, tp, tp, tp, tp, f32, vp]
            L.gqa_decode_paged_t.restype = c.c_int
            L.nvfp4_paged_ctx_attn_t.argtypes = [tp, f32, tp, tp, tp, tp, tp, tp, tp, tp, f32, vp]
            L.nvfp4_paged_ctx_attn_t.restype = c.c_int
            L.gqa_decode.argtypes = [vp, vp, i32p, vp, i64, i64, f32, vp]
            L.gqa_decode.restype = c.c_int
            L.nvfp4_paged_ctx_attn.argtypes = [vp, f32, vp, vp, vp, vp, i32p, i32p, i32p, vp, f32,
                                               i64, i64, i64, i64, vp]
            L.nvfp4_paged_ctx_attn.restype = c.c_int
            L.gqa_debug_dequant_pages.argtypes = [vp, vp, i32p, i32p, vp, i64, i64, i64, i64, vp]
            L.gqa_debug_dequant_pages.restype = c.c_int
            L.gqa_check_device_errors.argtypes = [c.c_int, c.POINTER(c.c_uint32)]
            L.gqa_check_device_errors.restype = c.c_int
            L.gqa_decode_noalloc.argtypes = [vp, vp, i32p, vp, i64, i64, f32, vp]
            L.gqa_decode_noalloc.restype = c.c_int
            L.gqa_decode_plan.argtypes = [i64, i64, c.POINTER(c.c_int32), c.POINTER(c.c_int32),
                                          c.POINTER(c.c_int32)]
            L.gqa_decode_plan.restype = c.c_int
            L.gqa_ctx_plan.argtypes = [i64, i64, i64, c.POINTER(c.c_int32), c.POINTER(c.c_int32),
                                       c.POINTER(c.c_int32), c.POINTER(c.c_int32), c.POINTER(c.c_int32)]
            L.gqa_ctx_plan.restype = c.c_int
            L.gqa_decode_paged.argtypes = [vp, vp, vp, i32p, i32p, vp, i64, i64, i64, f32, vp]
            L.gqa_decode_paged.restype = c.c_int
            L.gqa_debug_wait_expiry.argtypes = [c.c_int, vp]
            L.gqa_debug_wait_expiry.restype = c.c_int
            L.gqa_debug_starve_producers.argtypes = [c.c_int]
            L.gqa_debug_starve_producers.restype = c.c_int
            L.gqa_set_schedule.argtypes = [c.c_int, c.c_int, c.c_int]
            L.gqa_set_schedule.restype = c.c_int
            L.gqa_set_ctx_grid.argtypes = [c.c_int]
            L.gqa_set_ctx_grid.restype = c.c_int
            L.gqa_release_workspace.argtypes = []
            L.gqa_release_workspace.restype = c.c_int
            _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise GqaError(status, lib().gqa_last_error().decode(errors="replace"))


def _stream_for(t: torch.Tensor):
    if t.is_cuda:
        return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)
    if torch.cuda.is_available():
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ctypes.c_void_p(0)


def _need(t: torch.Tensor, name: str, dtypes, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}; expected {tuple(shape)}")


def _p(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


_E4M3 = (torch.uint8, torch.float8_e4m3fn)


def _ref(d):
    return ctypes.byref(d)


def gqa_decode(q: torch.Tensor, kv: torch.Tensor, seq_lens: torch.Tensor, *, out: torch.Tensor | None = None,
               q_scale: float = 1.0) -> torch.Tensor:
    """FP16 GQA decode of one token per sequence (see include/gqa.h).

    q [B,32,128] f16, kv [B,2,8,cap,128] f16, seq_lens [B] int32, all on one
    CUDA device (asynchronous on its current stream) or all on the host
    (staged through the device, synchronous).
    """
    if out is None:
        out = torch.empty_like(q)
    ds = [_desc(q, "q"), _desc(kv, "kv"), _desc(seq_lens, "seq_lens"), _desc(out, "out")]
    _check(lib().gqa_decode_t(*map(_ref, ds), float(q_scale), _stream_for(q)))
    return out


def gqa_decode_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, block_table: torch.Tensor,
                     seq_lens: torch.Tensor, *, out: torch.Tensor | None = None, q_scale: float = 1.0) -> torch.Tensor:
    """gqa_decode over a paged K/V cache (see include/gqa.h): q [B,32,128]
    f16, k_pages / v_pages [num_pages,8,64,128] f16, block_table
    [B, max_pages_per_seq] int32, seq_lens [B] int32, all on one CUDA device
    or all on the host."""
    if out is None:
        out = torch.empty_like(q)
    ds = [_desc(q, "q"), _desc(k_pages, "k_pages"), _desc(v_pages, "v_pages"), _desc(block_table, "block_table"),
          _desc(seq_lens, "seq_lens"), _desc(out, "out")]
    _check(lib().gqa_decode_paged_t(*map(_ref, ds), float(q_scale), _stream_for(q)))
    return out


def gqa_decode_noalloc(q: torch.Tensor, kv: torch.Tensor, seq_lens: torch.Tensor, *, out: torch.Tensor,
                       q_scale: float = 1.0) -> torch.Tensor:
    """gqa_decode without any device allocation (see include/gqa.h): CUDA
    tensors only, caller-provided `out`, split partials in the library's
    16 MiB static device array."""
    B = q.shape[0]
    _need(q, "q", (torch.float16,), (B, HQ, D))
    if kv.dim() != 5:
        raise ValueError("kv must be [batch, 2, 8, capacity, 128]")
    _need(kv, "kv", (torch.float16,), (B, 2, HKV, kv.shape[3], D))
    _need(seq_lens, "sequence_lengths", (torch.int32,), (B,))
    _need(out, "out", (torch.float16,), (B, HQ, D))
    _check(lib().gqa_decode_noalloc(_p(q), _p(kv), _p(seq_lens), _p(out), B, kv.shape[3], float(q_scale),
                                    _stream_for(q)))
    return out


def nvfp4_paged_ctx_attn(q_fp8, k_fp4, k_sf, v_fp4, v_sf, block_table, qo_indptr, kv_lens, *,
                         q_scale: float = 1.0, out_scale: float = 1.0, out=None) -> torch.Tensor:
    """Paged NVFP4 context attention, bottom-right causal (see include/gqa.h).

    Returns out_fp8 [total_q,32,128] as uint8 E4M3 codes (or writes `out`).
    """
    if out is None:
        out = torch.empty((q_fp8.shape[0], HQ, D), dtype=torch.uint8, device=q_fp8.device)
    ds = [_desc(t, n) for t, n in ((q_fp8, "q_fp8"), (k_fp4, "k_fp4"), (k_sf, "k_sf"), (v_fp4, "v_fp4"),
                                   (v_sf, "v_sf"), (block_table, "block_table"), (qo_indptr, "qo_indptr"),
                                   (kv_lens, "kv_lens"), (out, "out_fp8"))]
    r = list(map(_ref, ds))
    _check(lib().nvfp4_paged_ctx_attn_t(r[0], float(q_scale), *r[1:9], float(out_scale), _stream_for(q_fp8)))
    return out


def gqa_debug_dequant_pages(fp4, sf, block_table, kv_lens, max_kv: int) -> torch.Tensor:
    """E4M3 codes [B, max_kv, 8, 128] from the context kernel's dequant routine."""
    P = fp4.shape[0]
    _need(fp4, "fp4", (torch.uint8,), (P, HKV, PAGE, D // 2))
    _need(sf, "sf", _E4M3, (P, HKV, PAGE, D // 16))
    B = kv_lens.shape[0]
    _need(block_table, "block_table", (torch.int32,))
    _need(kv_lens, "kv_lens", (torch.int32,), (B,))
    out = torch.empty((B, max_kv, HKV, D), dtype=torch.uint8, device=fp4.device)
    _check(lib().gqa_debug_dequant_pages(_p(fp4), _p(sf), _p(block_table), _p(kv_lens), _p(out), B, P,
                                         block_table.shape[1], int(max_kv), _stream_for(fp4)))
    return out


def gqa_decode_plan(batch: int, capacity: int) -> dict:
    """tokens_per_split, num_splits and num_launches of a gqa_decode call."""
    t, n, l = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib().gqa_decode_plan(int(batch), int(capacity), ctypes.byref(t), ctypes.byref(n), ctypes.byref(l)))
    return {"tokens_per_split": t.value, "num_splits": n.value, "num_launches": l.value}


def gqa_ctx_plan(batch: int, total_q: int, max_pages_per_seq: int) -> dict:
    """tiles_per_split, num_splits, num_launches and the kernel choice (persistent grid, decode-shaped
    kernel) of an nvfp4_paged_ctx_attn call."""
    t, n, l, p, d = (ctypes.c_int32() for _ in range(5))
    _check(lib().gqa_ctx_plan(int(batch), int(total_q), int(max_pages_per_seq), ctypes.byref(t), ctypes.byref(n),
                              ctypes.byref(l), ctypes.byref(p), ctypes.byref(d)))
    return {"tiles_per_split": t.value, "num_splits": n.value, "num_launches": l.value, "persistent": p.value,
            "decode_shaped": d.value}


def gqa_debug_wait_expiry(device: int = 0) -> None:
    """Launch the failure-detection check (see include/gqa.h): one wait that
    nothing completes expires after about 2 s and sets bit 0 of the error word."""
    import torch
    stream = torch.cuda.current_stream(device).cuda_stream
    _check(lib().gqa_debug_wait_expiry(int(device), ctypes.c_void_p(stream)))


def gqa_debug_starve_producers(enable: bool) -> None:
    """Test switch (see include/gqa.h): producers issue no copies, so every
    consumer's bounded wait expires (~2 s); enable=False restores normal
    operation."""
    _check(lib().gqa_debug_starve_producers(1 if enable else 0))


CTX_GRID_PLANNED, CTX_GRID_PER_UNIT, CTX_GRID_PERSISTENT, CTX_GRID_DECODE_SHAPED = 0, 1, 2, 3


def gqa_set_ctx_grid(mode: int) -> None:
    """Grid of later context calls (process-wide test switch, see
    include/gqa.h): 0 as planned, 1 one CTA per unit, 2 persistent, 3 decode-shaped."""
    _check(lib().gqa_set_ctx_grid(int(mode)))


def gqa_set_schedule(ctx_packed_stages: int = 0, ctx_kv_slots: int = 0, decode_stages: int = 0) -> None:
    """Study switch (see include/gqa.h): ring depths of later launches; 0 =
    production depth.  Raises GqaError for a depth that is not instantiated."""
    _check(lib().gqa_set_schedule(int(ctx_packed_stages), int(ctx_kv_slots), int(decode_stages)))


# the production depths first: (4, 4) for the one-CTA-per-unit context kernel, decode depth 8
CTX_SCHEDULES = [(4, 4), (6, 4), (8, 4), (10, 4), (6, 3), (12, 3), (6, 5), (6, 2)]
DECODE_SCHEDULES = [8, 4, 12, 16]


def gqa_check_device_errors(device: int = 0) -> int:
    """Synchronise `device`; return (and clear) the kernels' error word."""
    w = ctypes.c_uint32(0)
    st = lib().gqa_check_device_errors(int(device), ctypes.byref(w))
    if st not in (0, 6, 1):
        _check(st)
    return int(w.value)


def gqa_release_workspace() -> None:
    _check(lib().gqa_release_workspace())
