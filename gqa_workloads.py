"""Seeded synthetic inputs for GQA decode and NVFP4 paged context attention.

This module is shared by the tests, the smoke check and the benchmark.  It
holds input generation only -- random draws, the NVFP4 *encoding* of the
synthetic K/V (how the pages are produced), and the page scatter through a
shuffled block table.  None of the attention or dequantisation arithmetic
lives here: the CUDA library and the CPU oracle each do their own.

The named workloads mirror the shapes, value distributions and
structure of the benchmark workloads this library is measured on:

* decode_b2_cap256      B=2,  cap 256,    lengths {1, 200},         seed 0
* decode_b64_cap8192    B=64, cap 8192,   lengths U{1..8192},       seed 1
* decode_b8_cap131072   B=8,  cap 131072, lengths all 131072,       seed 2, q_scale 0.5
* decode_paged_<name>   any of the above re-laid out into 64-token HND pages through a
                        shuffled block table (randperm seeded with seed + 1000)
* ctx_b4_q2048_kv2048   batch 4, q_len = kv_len = 2048,             seed 3
* ctx_b2_q4096_kv65536  batch 2, q_len 4096 ending a 65536-token KV, seed 4, out_scale 2^-6
* ctx_b2_q1_kv4096      batch 2, q_len 1 over 4096 keys,            seed 8, out_scale 2^-4
* ctx_b1_q32_kv32768    batch 1, q_len 32 over 32768 keys,          seed 9, out_scale 2^-6
* ctx_b64_q1_kv8192     batch 64, q_len 1 over 8192 keys,           seed 10, out_scale 2^-4
* ctx_b64_q8_kv8192     batch 64, q_len 8 over 8192 keys,           seed 11, out_scale 2^-4

STUDY_WORKLOADS holds shapes used only to profile the kernels (not benchmark
configurations).  The benchmark generates its inputs on the GPU (CUDA
generator, same recipe); the GPU tests of the full-size configurations use
those same device-generated inputs.

Draw order.  Decode: q, then kv, then the lengths (when random).  Context:
Q, then K, then V, then the page permutation.  All draws come from one
``torch.Generator`` on the device named by ``device`` (CPU by default), so a
workload is reproducible per device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

HQ, HKV, D, PAGE = 32, 8, 128, 64


# ----------------------------------------------------------------- decode ---

@dataclass
class DecodeInputs:
    q: torch.Tensor          # [B, 32, 128] float16
    kv: torch.Tensor         # [B, 2, 8, cap, 128] float16
    seq_lens: torch.Tensor   # [B] int32
    q_scale: float

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def capacity(self) -> int:
        return self.kv.shape[3]

    def kv_bytes_read(self) -> int:
        """K and V bytes the decode must read: sum of lengths x 8 heads x 2 x 128 x 2 B."""
        lens = self.seq_lens.clamp(0, self.capacity).to(torch.int64)
        return int(lens.sum().item()) * HKV * 2 * D * 2


def make_decode_inputs(batch: int, capacity: int, seq_lens=None, *, seed: int, q_scale: float = 1.0,
                       device="cpu", random_lens: tuple[int, int] | None = None) -> DecodeInputs:
    """q, kv ~ N(0,1) float16.  seq_lens: explicit list, or drawn U{lo..hi}."""
    g = torch.Generator(device=device).manual_seed(seed)
    q = torch.randn(batch, HQ, D, generator=g, device=device).half()
    kv = torch.empty(batch, 2, HKV, capacity, D, dtype=torch.float16, device=device)
    for b in range(batch):  # one sequence at a time bounds the fp32 temporary
        kv[b] = torch.randn(2, HKV, capacity, D, generator=g, device=device).half()
    if random_lens is not None:
        lo, hi = random_lens
        lens = torch.randint(lo, hi + 1, (batch,), generator=g, device=device).to(torch.int32)
    else:
        lens = torch.tensor(list(seq_lens), dtype=torch.int32, device=device)
    return DecodeInputs(q, kv, lens, float(q_scale))


@dataclass
class PagedDecodeInputs:
    """The stacked workload re-laid out into 64-token HND pages."""
    q: torch.Tensor            # [B, 32, 128] float16
    k_pages: torch.Tensor      # [num_pages, 8, 64, 128] float16
    v_pages: torch.Tensor
    block_table: torch.Tensor  # [B, capacity / 64] int32
    seq_lens: torch.Tensor     # [B] int32
    q_scale: float

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def capacity(self) -> int:
        return self.block_table.shape[1] * PAGE

    def kv_bytes_read(self) -> int:
        """K/V bytes the kernels read: 4096 per token (8 heads x 128 x 2 B x K,V)."""
        n = self.seq_lens.clamp(0, self.capacity).to(torch.int64).sum().item()
        return int(n) * HKV * D * 2 * 2


def page_decode_inputs(x: DecodeInputs, *, seed: int, shuffle: bool = True) -> PagedDecodeInputs:
    """Scatter a stacked decode workload into 64-token pages, physical page of
    (b, logical page p) = perm[b * (cap / 64) + p] (a randperm drawn after the
    stacked workload's draws, or the identity)."""
    B, cap = x.batch, x.capacity
    assert cap % PAGE == 0
    mp = cap // PAGE
    dev = x.q.device
    if shuffle:
        g = torch.Generator(device=dev).manual_seed(seed + 1000)
        perm = torch.randperm(B * mp, generator=g, device=dev)
    else:
        perm = torch.arange(B * mp, device=dev)
    k_pages = torch.empty(B * mp, HKV, PAGE, D, dtype=torch.float16, device=dev)
    v_pages = torch.empty_like(k_pages)
    for b in range(B):  # [8, cap, 128] -> [mp, 8, 64, 128]
        phys = perm[b * mp:(b + 1) * mp]
        k_pages[phys] = x.kv[b, 0].view(HKV, mp, PAGE, D).permute(1, 0, 2, 3)
        v_pages[phys] = x.kv[b, 1].view(HKV, mp, PAGE, D).permute(1, 0, 2, 3)
    block_table = perm.view(B, mp).to(torch.int32)
    return PagedDecodeInputs(x.q, k_pages, v_pages, block_table, x.seq_lens, x.q_scale)


# -------------------------------------------------------------- NVFP4 ctx ---

@dataclass
class CtxInputs:
    q_fp8: torch.Tensor        # [total_q, 32, 128] uint8 (E4M3 codes)
    k_fp4: torch.Tensor        # [num_pages, 8, 64, 64] uint8 (two E2M1 codes per byte)
    k_sf: torch.Tensor         # [num_pages, 8, 64, 8] uint8 (E4M3 block scales)
    v_fp4: torch.Tensor
    v_sf: torch.Tensor
    block_table: torch.Tensor  # [batch, max_pages_per_seq] int32
    qo_indptr: torch.Tensor    # [batch + 1] int32
    kv_lens: torch.Tensor      # [batch] int32
    q_scale: float
    out_scale: float

    @property
    def batch(self) -> int:
        return self.kv_lens.shape[0]

    @property
    def total_q(self) -> int:
        return self.q_fp8.shape[0]

    def page_bytes_read(self) -> int:
        """Packed K/V codes and scales of every page the sequences' visible keys
        touch, once: 64 tokens x 8 heads x (64 + 8) B per page, K and V."""
        kl = self.kv_lens.cpu().tolist()
        pages = sum((n + PAGE - 1) // PAGE for n in kl)
        return pages * PAGE * HKV * (D // 2 + D // 16) * 2

    def causal_flops(self) -> int:
        """4 * D * (visible query/key pairs) * 32 heads, bottom-right causal."""
        qi = self.qo_indptr.cpu().tolist()
        kl = self.kv_lens.cpu().tolist()
        pairs = 0
        for b in range(len(kl)):
            ql, kvl = qi[b + 1] - qi[b], kl[b]
            for_first = kvl - ql + 1  # keys seen by query 0
            # query i sees min(kv_len, max(0, kv_len - q_len + i + 1)) keys
            for i0 in range(ql):
                n = for_first + i0
                pairs += max(0, min(kvl, n))
        return 4 * D * pairs * HQ


# E2M1 magnitudes in code order 0..7.
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _encode_e2m1(y: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 code (4-bit, sign in bit 3) of each value, ties to the even
    mantissa, saturating at +-6.  Used only to *produce* synthetic pages."""
    a = y.abs()
    mags = torch.tensor(_E2M1_MAG, dtype=y.dtype, device=y.device)
    mids = (mags[1:] + mags[:-1]) / 2  # 0.25 0.75 1.25 1.75 2.5 3.5 5
    lower = torch.bucketize(a, mids, right=False)  # a == mid -> lower code
    # a tie rounds to the code with an even mantissa bit (code & 1 == 0):
    # when the lower code is odd, take the upper one.
    at_mid = torch.zeros_like(a, dtype=torch.bool)
    for k in range(7):
        at_mid |= a == mids[k]
    bump = at_mid & ((lower % 2) == 1)
    idx = lower + bump.to(lower.dtype)
    sign = (y < 0) & (idx > 0)
    return (idx | (sign.to(idx.dtype) << 3)).to(torch.uint8)


def quantize_nvfp4(x: torch.Tensor):
    """x [..., 128] float32 -> (packed [..., 64] uint8, scales [..., 8] uint8 E4M3).

    Per 16-element block: scale = E4M3(amax / 6); code = E2M1(x / scale);
    a zero scale gives zero codes.  Element 2i goes in the low nibble of byte i.
    """
    shp = x.shape[:-1]
    blocks = x.reshape(*shp, D // 16, 16)
    amax = blocks.abs().amax(dim=-1)
    sf = (amax / 6.0).to(torch.float8_e4m3fn)
    sf_val = sf.to(torch.float32)
    safe = torch.where(sf_val > 0, sf_val, torch.ones_like(sf_val))
    codes = _encode_e2m1(blocks / safe.unsqueeze(-1))
    codes = torch.where((sf_val > 0).unsqueeze(-1), codes, torch.zeros_like(codes))
    codes = codes.reshape(*shp, D)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).to(torch.uint8)
    return packed.contiguous(), sf.view(torch.uint8).contiguous()


def make_ctx_inputs(q_lens, kv_lens, *, seed: int, q_scale: float = 1.0, out_scale: float = 1.0,
                    device="cpu", shuffle: bool = True) -> CtxInputs:
    """Q ~ N(0,1) cast to E4M3; K, V ~ N(0,1) quantised to NVFP4 and scattered
    into 64-token HND pages through a (shuffled) block table."""
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    assert len(q_lens) == len(kv_lens)
    B = len(q_lens)
    g = torch.Generator(device=device).manual_seed(seed)
    total_q = sum(q_lens)
    q = torch.randn(total_q, HQ, D, generator=g, device=device).to(torch.float8_e4m3fn).view(torch.uint8)
    pages_per = [math.ceil(n / PAGE) for n in kv_lens]
    total_pages = max(1, sum(pages_per))
    max_pages = max(1, max(pages_per) if pages_per else 1)

    def draw_pages():
        fp4 = torch.zeros(total_pages, HKV, PAGE, D // 2, dtype=torch.uint8, device=device)
        sf = torch.zeros(total_pages, HKV, PAGE, D // 16, dtype=torch.uint8, device=device)
        per_seq = []
        for b in range(B):
            x = torch.randn(kv_lens[b], HKV, D, generator=g, device=device)
            per_seq.append(quantize_nvfp4(x))
        return fp4, sf, per_seq

    k_fp4, k_sf, k_seq = draw_pages()
    v_fp4, v_sf, v_seq = draw_pages()
    if shuffle:
        perm = torch.randperm(total_pages, generator=g, device=device).to(torch.int32)
    else:
        perm = torch.arange(total_pages, dtype=torch.int32, device=device)
    block_table = torch.zeros(B, max_pages, dtype=torch.int32, device=device)
    off = 0
    for b in range(B):
        n = pages_per[b]
        phys = perm[off:off + n].to(torch.int64)
        block_table[b, :n] = perm[off:off + n]
        off += n
        if n == 0:
            continue
        pad = n * PAGE - kv_lens[b]
        for (dst_fp4, dst_sf, seq) in ((k_fp4, k_sf, k_seq[b]), (v_fp4, v_sf, v_seq[b])):
            packed, sf = seq
            if pad:
                packed = torch.cat([packed, packed.new_zeros(pad, HKV, D // 2)])
                sf = torch.cat([sf, sf.new_zeros(pad, HKV, D // 16)])
            # [n*64, 8, X] -> [n, 64, 8, X] -> [n, 8, 64, X]  (HND pages)
            dst_fp4[phys] = packed.view(n, PAGE, HKV, D // 2).permute(0, 2, 1, 3)
            dst_sf[phys] = sf.view(n, PAGE, HKV, D // 16).permute(0, 2, 1, 3)
    qo = torch.tensor([0] + list(_cumsum(q_lens)), dtype=torch.int32, device=device)
    kl = torch.tensor(kv_lens, dtype=torch.int32, device=device)
    return CtxInputs(q, k_fp4, k_sf, v_fp4, v_sf, block_table, qo, kl, float(q_scale), float(out_scale))


def _cumsum(xs):
    s = 0
    for x in xs:
        s += x
        yield s


# ------------------------------------------------------ named workloads ---

DECODE_WORKLOADS = {
    "decode_b2_cap256": dict(batch=2, capacity=256, seq_lens=[1, 200], seed=0, q_scale=1.0),
    "decode_b64_cap8192": dict(batch=64, capacity=8192, random_lens=(1, 8192), seed=1, q_scale=1.0),
    "decode_b8_cap131072": dict(batch=8, capacity=131072, seq_lens=[131072] * 8, seed=2, q_scale=0.5),
}

CTX_WORKLOADS = {
    "ctx_b4_q2048_kv2048": dict(q_lens=[2048] * 4, kv_lens=[2048] * 4, seed=3, out_scale=1.0),
    # The configuration names no output scale.  2^-6 (a power of two, so the division is exact) lifts the
    # outputs -- averages over ~63 k keys of N(0,1) values, |O| ~ 5e-3, max ~ 0.03 -- into E4M3's normal
    # range; at out_scale 1 they would sit among its subnormals, where the format alone misses a 3e-2
    # relative-L2 bound.
    "ctx_b2_q4096_kv65536": dict(q_lens=[4096] * 2, kv_lens=[65536] * 2, seed=4, out_scale=2.0 ** -6),
    # the ctx page's latency-bound GB300 rows "2 x 1 x 4096" and "1 x 32 x 32768", read as
    # batch x q_len x kv_len: too few units to fill the GPU, so the KV range is split.  The rows give
    # no output scale; powers of two keep their outputs (|O| ~ 2e-2 and ~ 7e-3) in E4M3's normal range.
    "ctx_b2_q1_kv4096": dict(q_lens=[1, 1], kv_lens=[4096, 4096], seed=8, out_scale=2.0 ** -4),
    "ctx_b1_q32_kv32768": dict(q_lens=[32], kv_lens=[32768], seed=9, out_scale=2.0 ** -6),
    # decode-shaped NVFP4 calls at a realistic batch (64 sequences of 8192 keys, 1 or 8 new queries each):
    # 512 units, enough to fill the GPU without splitting the KV range; memory-bound (the page bytes)
    "ctx_b64_q1_kv8192": dict(q_lens=[1] * 64, kv_lens=[8192] * 64, seed=10, out_scale=2.0 ** -4),
    "ctx_b64_q8_kv8192": dict(q_lens=[8] * 64, kv_lens=[8192] * 64, seed=11, out_scale=2.0 ** -4),
}

# Not benchmark configurations: shapes used only to profile or study the kernels.
STUDY_WORKLOADS = {
    # one wave of 128 long units (1024 queries x 8 KV heads over 16384 keys), so that counters show
    # the steady state without per-unit start-up
    "ctx_b1_q1024_kv16384": dict(q_lens=[1024], kv_lens=[16384], seed=7),
}


def decode_workload(name: str, device="cpu"):
    """A stacked decode workload, or (decode_paged_*) the same draws re-laid
    out into pages through a shuffled block table."""
    if name.startswith("decode_paged_"):
        base = "decode_" + name[len("decode_paged_"):]
        spec = DECODE_WORKLOADS[base]
        return page_decode_inputs(make_decode_inputs(**spec, device=device), seed=spec["seed"])
    return make_decode_inputs(**DECODE_WORKLOADS[name], device=device)


def ctx_workload(name: str, device="cpu", **overrides) -> CtxInputs:
    """A named context workload (benchmark or study shape); keyword overrides
    (e.g. out_scale) replace entries of its spec."""
    spec = dict(CTX_WORKLOADS[name] if name in CTX_WORKLOADS else STUDY_WORKLOADS[name])
    spec.update(overrides)
    return make_ctx_inputs(**spec, device=device)
