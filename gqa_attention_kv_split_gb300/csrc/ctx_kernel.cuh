// ctx_kernel.cuh -- the NVFP4 paged context (prefill) attention kernel for
// sm_103a, as a template over the split-KV mode and the depths of its two
// shared-memory rings (so that ring depths can be studied against one
// another; every instance computes the same result, bit for bit).
//
// Operation ("GB300 NVFP4 Context Attention: scale slot 조기 반납과 8단 packed
// K/V ring", introduction): FP8-E4M3 query and output, NVFP4 K/V pages in HND
// layout with E4M3 block scales, dequantised to E4M3 in shared memory, head
// dim 128, bottom-right causal mask.  For sequence b, query i sees key j iff
// j <= kv_len - q_len + i;  O = softmax(q K^T * q_scale / sqrt(128)) V, and
// out = E4M3(O / out_scale).
//
// Design (the page's Cake schedule -- 512 threads, 8-stage packed ring, early
// scale-slot release -- is prior art; this is our own GB300 layout):
//  * Work unit = (sequence b, KV head g, block of 64 queries).  The 4 query
//    heads of the group are stacked into the MMA's M dimension: M-tile T
//    (T = 0, 1) holds queries 32T..32T+31 of the block x 4 heads, row
//    r = 4 * query + head.  One dequantised K/V tile therefore feeds 256 rows.
//  * KV tiles of 64 keys (one page).  TMEM (512 columns) per M-tile T: two
//    S buffers (64 f32 columns each, tile j in buffer j & 1) and O (128
//    columns).  The softmax writes P of tile j (64 f16 weights per row = 32
//    columns) over the first half of the S buffer it read, and P V reads it
//    there as its TMEM A operand.  So S of tile j+1 is computed into the
//    other buffer while the softmax works on tile j; S of tile j+2 waits
//    only for the P V of tile j, the last reader of its buffer.
//  * Warp roles (16 warps): 0 = bulk-copy producer of packed NVFP4 pages +
//    scales through the block table into a kNP-stage ring; 1 and 3 = issuers
//    of S = Q K^T for M-tile 0 and 1 (warp 1 also owns the TMEM allocation);
//    2 = Q loader (two TMA boxes through a 128-byte-swizzling tensor map),
//    then issuer of O += P V for both M-tiles; 4-7 and 8-11 = softmax of
//    M-tile 0 and 1 (one thread per TMEM lane = row); 12-15 = dequantisers
//    writing the K tile (E4M3) and the V tile (its E4M3 values as f16) into
//    kNK slots, in the 128-byte swizzled layouts the MMA descriptors read (K
//    as the K-major B operand of S = Q K^T, V as the MN-major B operand of
//    O = P V).
//  * Online softmax in the exp2 domain with a lazy running maximum m: m is
//    raised only when a row's maximum exceeds it by more than 2^8, so O is
//    rescaled rarely.
//  * S = Q K^T is an FP8 (E4M3 x E4M3) product.  P V is an F16 product: P is
//    rounded to f16 (11 significant bits) and V's dequantised E4M3 values
//    are widened to f16 exactly.  A one-term E4M3 P carries ~2 % relative
//    error per weight, which puts ~3 % of the outputs more than 2 E4M3 ulps
//    from the exact result.
//  * Split-KV (kSplit): when the units cannot fill the GPU (short query
//    lengths, few sequences), grid.y divides each unit's KV tiles into
//    contiguous ranges; each range writes its unnormalised O and (m, l) in
//    f32, and a merge kernel, launched as a programmatic dependent grid,
//    combines them by their maxima.  A unit whose queries all lie in M-tile
//    0 leaves M-tile 1 idle in both modes.
//  * Robustness: every wait is bounded (2 s); a thread whose wait expires
//    records it in the error word and leaves its loop, and the CTA then
//    drains the MMAs and bulk copies it issued before it frees TMEM.
//    qo_indptr is validated on the device (error bit kErrBadIndptr); no load
//    or store leaves [0, total_q) whatever its values.  (The checks cost
//    ~1-2 % against the same kernel without them.)
#pragma once
#include <cuda.h>  // CUtensorMap
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "nvfp4.cuh"
#include "tcgen05.cuh"

namespace gqa {
namespace ctx {

constexpr int kQB = 64;                       // queries per work unit
constexpr int kQT = 32;                       // queries per M=128 tile (x 4 heads)
constexpr int kKT = 64;                       // keys per KV tile (one page)
constexpr int kThreads = 512;
constexpr int kQTile = 128 * 128;             // one M-tile of Q, E4M3: 16 KB
constexpr int kKVTile = kKT * 128;            // one K tile, E4M3: 8 KB
constexpr int kVHalf = kKT * 64 * 2;          // one V tile half (64 of the 128 d), F16: 8 KB
constexpr int kPackedPage = kPage * kD / 2;   // 4 KB of codes per (page, KV head)
constexpr int kScalePage = kPage * kD / 16;   // 512 B of scales per (page, KV head)
constexpr float kRescaleLog2 = 8.f;           // lazy-maximum threshold when a row's maximum is recomputed
constexpr float kMaxTileSum = 32768.f;        // a tile's row sum of P up to which no P can overflow f16
constexpr uint32_t kTmemCols = 512;
// TMEM columns of M-tile T, from T * 256: two S/P buffers (64 f32 columns of
// S each, tile j in buffer j & 1; P of the tile, as f16 pairs, overwrites the
// buffer's first 32 columns), then O (128 columns).
constexpr uint32_t kTmemPerTile = 256;
constexpr uint32_t kTmemSP = 64;  // columns per S/P buffer
constexpr uint32_t kTmemO = 128;
// Ring depths of the production instances (packed-page stages, dequantised
// K/V slots), chosen by the ring-depth study (interleaved timing, outputs
// byte-identical at every depth): the one-CTA-per-unit kernel of unsplit
// calls runs 4 stages (1.6-2.4 % ahead of 6 on long units); the persistent
// grid (0.9 % ahead at 6) and split-KV calls (no difference) run 6.
constexpr int kCtxStagesDefault = 4;
constexpr int kCtxStagesPersistent = 6;
constexpr int kCtxStagesSplit = 6;
constexpr int kCtxSlotsDefault = 4;

// Error word of the context kernels of one translation unit (bitwise OR of
// the kErr* codes); read and cleared by the host.
static __device__ uint32_t g_ctx_err;

template <int kNP, int kNK>
struct Smem {
  uint8_t q[2][kQTile];             // M-tiles 0/1 of Q (128B-swizzled, K-major A operand)
  uint8_t k[kNK][kKVTile];          // E4M3 K tiles (128B-swizzled, K-major B operand of S = Q K^T)
  uint8_t v[kNK][2 * kVHalf];       // V tiles as F16 (128B-swizzled, MN-major B operand of O += P V)
  uint8_t pk[kNP][2][kPackedPage];  // [stage][K=0,V=1][slot*64 + byte]
  uint8_t sf[kNP][2][kScalePage];   // [stage][K,V][slot*8 + block]
  uint64_t pk_full[kNP], pk_empty[kNP];
  uint64_t kv_ready[kNK], kv_free[kNK];   // dequantised K and V of a slot written / slot consumed
  uint64_t s_full[2][2];                  // [M-tile][buffer]: S computed
  uint64_t p_full[2][2], p_free[2][2];    // [M-tile][buffer]: P written / the P V that read it completed
  uint64_t q_ready, o_final[2];           // Q loaded; every MMA of M-tile T complete
  uint64_t drain[3];                // teardown after an expired wait: MMAs of issuer warps 1..3 complete
  uint2 ktab[256];                  // E4M3 magnitudes of the 8 E2M1 codes for every scale byte (K and V)
  uint32_t tmem_base;
  int unit_b, unit_qb;
};

template <int kNP, int kNK>
constexpr size_t smem_bytes() {
  return sizeof(Smem<kNP, kNK>) + 1024;  // + alignment slack
}

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a 128B-swizzled tile
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

// Query length of sequence b, clamped to [0, total_q] in 64-bit arithmetic
// (meaningless offsets must not overflow or index outside the output).
__device__ __forceinline__ int q_len_of(const int32_t* __restrict__ qo, int b, int64_t total_q) {
  int64_t d = (int64_t)qo[b + 1] - (int64_t)qo[b];
  d = d < 0 ? 0 : (d > total_q ? total_q : d);
  return (int)d;
}

// Work index t -> (b, query block), longest first: rounds r = 0, 1, ...; in
// round r every sequence with more than r query blocks contributes its block
// (n_blocks - 1 - r), in batch order.  All lanes of the calling warp get the
// same answer; b = -1 when t is past the last unit.
static __device__ void find_unit(const int32_t* __restrict__ qo, int B, int64_t total_q, int t, int& out_b,
                          int& out_qb) {
  const int lane = threadIdx.x & 31;
  out_b = -1;
  out_qb = -1;
  int nqb0 = 0;  // blocks of sequence lane, read once (the rounds below reuse it)
  if (lane < B) nqb0 = (q_len_of(qo, lane, total_q) + kQB - 1) / kQB;
  for (int r = 0;; ++r) {
    int cnt = 0;
    bool any = false;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int nqb = nqb0;
      if (b0 > 0) nqb = b < B ? (q_len_of(qo, b, total_q) + kQB - 1) / kQB : 0;
      const unsigned bal = __ballot_sync(0xffffffffu, nqb > r);
      const int c = __popc(bal);
      if (t >= cnt && t < cnt + c) {
        unsigned m = bal;
        for (int i = 0; i < t - cnt; ++i) m &= m - 1;  // drop the lower set bits
        const int bb = b0 + __ffs(m) - 1;
        out_b = bb;
        out_qb = (q_len_of(qo, bb, total_q) + kQB - 1) / kQB - 1 - r;
        return;
      }
      cnt += c;
      any |= (bal != 0u);
    }
    if (!any) return;
    t -= cnt;
  }
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// 2^x on two f16 values at once (relative error below 2^-9).
__device__ __forceinline__ uint32_t ex2_h2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t hadd2_u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Sum of the two halves of an f16x2 word, in f32.
__device__ __forceinline__ float h2_sum_f32(uint32_t h) {
  const __half2 v = *reinterpret_cast<const __half2*>(&h);
  return __low2float(v) + __high2float(v);
}
// Two floats -> f16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Four floats -> four E4M3 bytes (e0 in the low byte), round to nearest
// even, saturating to +-448: two hardware conversions of two values each
// (the first source operand lands in the upper byte).
__device__ __forceinline__ uint32_t f4_to_e4m3x4(float e0, float e1, float e2, float e3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(e0), "f"(e1), "f"(e2), "f"(e3));
  return r;
}

// 3-D tiled TMA load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

template <bool kSplit, int kNP, int kNK>
__global__ void __launch_bounds__(kThreads, 1)
    ctx_nvfp4_kernel(const __grid_constant__ CtxArgs a, const __grid_constant__ CUtensorMap q_map, const float scale_log2,
                     const float inv_out_scale, const int tiles_per_split, float* __restrict__ part_o,
                     float2* __restrict__ part_ml) {
  static_assert(kNK >= 2 && kNP >= 2, "rings need at least two slots");
  using SM = Smem<kNP, kNK>;
  extern __shared__ uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.x % kHkv;
  const int B = (int)a.batch;

  if (warp == 0) {
    int ub, uqb;
    find_unit(a.qo_indptr, B, a.total_q, (int)(blockIdx.x / kHkv), ub, uqb);
    if (lane == 0) {
      sm.unit_b = ub;
      sm.unit_qb = uqb;
    }
  } else if (warp == 2 && blockIdx.y == 0) {
    // Metadata check (beside the unit lookup, not before it): CTA x checks
    // sequences [32 x, 32 x + 32) (grid.x >= batch / 32 always), CTA 0 the ends.
    const int64_t bq = (int64_t)blockIdx.x * 32 + lane;
    bool bad = bq < B && a.qo_indptr[bq + 1] < a.qo_indptr[bq];
    if (blockIdx.x == 0 && lane == 0) bad |= a.qo_indptr[0] != 0 || (int64_t)a.qo_indptr[B] != a.total_q;
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&g_ctx_err, kErrBadIndptr);
  } else if (warp == 3 && !kSplit && blockIdx.x == 0) {
    // Rows past the last offset belong to no unit: they are written as zeros
    // (only when qo_indptr is invalid; in split mode the merge does this).
    const int64_t last = a.qo_indptr[B];
    if (last < a.total_q) {
      const int64_t r0 = last > 0 ? last : 0;
      uint4* o = reinterpret_cast<uint4*>(a.out + r0 * kHq * kD);
      const int64_t n16 = (a.total_q - r0) * (kHq * kD / 16);
      for (int64_t i = lane; i < n16; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) {
    sm.ktab[i] = nvfp4_scale_table((uint32_t)i);
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < kNP; ++i) {
      mbar_init(smem_u32(&sm.pk_full[i]), 1);
      mbar_init(smem_u32(&sm.pk_empty[i]), 4);
    }
    for (int i = 0; i < kNK; ++i) {
      mbar_init(smem_u32(&sm.kv_ready[i]), 4);
      mbar_init(smem_u32(&sm.kv_free[i]), 3);  // S of both M-tiles, P V of both
    }
    for (int t = 0; t < 2; ++t) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(smem_u32(&sm.s_full[t][i]), 1);
        mbar_init(smem_u32(&sm.p_full[t][i]), 4);
        mbar_init(smem_u32(&sm.p_free[t][i]), 1);
      }
      mbar_init(smem_u32(&sm.o_final[t]), 1);
    }
    mbar_init(smem_u32(&sm.q_ready), 1);
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&sm.drain[i]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int b = sm.unit_b;
  if (b < 0) return;  // past the last unit: the whole CTA leaves
  const int qb = sm.unit_qb;
  const int64_t qo = a.qo_indptr[b];
  const int q_len = q_len_of(a.qo_indptr, b, a.total_q);
  int kv_len = a.kv_lens[b];
  const int kv_cap = (int)(a.max_pages_per_seq * kPage);
  kv_len = kv_len < 0 ? 0 : (kv_len > kv_cap ? kv_cap : kv_len);
  const int q0 = qb * kQB;
  const int q_last = min(q0 + kQB, q_len) - 1;
  const int n_keys = min(kv_len, kv_len - q_len + q_last + 1);
  const int unit_tiles = n_keys > 0 ? (n_keys + kKT - 1) / kKT : 0;
  // Split-KV (kSplit): this CTA takes the unit's tiles
  // [t_begin, t_begin + tiles_per_split) and writes partial results.  Loop
  // indices j below are local (tile t_begin + j); the ring and barrier
  // phases count local tiles.
  const int t_begin = kSplit ? (int)blockIdx.y * tiles_per_split : 0;
  const int n_tiles = kSplit ? max(0, min(unit_tiles - t_begin, tiles_per_split)) : unit_tiles;
  // M-tile 1 holds queries q0 + 32 .. q0 + 63; when none of them exists (a
  // sequence's last block of at most 32 queries) it is not computed: its S
  // issuer only releases the K/V slots and its softmax warps stay idle.
  const bool t1_live = q0 + kQT < q_len;

  if (warp == 1) {
    tc::tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const uint32_t tmem = sm.tmem_base;
  auto wait_all = [](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, &g_ctx_err));
  };
  int issued = 0;       // producer: pages whose copies were issued
  bool failed = false;  // a wait of this thread's role expired

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // One page per KV tile: packed K and V codes (4 KB each) and their scales
    // (512 B each) through the block table.  The page numbers are read 32 at
    // a time by the whole warp, one chunk ahead of use, so no copy waits for
    // a block-table read; lane 0 issues the copies.  (a.starve: a test of the
    // bounded waits -- no copy is issued, so every consumer's wait expires.)
    if (n_tiles > 0 && !a.starve) {
      const uint64_t pol = policy_evict_last();  // pages are re-read by the other query blocks
      const int32_t* bt = a.block_table + (int64_t)b * a.max_pages_per_seq + t_begin;
      int cur = lane < n_tiles ? bt[lane] : 0;
      int nxt = 32 + lane < n_tiles ? bt[32 + lane] : 0;
      for (int j = 0; j < n_tiles; ++j) {
        if (j > 0 && (j & 31) == 0) {
          cur = nxt;
          nxt = j + 32 + lane < n_tiles ? bt[j + 32 + lane] : 0;
        }
        int phys = __shfl_sync(0xffffffffu, cur, j & 31);
        const int st = j % kNP;
        if (j >= kNP && !wait_all(&sm.pk_empty[st], ((j / kNP) - 1) & 1)) {
          failed = true;
          break;
        }
        if (lane == 0) {
          if (phys < 0 || phys >= a.num_pages) {
            atomicOr(&g_ctx_err, kErrBadIndex);
            phys = 0;
          }
          const int64_t row = ((int64_t)phys * kHkv + g) * kPage;
          const uint32_t fb = smem_u32(&sm.pk_full[st]);
          mbar_arrive_expect_tx(fb, 2u * (kPackedPage + kScalePage));
          bulk_g2s_hint(smem_u32(sm.pk[st][0]), a.k_fp4 + row * (kD / 2), kPackedPage, fb, pol);
          bulk_g2s_hint(smem_u32(sm.sf[st][0]), a.k_sf + row * (kD / 16), kScalePage, fb, pol);
          bulk_g2s_hint(smem_u32(sm.pk[st][1]), a.v_fp4 + row * (kD / 2), kPackedPage, fb, pol);
          bulk_g2s_hint(smem_u32(sm.sf[st][1]), a.v_sf + row * (kD / 16), kScalePage, fb, pol);
        }
        issued = j + 1;
        __syncwarp();
      }
    }
  } else if (warp == 1 || warp == 3) {
    // -------------------------------------------------------- S issuers
    // Warp 1 issues S = Q K^T of M-tile 0, warp 3 that of M-tile 1: S_T(j)
    // into buffer j & 1 once K/V of tile j are dequantised and P V_T(j-2),
    // which read P_T(j-2) from that buffer, has completed (p_free), so S of
    // the next tile is computed while the softmax works on this one.  Waiting
    // for that P V also orders this S after the softmax's reads of S_T(j-2)
    // and its writes of P_T(j-2).  tcgen05.mma issue blocks while the tensor
    // pipe is busy, so S and P V have separate issuing warps and an S is
    // never queued behind a P V the softmax is not waiting for.  The whole
    // warp runs this code (descriptor arithmetic stays warp-uniform, which
    // keeps it in the uniform datapath the MMA reads); one elected lane
    // issues each MMA and commit.
    const int T = warp == 1 ? 0 : 1;
    if (n_tiles > 0) {
      constexpr uint32_t idS = tc::idesc_e4m3_f32(128, kKT, false);  // B = K tile, K-major
      const uint64_t dq = tc::sw128_desc(smem_u32(sm.q[T]));
      const uint64_t dk0 = tc::sw128_desc(smem_u32(sm.k[0]));
      const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0) + (uint32_t)T * kTmemPerTile;
      bool ok = wait_all(&sm.q_ready, 0);
      if (T == 1 && !t1_live) {
        for (int j = 0; ok && j < n_tiles; ++j) {
          ok = wait_all(&sm.kv_ready[j % kNK], (j / kNK) & 1);
          if (ok && lane == 0) mbar_arrive(smem_u32(&sm.kv_free[j % kNK]));
        }
      } else {
        for (int j = 0; ok && j < n_tiles; ++j) {
          ok = wait_all(&sm.kv_ready[j % kNK], (j / kNK) & 1) &&
               (j < 2 || wait_all(&sm.p_free[T][j & 1], ((j >> 1) - 1) & 1));
          if (!ok) break;
          tc::fence_after_thread_sync();
          const uint64_t dk = dk0 + (uint64_t)((j % kNK) * (kKVTile >> 4));
          const uint32_t ts = tm + (uint32_t)(j & 1) * kTmemSP;
          if (tc::elect_one()) {
#pragma unroll
            for (int k = 0; k < 4; ++k) tc::mma_e4m3(ts, dq + 2 * k, dk + 2 * k, idS, k > 0);
            tc::commit(smem_u32(&sm.s_full[T][j & 1]));
            tc::commit(smem_u32(&sm.kv_free[j % kNK]));
          }
          __syncwarp();
        }
      }
      if (!ok) failed = true;
    }
  } else if (warp == 2) {
    // --------------------------------------------------- Q loader, P V issuer
    // One TMA box per M-tile: [32 queries][4 heads][128 d] = rows r = 4*query
    // + head, 128-byte swizzled by the tensor map.  Rows past total_q read as
    // zero; rows of the next sequence are computed but never stored.  (With
    // an invalid qo_indptr the box may start anywhere: loads out of range
    // read zeros, and the coordinate is kept where no int overflow occurs.)
    if (lane == 0 && n_tiles > 0) {
      const int64_t z0 = qo + q0;
      const int z = (z0 >= 0 && z0 < a.total_q) ? (int)z0 : (int)a.total_q;
      const uint32_t qb_ = smem_u32(&sm.q_ready);
      mbar_arrive_expect_tx(qb_, 2u * kQTile);
      tma_load_3d(smem_u32(sm.q[0]), &q_map, 0, g * kGroup, z, qb_);
      tma_load_3d(smem_u32(sm.q[1]), &q_map, 0, g * kGroup, z + kQT, qb_);
    }
    __syncwarp();
    // Then O_T += P_T(j) V_j for T = 0, 1 in tile order, once the softmax has
    // written P_T(j) (p_full).  P_T(j) is in buffer j & 1 of M-tile T; the
    // commit on p_free tells the S issuer when that buffer may take S_T(j+2)
    // (and the softmax when O_T holds every P V up to tile j).  The V tile
    // was published with K (kv_ready) before S_T(j); the wait below is
    // already satisfied.
    if (n_tiles > 0) {
      constexpr uint32_t idO = tc::idesc_f16_f32(128, 128, true);  // B = V tile (F16), MN-major
      const uint64_t dv0 = tc::sw128_desc_lbo(smem_u32(sm.v[0]), kVHalf);
      const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
      bool ok = true;
      const int n_mt = t1_live ? 2 : 1;  // M-tiles computed
      for (int j = 0; ok && j < n_tiles; ++j) {
        ok = wait_all(&sm.kv_ready[j % kNK], (j / kNK) & 1);
        const uint64_t dv = dv0 + (uint64_t)((j % kNK) * ((2 * kVHalf) >> 4));
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (t >= n_mt) break;
          ok = ok && wait_all(&sm.p_full[t][j & 1], (j >> 1) & 1);
          if (!ok) break;
          tc::fence_after_thread_sync();
          const uint32_t tt = tm + (uint32_t)t * kTmemPerTile;
          const uint32_t pa = tt + (uint32_t)(j & 1) * kTmemSP;
          if (tc::elect_one()) {
            // K = 16 keys per MMA: 8 TMEM columns of P, 16 rows (2048 B) of V
#pragma unroll
            for (int k = 0; k < kKT / 16; ++k)
              tc::mma_f16_tmem_a(tt + kTmemO, pa + 8 * k, dv + 128 * k, idO, (j > 0 || k > 0) ? 1u : 0u);
            tc::commit(smem_u32(&sm.p_free[t][j & 1]));
            if (t == n_mt - 1) tc::commit(smem_u32(&sm.kv_free[j % kNK]));
          }
          __syncwarp();
        }
      }
      if (ok && tc::elect_one()) {
        tc::commit(smem_u32(&sm.o_final[0]));
        tc::commit(smem_u32(&sm.o_final[1]));
      }
      __syncwarp();
      if (!ok) failed = true;
    }
  } else if (warp < 8 || (warp < 12 && t1_live)) {
    // -------------------------------------------------------------- softmax
    const int T = (warp - 4) >> 2;
    const int sub = warp & 3;
    const int r = 32 * sub + lane;  // TMEM lane = row of M-tile T
    const int qrow = q0 + T * kQT + (r >> 2);
    const int hh = r & 3;
    int lim_key = kv_len - q_len + qrow;  // last visible key (inclusive)
    if (lim_key > kv_len - 1) lim_key = kv_len - 1;
    const uint32_t lane_off = (uint32_t)(32 * sub) << 16;
    const uint32_t tT = tmem + lane_off + (uint32_t)T * kTmemPerTile;
    const uint32_t tO = tT + kTmemO;
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    const bool neg_scale = scale_log2 < 0.f;
    const int n_mine = (T == 1 && !t1_live) ? 0 : n_tiles;  // tiles this M-tile computes
    for (int j = 0; j < n_mine; ++j) {
      // warp-uniform outcome: the TMEM accesses below are warp-collective
      if (!wait_all(&sm.s_full[T][j & 1], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc::fence_after_thread_sync();
      // buffer j & 1: S of the tile, then P over its first 32 columns (the
      // P V that read the buffer's previous P completed before this S was
      // issued)
      const uint32_t tS = tT + (uint32_t)(j & 1) * kTmemSP;
      const uint32_t tP = tS;
      const int kbase = (t_begin + j) * kKT;
      const bool masked = kbase + kKT - 1 > lim_key;
      // the tile's 64 logits stay in registers while P is written in their place
      uint32_t v0[32], v1[32];
      tc::ld32(tS, v0);
      tc::ld32(tS + 32, v1);
      tc::ld_wait();
      const bool mask_warp = __any_sync(0xffffffffu, masked);
      // P = 2^(x - m_used) in f16 -- x = s * scale_log2 - m_used is formed in
      // f32 and rounded to f16, then one ex2 per key pair -- written to the
      // buffer as the A operand of the F16 P V product: keys 32c..32c+31 ->
      // columns 16c..16c+15, two keys per column.  Returns the row's sum of
      // those f16 weights (a pairwise tree of f16 additions per 32 keys, then
      // f32).  Masked keys (and every key of a row that has seen none) become
      // 2^-inf = 0.  Two copies of the loop, so that the common unmasked tile
      // carries no per-key mask test; the choice is made per warp (any lane
      // masked): the TMEM stores are warp-collective and must not diverge.
      auto pass_p = [&](auto masked_tile) {
        constexpr bool kMasked = decltype(masked_tile)::value;
        const float2 cc = make_float2(scale_log2, scale_log2);
        const float2 mm = make_float2(-m_used, -m_used);
        float lsum_c = 0.f;
#pragma unroll
        for (int c = 0; c < kKT / 32; ++c) {
          const uint32_t* v = c == 0 ? v0 : v1;
          uint32_t pp[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {  // keys 2q, 2q+1 of the chunk
            float2 x = __ffma2_rn(make_float2(u2f(v[2 * q]), u2f(v[2 * q + 1])), cc, mm);
            if (kMasked) {
              const int k0 = kbase + 32 * c + 2 * q;
              if (k0 > lim_key) x.x = -INFINITY;
              if (k0 + 1 > lim_key) x.y = -INFINITY;
            }
            pp[q] = ex2_h2(f2_to_h2(x.x, x.y));
          }
          tc::st16(tP + 16 * c, pp);
          uint32_t t8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) t8[i] = hadd2_u(pp[2 * i], pp[2 * i + 1]);
#pragma unroll
          for (int i = 0; i < 4; ++i) t8[i] = hadd2_u(t8[2 * i], t8[2 * i + 1]);
          t8[0] = hadd2_u(hadd2_u(t8[0], t8[1]), hadd2_u(t8[2], t8[3]));
          lsum_c += h2_sum_f32(t8[0]);
        }
        return lsum_c;
      };
      // Optimistic pass with the running maximum as it stands.  A row sum of
      // at most 2^15 bounds every P of the row by about 2^15 < 65504, so the
      // f16 values are finite and the tile is done (an overflowing weight or
      // partial sum is inf and fails the test).  Otherwise (a row's first
      // keys, where m_used is -inf, or a maximum that grew by more than ~9) the
      // warp finds the rows' maxima, raises m where it grew by more than
      // 2^kRescaleLog2 (rescaling O and l), and computes P again.
      float lsum = mask_warp ? pass_p(std::true_type{}) : pass_p(std::false_type{});
      if (__any_sync(0xffffffffu, !(lsum <= kMaxTileSum))) {
        // extreme raw logit of the row (max, or min for a negative scale),
        // then the scaled maximum in the exp2 domain
        float ext = neg_scale ? INFINITY : -INFINITY;
        if (!masked) {
          float e0 = ext, e1 = u2f(v0[0]), e2 = u2f(v1[0]), e3 = u2f(v1[1]);
          if (!neg_scale) {
#pragma unroll
            for (int i = 1; i < 31; i += 2) {
              e0 = max3(e0, u2f(v0[i]), u2f(v0[i + 1]));
              e1 = max3(e1, u2f(v1[i + 1]), u2f(v1[i + 2]));
            }
            ext = max3(max3(e0, e1, e2), e3, u2f(v0[31]));
          } else {
#pragma unroll
            for (int i = 1; i < 31; i += 2) {
              e0 = min3(e0, u2f(v0[i]), u2f(v0[i + 1]));
              e1 = min3(e1, u2f(v1[i + 1]), u2f(v1[i + 2]));
            }
            ext = min3(min3(e0, e1, e2), e3, u2f(v0[31]));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (kbase + i <= lim_key) ext = neg_scale ? fminf(ext, u2f(v0[i])) : fmaxf(ext, u2f(v0[i]));
            if (kbase + 32 + i <= lim_key) ext = neg_scale ? fminf(ext, u2f(v1[i])) : fmaxf(ext, u2f(v1[i]));
          }
        }
        const float mx = (ext == INFINITY || ext == -INFINITY) ? -INFINITY : ext * scale_log2;
        const float m_new = fmaxf(m_used, mx);
        const bool raise = m_new > m_used + kRescaleLog2;  // also true for the first finite maximum
        const float alpha = raise ? fast_exp2(m_used - m_new) : 1.f;  // 0 when m_used was -inf
        if (__any_sync(0xffffffffu, raise && j > 0)) {
          // O_T must hold P V of every tile < j before it is rescaled (the P V
          // of tile j - 1, the last one issued for this M-tile, has completed)
          if (!wait_all(&sm.p_free[T][(j - 1) & 1], ((j - 1) >> 1) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after_thread_sync();
          // (16 columns at a time: the tile's 64 logits are still live)
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t o[16];
            tc::ld16(tO + 16 * c, o);
            tc::ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(u2f(o[i]) * alpha);
            tc::st16(tO + 16 * c, o);
          }
          tc::st_wait();
        }
        if (raise) {
          l *= alpha;
          m_used = m_new;
        }
        tc::st_wait();  // the optimistic P stores complete before they are overwritten
        lsum = mask_warp ? pass_p(std::true_type{}) : pass_p(std::false_type{});
      }
      l += lsum;
      tc::st_wait();
      tc::fence_before_thread_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_full[T][j & 1]));
    }
    if (!ok) failed = true;
    // ------------------------------------------------------------ epilogue
    // output row qo + qrow; rows outside the sequence or outside [0, total_q) are computed, never stored
    const bool row_ok = qrow < q_len && qo + qrow >= 0 && qo + qrow < a.total_q;
    bool have_o = false;
    if (ok && n_mine > 0) {
      have_o = wait_all(&sm.o_final[T], 0);
      if (!have_o) failed = true;
      tc::fence_after_thread_sync();
    }
    if constexpr (kSplit) {
      // Split-KV: this range's unnormalised O and its (m, l), in the exp2
      // domain of the scaled logits: O = sum 2^(x - m) V, l = sum 2^(x - m).
      // A range in which the row sees no key leaves l = 0.
      const int64_t prow = ((int64_t)blockIdx.y * a.total_q + qo + qrow) * kHq + g * kGroup + hh;
      float4* po = reinterpret_cast<float4*>(part_o + prow * kD);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        if (have_o) {
          tc::ld32(tO + 32 * c, o);
          tc::ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            po[8 * c + i] = make_float4(u2f(o[4 * i]), u2f(o[4 * i + 1]), u2f(o[4 * i + 2]), u2f(o[4 * i + 3]));
        }
      }
      if (row_ok) part_ml[prow] = make_float2(have_o ? m_used : -INFINITY, have_o ? l : 0.f);
    } else {
      const float inv = (l > 0.f) ? inv_out_scale / l : 0.f;
      uint8_t* dst = a.out + ((qo + qrow) * kHq + g * kGroup + hh) * kD;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        if (have_o) {
          tc::ld32(tO + 32 * c, o);
          tc::ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t pk[8];
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 x = __fmul2_rn(make_float2(u2f(o[4 * i]), u2f(o[4 * i + 1])), inv2);
          const float2 y = __fmul2_rn(make_float2(u2f(o[4 * i + 2]), u2f(o[4 * i + 3])), inv2);
          pk[i] = f4_to_e4m3x4(x.x, x.y, y.x, y.y);
        }
        if (row_ok) {
          *reinterpret_cast<uint4*>(dst + 32 * c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(dst + 32 * c + 16) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
    }
  } else {
    // ---------------------------------------------------------- dequantisers
    // Tile j (64 keys): K then V, each 256 items of (key, pair of adjacent
    // 16-element blocks), 2 of each per thread: one 16-byte load of codes,
    // one 2-byte load of scales and two scale-table entries per 32 elements.
    // All of a tile's loads -- codes, scales and both scale tables -- are
    // issued before the wait for the K/V slot (they only need the packed
    // stage), so their latencies overlap one another and the wait; K and V
    // are then written and published together.  Keys past kv_len (only in a
    // sequence's last tile) read as zero.
    // Warps 12-15 dequantise every tile; when M-tile 1 is idle its softmax
    // warps 8-11 form a second group: group 0 takes the even tiles, group 1
    // the odd ones, so two tiles' chains (page wait, loads, table lookups,
    // conversion, slot wait, stores, publication) overlap -- a tile's chain,
    // not the dequantisers' issue rate, bounds the one-M-tile calls.  Each
    // tile is still written and published by one group of four warps.
    const int group = warp >= 12 ? 0 : 1;
    const int j_step = t1_live ? 1 : 2;
    const int dt = (threadIdx.x & 127);
    const int key0 = dt >> 2;  // items dt + 128 it: key = key0 + 32 it, block pair pb = dt & 3
    const int pb = dt & 3;
    // V: blocks 2 pb and 2 pb + 1 are d = 32 pb .. 32 pb + 31, i.e. half pb / 2,
    // 16-byte chunks 4 (pb % 2) .. 4 (pb % 2) + 3
    const int vc0 = 4 * (pb & 1);
    bool ok = true;
    for (int j = group; j < n_tiles; j += j_step) {
      const int st = j % kNP;
      const int slot = j % kNK;
      if (!mbar_wait(smem_u32(&sm.pk_full[st]), (j / kNP) & 1, &g_ctx_err)) {
        ok = false;
        break;
      }
      uint4 packed[2][2];
      uint2 ktab[2][2];
      uint2 vtab[2][2];
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int key = key0 + 32 * it;
        packed[0][it] = *reinterpret_cast<const uint4*>(&sm.pk[st][0][key * 64 + pb * 16]);
        packed[1][it] = *reinterpret_cast<const uint4*>(&sm.pk[st][1][key * 64 + pb * 16]);
        const uint32_t ks = *reinterpret_cast<const uint16_t*>(&sm.sf[st][0][key * 8 + pb * 2]);
        const uint32_t vs = *reinterpret_cast<const uint16_t*>(&sm.sf[st][1][key * 8 + pb * 2]);
        ktab[it][0] = sm.ktab[ks & 0xffu];
        ktab[it][1] = sm.ktab[ks >> 8];
        vtab[it][0] = sm.ktab[vs & 0xffu];
        vtab[it][1] = sm.ktab[vs >> 8];
      }
      if (j >= kNK && !mbar_wait(smem_u32(&sm.kv_free[slot]), ((j / kNK) - 1) & 1, &g_ctx_err)) {
        ok = false;
        break;
      }
      if ((t_begin + j + 1) * kKT > kv_len) {
        // last tile: zero the codes of keys past kv_len (code 0 dequantises to +0)
#pragma unroll
        for (int kv = 0; kv < 2; ++kv)
#pragma unroll
          for (int it = 0; it < 2; ++it)
            if ((t_begin + j) * kKT + key0 + 32 * it >= kv_len) packed[kv][it] = make_uint4(0u, 0u, 0u, 0u);
      }
      uint8_t* kt = sm.k[slot];
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int key = key0 + 32 * it;
        *reinterpret_cast<uint4*>(kt + swz(key, 2 * pb)) =
            dequant16_e4m3(make_uint2(packed[0][it].x, packed[0][it].y), ktab[it][0]);
        *reinterpret_cast<uint4*>(kt + swz(key, 2 * pb + 1)) =
            dequant16_e4m3(make_uint2(packed[0][it].z, packed[0][it].w), ktab[it][1]);
      }
      uint8_t* half = sm.v[slot] + (pb >> 1) * kVHalf;
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int key = key0 + 32 * it;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t w0 = h == 0 ? packed[1][it].x : packed[1][it].z;
          const uint32_t w1 = h == 0 ? packed[1][it].y : packed[1][it].w;
          *reinterpret_cast<uint4*>(half + swz(key, vc0 + 2 * h)) = nvfp4_to_f16_8(w0, vtab[it][h]);
          *reinterpret_cast<uint4*>(half + swz(key, vc0 + 2 * h + 1)) = nvfp4_to_f16_8(w1, vtab[it][h]);
        }
      }
      // one proxy fence and one publication per tile (K and V together: a
      // second fence per tile for an earlier K costs more than it gains)
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.kv_ready[slot]));
        mbar_arrive(smem_u32(&sm.pk_empty[st]));
      }
    }
    if (!ok) failed = true;
  }

  // ---------------------------------------------------------------- teardown
  tc::fence_before_thread_sync();
  if (__syncthreads_or(failed)) {
    // A wait expired somewhere in this CTA: before TMEM is freed and the CTA
    // exits, let every MMA its issuers started and every bulk copy its
    // producer started complete (bounded waits again), so that nothing lands
    // in TMEM or shared memory that a later CTA on this SM may own.
    if (warp >= 1 && warp <= 3) {
      if (tc::elect_one()) tc::commit(smem_u32(&sm.drain[warp - 1]));
      __syncwarp();
      mbar_wait(smem_u32(&sm.drain[warp - 1]), 0, &g_ctx_err);
    } else if (warp == 0) {
      for (int jj = max(0, issued - kNP); jj < issued; ++jj)
        mbar_wait(smem_u32(&sm.pk_full[jj % kNP]), (jj / kNP) & 1, &g_ctx_err);
    }
    tc::fence_before_thread_sync();
    __syncthreads();
  }
  // Split-KV: the partials are written; let the merge grid be launched (it
  // waits for this grid's completion before it reads them).
  if constexpr (kSplit) asm volatile("griddepcontrol.launch_dependents;");
  if (warp == 1) {
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Launch of one instance of the attention kernel; the dynamic-shared-memory
// opt-in is made once per device and instance (cached bitmask).  (Internal
// linkage: every translation unit that launches an instance owns it, and its
// error word.)
template <bool kSplit, int kNP, int kNK>
static cudaError_t launch_attention(const CtxArgs& a, const CUtensorMap& q_map, dim3 grid, float scale_log2,
                                    float inv_out_scale, int tiles_per_split, float* part_o, float2* part_ml,
                                    cudaStream_t stream) {
  static std::atomic<uint64_t> ready{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  constexpr size_t smem = smem_bytes<kNP, kNK>();
  static_assert(smem <= 232448, "shared memory of this ring depth exceeds the per-block maximum");
  if (!(ready.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(ctx_nvfp4_kernel<kSplit, kNP, kNK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    ready.fetch_or(bit, std::memory_order_acq_rel);
  }
  ctx_nvfp4_kernel<kSplit, kNP, kNK><<<grid, kThreads, smem, stream>>>(a, q_map, scale_log2, inv_out_scale,
                                                                       tiles_per_split, part_o, part_ml);
  return cudaGetLastError();
}

// Reads and clears this translation unit's error word (synchronises the device).
static cudaError_t read_ctx_error_word(uint32_t* word) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  uint32_t zero = 0;
  if ((e = cudaMemcpyFromSymbol(word, g_ctx_err, sizeof(uint32_t))) != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_ctx_err, &zero, sizeof(uint32_t));
}

}  // namespace ctx
}  // namespace gqa
