// ctx_nvfp4.cu -- NVFP4 paged context (prefill) attention for sm_103a, and
// the test export of its dequantisation.
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
//    S buffers (64 fp32 columns each, tile j in buffer j & 1) and O (128
//    columns).  The softmax writes P of tile j (64 f16 weights per row = 32
//    columns) over the first half of the S buffer it read, and PV reads it
//    there as its TMEM A operand.  So S of tile j+1 is computed into the
//    other buffer while the softmax works on tile j; S of tile j+2 waits
//    only for the PV of tile j, the last reader of its buffer.
//  * Warp roles (16 warps): 0 = bulk-copy producer of packed NVFP4 pages +
//    scales through the block table into a 6-stage ring; 1 and 3 = issuers
//    of S = Q K^T for M-tile 0 and 1 (warp 1 also owns the TMEM allocation);
//    2 = Q loader (two TMA boxes through a 128-byte-swizzling tensor map),
//    then issuer of O += P V for both M-tiles; 4-7 and 8-11 = softmax of
//    M-tile 0 and 1 (one thread per TMEM lane = row); 12-15 = dequantisers
//    writing the K tile (E4M3) and the V tile (its E4M3 values widened to
//    F16) in the 128-byte swizzled layouts the MMA descriptors read (K as the
//    K-major B operand of S = Q K^T, V as the MN-major B operand of O = P V).
//  * Per M-tile T and KV tile j: S_T(j) is issued once K of tile j is
//    dequantised and PV_T(j-2) has completed; PV_T(j) once the softmax has
//    written P_T(j).  A softmax warp that raises its running maximum waits
//    for the PV of the previous tile before rescaling O in TMEM.
//  * Online softmax in the exp2 domain with a lazy running maximum m: m is
//    raised only when a row's maximum exceeds it by more than 2^8, so O is
//    rescaled rarely.
//  * S = Q K^T is an FP8 (E4M3 x E4M3) product.  P V is an F16 product: P is
//    rounded to f16 (11 significant bits) and V's dequantised E4M3 values
//    are widened to f16 exactly.  A one-term E4M3 P carries ~2 % relative
//    error per weight, which puts ~3 % of the outputs more than 2 E4M3 ulps
//    from the exact result; an f16 P costs no more tensor time than the
//    two E4M3 terms (hi + lo) it would take to match it, and one conversion
//    per two weights instead of a split.
//  * Split-KV (ctx_nvfp4_kernel<true>): when the units cannot fill the GPU
//    (short query lengths, few sequences), grid.y divides each unit's KV
//    tiles into contiguous ranges; each range writes its unnormalised O and
//    (m, l) in f32, and ctx_merge_kernel, launched as a programmatic
//    dependent grid, combines them by their maxima.  A unit whose queries
//    all lie in M-tile 0 leaves M-tile 1 idle in both instances.
#include <cuda.h>  // CUtensorMap and the cuTensorMapEncodeTiled prototype (resolved at run time)
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <type_traits>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "nvfp4.cuh"
#include "tcgen05.cuh"

namespace gqa {
namespace {

__device__ uint32_t g_ctx_err;

// ---------------------------------------------------------------------------
// Debug export: dense gather of dequantised tokens, one thread per (token,
// KV head, 16-element block), through the same dequant16 as the kernel.
// ---------------------------------------------------------------------------
__global__ void dequant_pages_kernel(const uint8_t* __restrict__ fp4, const uint8_t* __restrict__ sf,
                                     const int32_t* __restrict__ block_table, const int32_t* __restrict__ kv_lens,
                                     uint8_t* __restrict__ out, int64_t num_pages, int64_t max_pages_per_seq,
                                     int64_t max_kv) {
  const int b = blockIdx.y;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // over max_kv * 8 * 8
  if (idx >= max_kv * kHkv * 8) return;
  const int64_t t = idx / (kHkv * 8);
  const int g = (int)((idx / 8) % kHkv);
  const int blk = (int)(idx % 8);
  int64_t len = kv_lens[b];
  len = len < 0 ? 0 : (len > max_kv ? max_kv : len);
  uint4 r = make_uint4(0u, 0u, 0u, 0u);
  if (t < len) {
    const int64_t page = block_table[(int64_t)b * max_pages_per_seq + t / kPage];
    if (page >= 0 && page < num_pages) {
      const int64_t row = (page * kHkv + g) * kPage + (t % kPage);
      const uint2 packed = *reinterpret_cast<const uint2*>(fp4 + row * (kD / 2) + blk * 8);
      r = dequant16(packed, sf[row * (kD / 16) + blk]);
    } else {
      atomicOr(&g_ctx_err, kErrBadIndex);
    }
  }
  *reinterpret_cast<uint4*>(out + (((int64_t)b * max_kv + t) * kHkv + g) * kD + blk * 16) = r;
}

// ---------------------------------------------------------------------------
// Context attention kernel.
// ---------------------------------------------------------------------------
constexpr int kQB = 64;                    // queries per work unit
constexpr int kQT = 32;                    // queries per M=128 tile (x 4 heads)
constexpr int kKT = 64;                    // keys per KV tile (one page)
constexpr int kNK = 4;                     // E4M3 K/V tile slots
constexpr int kNP = 6;                     // packed-page ring stages
constexpr int kCtxThreads = 512;
constexpr int kQTile = 128 * 128;          // one M-tile of Q, E4M3: 16 KB
constexpr int kKVTile = kKT * 128;         // one K tile, E4M3: 8 KB
constexpr int kVHalf = kKT * 64 * 2;       // one V tile half (64 of the 128 d), F16: 8 KB
constexpr int kPackedPage = kPage * kD / 2;   // 4 KB of codes per (page, KV head)
constexpr int kScalePage = kPage * kD / 16;   // 512 B of scales per (page, KV head)
constexpr float kRescaleLog2 = 8.f;        // lazy-maximum threshold when a row's maximum is recomputed
constexpr float kMaxTileSum = 32768.f;     // a tile's row sum of P up to which no P can overflow f16
constexpr uint32_t kTmemCols = 512;
// TMEM columns of M-tile T, from T*256: two S/P buffers (64 f32 columns of S
// each, tile j in buffer j & 1; P of the tile, as f16 pairs, overwrites the
// buffer's first 32 columns), O (128 columns).
constexpr uint32_t kTmemPerTile = 256;
constexpr uint32_t kTmemSP = 64;  // columns per S/P buffer
constexpr uint32_t kTmemO = 128;

struct CtxSmem {
  uint8_t q[2][kQTile];        // M-tiles 0/1 of Q (128B-swizzled, K-major A operand)
  uint8_t k[kNK][kKVTile];     // E4M3 K tiles (128B-swizzled, K-major B operand of S = Q K^T)
  uint8_t v[kNK][2 * kVHalf];  // V tiles as F16 (128B-swizzled, MN-major B operand of O += P V; d 0-63, then 64-127)
  uint8_t pk[kNP][2][kPackedPage];  // [stage][K=0,V=1][slot*64 + byte]
  uint8_t sf[kNP][2][kScalePage];   // [stage][K,V][slot*8 + block]
  uint64_t pk_full[kNP], pk_empty[kNP];
  uint64_t kv_ready[kNK], kv_free[kNK];  // dequantised K and V tile of a slot written / slot consumed
  uint64_t s_full[2][2];                // [M-tile][buffer]: S computed
  uint64_t p_full[2][2], p_free[2][2];  // [M-tile][buffer]: P written / the PV that read it completed
  uint64_t o_final[2], q_ready;  // o_final: every MMA of an M-tile completed
  uint2 sftab[256];      // E4M3 magnitudes of the 8 E2M1 codes for every scale byte
  uint32_t tmem_base;
  int unit_b, unit_qb;
};
constexpr size_t kCtxSmemBytes = sizeof(CtxSmem) + 1024;  // + alignment slack

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a 128B-swizzled tile
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

// Work index t -> (b, query block), longest first: rounds r = 0, 1, ...; in
// round r every sequence with more than r query blocks contributes its block
// (n_blocks - 1 - r), in batch order.  All lanes of the calling warp get the
// same answer; b = -1 when t is past the last unit.
__device__ void find_unit(const int32_t* __restrict__ qo, int B, int t, int& out_b, int& out_qb) {
  const int lane = threadIdx.x & 31;
  out_b = -1;
  out_qb = -1;
  int nqb0 = 0;  // blocks of sequence lane, read once (the rounds below reuse it)
  if (lane < B) {
    const int ql = qo[lane + 1] - qo[lane];
    nqb0 = ql > 0 ? (ql + kQB - 1) / kQB : 0;
  }
  for (int r = 0;; ++r) {
    int cnt = 0;
    bool any = false;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int nqb = nqb0;
      if (b0 > 0) {
        nqb = 0;
        if (b < B) {
          const int ql = qo[b + 1] - qo[b];
          nqb = ql > 0 ? (ql + kQB - 1) / kQB : 0;
        }
      }
      const unsigned bal = __ballot_sync(0xffffffffu, nqb > r);
      const int c = __popc(bal);
      if (t >= cnt && t < cnt + c) {
        unsigned m = bal;
        for (int i = 0; i < t - cnt; ++i) m &= m - 1;  // drop the lower set bits
        const int bb = b0 + __ffs(m) - 1;
        const int ql = qo[bb + 1] - qo[bb];
        out_b = bb;
        out_qb = (ql + kQB - 1) / kQB - 1 - r;
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
// Two E4M3 bytes (low 16 bits, first element low) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)v));
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

// 3-D tiled TMA load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
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

template <bool kSplit>
__global__ void __launch_bounds__(kCtxThreads, 1)
    ctx_nvfp4_kernel(const CtxArgs a, const __grid_constant__ CUtensorMap q_map, const float scale_log2,
                     const float inv_out_scale, const int tiles_per_split, float* __restrict__ part_o,
                     float2* __restrict__ part_ml) {
  extern __shared__ uint8_t smem_raw[];
  CtxSmem& sm = *reinterpret_cast<CtxSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.x % kHkv;

  if (warp == 0) {
    int ub, uqb;
    find_unit(a.qo_indptr, (int)a.batch, (int)(blockIdx.x / kHkv), ub, uqb);
    if (lane == 0) {
      sm.unit_b = ub;
      sm.unit_qb = uqb;
    }
  }
  for (int i = threadIdx.x; i < 256; i += kCtxThreads) sm.sftab[i] = nvfp4_scale_table((uint32_t)i);
  if (threadIdx.x == 32) {
    for (int i = 0; i < kNP; ++i) {
      mbar_init(smem_u32(&sm.pk_full[i]), 1);
      mbar_init(smem_u32(&sm.pk_empty[i]), 4);
    }
    for (int i = 0; i < kNK; ++i) {
      mbar_init(smem_u32(&sm.kv_ready[i]), 4);
      mbar_init(smem_u32(&sm.kv_free[i]), 3);  // S of both M-tiles, PV of both
    }
    for (int t = 0; t < 2; ++t) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(smem_u32(&sm.s_full[t][i]), 1);
        mbar_init(smem_u32(&sm.p_full[t][i]), 4);
        mbar_init(smem_u32(&sm.p_free[t][i]), 1);
      }
    }
    mbar_init(smem_u32(&sm.o_final[0]), 1);
    mbar_init(smem_u32(&sm.o_final[1]), 1);
    mbar_init(smem_u32(&sm.q_ready), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int b = sm.unit_b;
  if (b < 0) return;  // past the last unit: the whole CTA leaves
  const int qb = sm.unit_qb;
  const int qo = a.qo_indptr[b];
  const int q_len = a.qo_indptr[b + 1] - qo;
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // One page per KV tile: packed K and V codes (4 KB each) and their scales
    // (512 B each) through the block table.  The page numbers are read 32 at
    // a time by the whole warp, one chunk ahead of use, so no copy waits for
    // a block-table read; lane 0 issues the copies.
    if (n_tiles > 0) {
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
        if (j >= kNP &&
            !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.pk_empty[st]), ((j / kNP) - 1) & 1, &g_ctx_err)))
          break;
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
        __syncwarp();
      }
    }
  } else if (warp == 1 || warp == 3) {
    // -------------------------------------------------------- S issuers
    // Warp 1 issues S = Q K^T of M-tile 0, warp 3 that of M-tile 1: S_T(j)
    // into buffer j & 1 once K of tile j is dequantised and PV_T(j-2), which
    // read P_T(j-2) from that buffer, has completed (p_free), so S of the
    // next tile is computed while the softmax works on this one.  Waiting
    // for that PV also orders this S after the softmax's reads of S_T(j-2)
    // and its writes of P_T(j-2).  tcgen05.mma issue blocks while the tensor
    // pipe is busy, so S and PV have separate issuing warps and an S is
    // never queued behind a PV the softmax is not waiting for.  The whole
    // warp runs this code (descriptor arithmetic stays warp-uniform, which
    // keeps it in the uniform datapath the MMA reads); one elected lane
    // issues each MMA and commit.
    const int T = warp == 1 ? 0 : 1;
    if (n_tiles > 0) {
      constexpr uint32_t idS = tc::idesc_e4m3_f32(128, kKT, false);  // B = K tile, K-major
      const uint64_t dq = tc::sw128_desc(smem_u32(sm.q[T]));
      const uint64_t dk0 = tc::sw128_desc(smem_u32(sm.k[0]));
      const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0) + (uint32_t)T * kTmemPerTile;
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, &g_ctx_err));
      };
      bool ok = wait_all(&sm.q_ready, 0);
      if (T == 1 && !t1_live) {
        for (int j = 0; ok && j < n_tiles; ++j) {
          ok = wait_all(&sm.kv_ready[j % kNK], (j / kNK) & 1);
          if (ok && lane == 0) mbar_arrive(smem_u32(&sm.kv_free[j % kNK]));
        }
        ok = false;  // nothing to issue
      }
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
  } else if (warp == 2) {
    // --------------------------------------------------- Q loader, PV issuer
    // One TMA box per M-tile: [32 queries][4 heads][128 d] = rows r = 4*query
    // + head, 128-byte swizzled by the tensor map.  Rows past total_q read as
    // zero; rows of the next sequence are computed but never stored.
    if (lane == 0 && n_tiles > 0) {
      const uint32_t qb_ = smem_u32(&sm.q_ready);
      mbar_arrive_expect_tx(qb_, 2u * kQTile);
      tma_load_3d(smem_u32(sm.q[0]), &q_map, 0, g * kGroup, qo + q0, qb_);
      tma_load_3d(smem_u32(sm.q[1]), &q_map, 0, g * kGroup, qo + q0 + kQT, qb_);
    }
    __syncwarp();
    // Then O_T += P_T(j) V_j for T = 0, 1 in tile order, once the softmax has
    // written P_T(j) (p_full).  P_T(j) is in buffer j & 1 of M-tile T; the
    // commit on p_free tells the S issuer when that buffer may take S_T(j+2)
    // (and the softmax when O_T holds every PV up to tile j).  The V tile was published
    // with K (kv_ready) before S_T(j); the wait below is already satisfied.
    if (n_tiles > 0) {
      constexpr uint32_t idO = tc::idesc_f16_f32(128, 128, true);  // B = V tile (F16), MN-major
      const uint64_t dv0 = tc::sw128_desc_lbo(smem_u32(sm.v[0]), kVHalf);
      const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, &g_ctx_err));
      };
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
      if (tc::elect_one()) {
        tc::commit(smem_u32(&sm.o_final[0]));
        tc::commit(smem_u32(&sm.o_final[1]));
      }
      __syncwarp();
    }
  } else if (warp < 12) {
    // -------------------------------------------------------------- softmax
    const int T = (warp - 4) >> 2;
    const int sub = warp & 3;
    const int r = 32 * sub + lane;  // TMEM lane = row of M-tile T
    const int qrow = q0 + T * kQT + (r >> 2);
    const int hh = r & 3;
    int lim = kv_len - q_len + qrow;  // last visible key (inclusive)
    if (lim > kv_len - 1) lim = kv_len - 1;
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
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full[T][j & 1]), (j >> 1) & 1, &g_ctx_err))) {
        ok = false;
        break;
      }
      tc::fence_after_thread_sync();
      // buffer j & 1: S of the tile, then P over its first 32 columns (the
      // PV that read the buffer's previous P completed before this S was
      // issued)
      const uint32_t tS = tT + (uint32_t)(j & 1) * kTmemSP;
      const uint32_t tP = tS;
      const int kbase = (t_begin + j) * kKT;
      const bool masked = kbase + kKT - 1 > lim;
      // the tile's 64 logits stay in registers while P is written in their place
      uint32_t v0[32], v1[32];
      tc::ld32(tS, v0);
      tc::ld32(tS + 32, v1);
      tc::ld_wait();
      const bool mask_warp = __any_sync(0xffffffffu, masked);
      // P = 2^(x - m_used) in f16 -- x = s * scale_log2 - m_used is formed in
      // f32 and rounded to f16, then one ex2 per key pair -- written to
      // buffer j & 1 as the A operand of the F16 PV product: keys
      // 32c..32c+31 -> columns 16c..16c+15, two keys per column.  Returns the
      // row's sum of those f16 weights (a pairwise tree of f16 additions per
      // 32 keys, then f32).  Masked keys (and every key of a row that has
      // seen none) become 2^-inf = 0.  Two copies of the loop, so that the
      // common unmasked tile carries no per-key mask test; the choice is made
      // per warp (any lane masked): the TMEM stores are warp-collective and
      // must not diverge.
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
              if (k0 > lim) x.x = -INFINITY;
              if (k0 + 1 > lim) x.y = -INFINITY;
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
            if (kbase + i <= lim) ext = neg_scale ? fminf(ext, u2f(v0[i])) : fmaxf(ext, u2f(v0[i]));
            if (kbase + 32 + i <= lim) ext = neg_scale ? fminf(ext, u2f(v1[i])) : fmaxf(ext, u2f(v1[i]));
          }
        }
        const float mx = (ext == INFINITY || ext == -INFINITY) ? -INFINITY : ext * scale_log2;
        const float m_new = fmaxf(m_used, mx);
        const bool raise = m_new > m_used + kRescaleLog2;  // also true for the first finite maximum
        const float alpha = raise ? fast_exp2(m_used - m_new) : 1.f;  // 0 when m_used was -inf
        if (__any_sync(0xffffffffu, raise && j > 0)) {
          // O_T must hold PV of every tile < j before it is rescaled (the PV
          // of tile j - 1, the last one issued, has completed)
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.p_free[T][(j - 1) & 1]), ((j - 1) >> 1) & 1,
                                                &g_ctx_err))) {
            ok = false;
            break;
          }
          tc::fence_after_thread_sync();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tc::ld32(tO + 32 * c, o);
            tc::ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(u2f(o[i]) * alpha);
            tc::st32(tO + 32 * c, o);
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
    // ------------------------------------------------------------ epilogue
    bool have_o = false;
    if (ok && n_mine > 0) {
      have_o = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.o_final[T]), 0, &g_ctx_err));
      tc::fence_after_thread_sync();
    }
    const bool store = qrow < q_len;
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
        if (store) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            po[8 * c + i] = make_float4(u2f(o[4 * i]), u2f(o[4 * i + 1]), u2f(o[4 * i + 2]), u2f(o[4 * i + 3]));
        }
      }
      if (store) part_ml[prow] = make_float2(have_o ? m_used : -INFINITY, have_o ? l : 0.f);
    }
    const float inv = (l > 0.f) ? inv_out_scale / l : 0.f;
    uint8_t* dst = a.out + ((int64_t)(qo + qrow) * kHq + g * kGroup + hh) * kD;
#pragma unroll 1
    for (int c = 0; !kSplit && c < 4; ++c) {
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
        const float2 a = __fmul2_rn(make_float2(u2f(o[4 * i]), u2f(o[4 * i + 1])), inv2);
        const float2 b = __fmul2_rn(make_float2(u2f(o[4 * i + 2]), u2f(o[4 * i + 3])), inv2);
        pk[i] = f4_to_e4m3x4(a.x, a.y, b.x, b.y);
      }
      if (store) {
        *reinterpret_cast<uint4*>(dst + 32 * c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(dst + 32 * c + 16) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
  } else {
    // ---------------------------------------------------------- dequantisers
    // Tile j (64 keys): K then V, each 256 items of (key, pair of adjacent
    // 16-element blocks), 2 of each per thread: one 16-byte load of codes,
    // one 2-byte load of scales and two scale-table entries per 32 elements.
    // All of a tile's loads are issued before the wait for the K/V slot
    // (they only need the packed stage), so their latencies overlap one
    // another and the wait; K and V are then written and published together.
    // Keys past kv_len (only in a sequence's last tile) read as zero.
    const int dt = threadIdx.x - 384;
    const int key0 = dt >> 2;  // items dt + 128 it: key = key0 + 32 it, block pair pb = dt & 3
    const int pb = dt & 3;
    // V: blocks 2 pb and 2 pb + 1 are d = 32 pb .. 32 pb + 31, i.e. half pb / 2,
    // 16-byte chunks 4 (pb % 2) .. 4 (pb % 2) + 3
    const int vc0 = 4 * (pb & 1);
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % kNP;
      const int slot = j % kNK;
      if (!mbar_wait(smem_u32(&sm.pk_full[st]), (j / kNP) & 1, &g_ctx_err)) break;
      uint4 packed[2][2];
      uint2 tab[2][2][2];
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
#pragma unroll
        for (int it = 0; it < 2; ++it) {
          const int key = key0 + 32 * it;
          packed[kv][it] = *reinterpret_cast<const uint4*>(&sm.pk[st][kv][key * 64 + pb * 16]);
          const uint32_t sf2 = *reinterpret_cast<const uint16_t*>(&sm.sf[st][kv][key * 8 + pb * 2]);
          tab[kv][it][0] = sm.sftab[sf2 & 0xffu];
          tab[kv][it][1] = sm.sftab[sf2 >> 8];
        }
      }
      if (j >= kNK && !mbar_wait(smem_u32(&sm.kv_free[slot]), ((j / kNK) - 1) & 1, &g_ctx_err)) break;
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
        const uint4 lo = dequant16_table(make_uint2(packed[0][it].x, packed[0][it].y), tab[0][it][0]);
        const uint4 hi = dequant16_table(make_uint2(packed[0][it].z, packed[0][it].w), tab[0][it][1]);
        *reinterpret_cast<uint4*>(kt + swz(key, 2 * pb)) = lo;
        *reinterpret_cast<uint4*>(kt + swz(key, 2 * pb + 1)) = hi;
      }
      uint8_t* half = sm.v[slot] + (pb >> 1) * kVHalf;
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int key = key0 + 32 * it;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 e = dequant16_table(h == 0 ? make_uint2(packed[1][it].x, packed[1][it].y)
                                                 : make_uint2(packed[1][it].z, packed[1][it].w),
                                          tab[1][it][h]);
          *reinterpret_cast<uint4*>(half + swz(key, vc0 + 2 * h)) =
              make_uint4(e4m3x2_to_f16x2(e.x), e4m3x2_to_f16x2(e.x >> 16), e4m3x2_to_f16x2(e.y),
                         e4m3x2_to_f16x2(e.y >> 16));
          *reinterpret_cast<uint4*>(half + swz(key, vc0 + 2 * h + 1)) =
              make_uint4(e4m3x2_to_f16x2(e.z), e4m3x2_to_f16x2(e.z >> 16), e4m3x2_to_f16x2(e.w),
                         e4m3x2_to_f16x2(e.w >> 16));
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.kv_ready[slot]));
        mbar_arrive(smem_u32(&sm.pk_empty[st]));
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc::fence_before_thread_sync();
  __syncthreads();
  // Split-KV: the partials are written; let the merge grid be launched (it
  // waits for this grid's completion before it reads them).
  if constexpr (kSplit) asm volatile("griddepcontrol.launch_dependents;");
  if (warp == 1) {
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Split-KV merge: one warp per (query row, head), lane l holding head-dim
// elements 4l .. 4l+3.  With M the largest m of the ranges that saw a key,
//   out = E4M3( sum_s 2^(m_s - M) O_s / (sum_s 2^(m_s - M) l_s) / out_scale ),
// and zeros when no range saw one (the same result as one unsplit pass, up
// to f32 rounding order).
// ---------------------------------------------------------------------------
constexpr int kMergeWarps = 8;
constexpr int kCtxSplitTargetCtas = 152;  // one wave: one CTA per SM
constexpr int kMinTilesPerSplit = 8;      // a split amortises the CTA's start-up over >= 512 keys

__global__ void __launch_bounds__(32 * kMergeWarps)
    ctx_merge_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml, uint8_t* __restrict__ out,
                     int64_t rows, int n_splits, float inv_out_scale) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);  // token * 32 + head
  // Launched as a programmatic dependent of the attention kernel: wait until
  // that grid has completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (row >= rows) return;
  // lane s holds range s's (m, l) (at most 32 ranges: the plan makes <= 19)
  float m_s = -INFINITY, l_s = 0.f;
  if (lane < n_splits) {
    const float2 ml = part_ml[(int64_t)lane * rows + row];
    if (ml.y > 0.f) {
      m_s = ml.x;
      l_s = ml.y;
    }
  }
  float mx = m_s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float w = l_s > 0.f ? fast_exp2(m_s - mx) : 0.f;  // mx is finite when some range saw a key
  float den = w * l_s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  // every range wrote its row (zeros where it saw no key), so the loads need no guard
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = 0; s < n_splits; ++s) {
    const float ws = __shfl_sync(0xffffffffu, w, s);
    const float4 o = reinterpret_cast<const float4*>(part_o + ((int64_t)s * rows + row) * kD)[lane];
    acc.x = fmaf(ws, o.x, acc.x);
    acc.y = fmaf(ws, o.y, acc.y);
    acc.z = fmaf(ws, o.z, acc.z);
    acc.w = fmaf(ws, o.w, acc.w);
  }
  const float inv = den > 0.f ? inv_out_scale / den : 0.f;
  reinterpret_cast<uint32_t*>(out + row * kD)[lane] = f4_to_e4m3x4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

std::atomic<uint64_t> g_ctx_smem_ready{0};

cudaError_t ensure_ctx_smem(int dev) {
  const uint64_t bit = 1ull << (dev & 63);
  if (g_ctx_smem_ready.load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaError_t e =
      cudaFuncSetAttribute(ctx_nvfp4_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCtxSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(ctx_nvfp4_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCtxSmemBytes);
  if (e != cudaSuccess) return e;
  g_ctx_smem_ready.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_dequant_pages(const uint8_t* fp4, const uint8_t* sf, const int32_t* block_table,
                                 const int32_t* kv_lens, uint8_t* out, int64_t batch, int64_t num_pages,
                                 int64_t max_pages_per_seq, int64_t max_kv, cudaStream_t stream) {
  const int64_t n = max_kv * kHkv * 8;
  dim3 grid((unsigned)((n + 255) / 256), (unsigned)batch);
  dequant_pages_kernel<<<grid, 256, 0, stream>>>(fp4, sf, block_table, kv_lens, out, num_pages, max_pages_per_seq,
                                                  max_kv);
  return cudaGetLastError();
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

// Tensor map over q [total_q][32 heads][128 d] (E4M3 bytes): boxes of
// [32 tokens][4 heads][128 d], 128-byte swizzle, zero fill out of range.
cudaError_t make_q_map(const uint8_t* q, int64_t total_q, CUtensorMap* map) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (!g_encode) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kHq, (cuuint64_t)total_q};
  const cuuint64_t strides[2] = {(cuuint64_t)kD, (cuuint64_t)kHq * kD};
  const cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)kGroup, (cuuint32_t)kQT};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(q), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

// Upper bound on the number of (sequence, 64-query block) units without
// reading qo_indptr on the host: sum_b ceil(q_b / 64) = sum_b floor((q_b + 63)
// / 64) <= floor((total_q + 63 batch) / 64).
static int64_t max_query_blocks(int64_t batch, int64_t total_q) {
  return (total_q + (int64_t)(kQB - 1) * batch) / kQB;
}

CtxPlan plan_ctx(int64_t batch, int64_t total_q, int64_t max_pages_per_seq) {
  CtxPlan p{0, 1};
  if (batch < 1 || total_q < 1 || max_pages_per_seq < 1) return p;
  // Launched units (an upper bound on the real ones, as the grid below).
  const int64_t units = max_query_blocks(batch, total_q) * kHkv;
  int64_t splits = kCtxSplitTargetCtas / units;
  const int64_t by_len = max_pages_per_seq / kMinTilesPerSplit;
  if (by_len < splits) splits = by_len;
  if (splits < 2) return p;
  const int64_t tps = (max_pages_per_seq + splits - 1) / splits;
  p.tiles_per_split = (int)tps;
  p.n_splits = (int)((max_pages_per_seq + tps - 1) / tps);
  return p;
}

size_t ctx_workspace_bytes(int64_t total_q, const CtxPlan& plan) {
  if (plan.n_splits <= 1) return 0;
  return (size_t)plan.n_splits * (size_t)total_q * kHq * (kD * sizeof(float) + sizeof(float2));
}

cudaError_t launch_ctx(const CtxArgs& a, const CtxPlan& plan, void* workspace, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = ensure_ctx_smem(dev)) != cudaSuccess) return e;
  alignas(64) CUtensorMap q_map;
  if ((e = make_q_map(a.q, a.total_q, &q_map)) != cudaSuccess) return e;
  const int64_t grid = max_query_blocks(a.batch, a.total_q) * kHkv;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const float scale_log2 = a.q_scale / sqrtf((float)kD) * 1.4426950408889634f;
  const float inv_out_scale = 1.f / a.out_scale;
  const bool split = plan.n_splits > 1;
  if (!split) {
    ctx_nvfp4_kernel<false><<<dim3((unsigned)grid, 1), kCtxThreads, kCtxSmemBytes, stream>>>(
        a, q_map, scale_log2, inv_out_scale, 0, nullptr, nullptr);
    return cudaGetLastError();
  }
  // the merge holds one range per lane
  if (!workspace || plan.tiles_per_split < 1 || plan.n_splits > 32) return cudaErrorInvalidValue;
  const int64_t rows = a.total_q * kHq;
  float* part_o = static_cast<float*>(workspace);
  float2* part_ml = reinterpret_cast<float2*>(part_o + (size_t)plan.n_splits * rows * kD);
  ctx_nvfp4_kernel<true><<<dim3((unsigned)grid, (unsigned)plan.n_splits), kCtxThreads, kCtxSmemBytes, stream>>>(
      a, q_map, scale_log2, inv_out_scale, plan.tiles_per_split, part_o, part_ml);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t mblocks = (rows + kMergeWarps - 1) / kMergeWarps;
  if (mblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // programmatic dependent launch: the merge's launch overlaps the attention
  // kernel's tail (the merge waits for it with griddepcontrol.wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)mblocks);
  cfg.blockDim = dim3(32 * kMergeWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ctx_merge_kernel, (const float*)part_o, (const float2*)part_ml, a.out, rows,
                            plan.n_splits, inv_out_scale);
}

cudaError_t ctx_read_errors(uint32_t* word) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  uint32_t zero = 0;
  if ((e = cudaMemcpyFromSymbol(word, g_ctx_err, sizeof(uint32_t))) != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_ctx_err, &zero, sizeof(uint32_t));
}

}  // namespace gqa
