// ctx_persistent.cuh -- the persistent form of the NVFP4 paged context
// attention kernel (sm_103a) for calls whose work units are short.
//
// Operation, work unit, warp roles, TMEM layout, online softmax and
// arithmetic: those of ctx_nvfp4_kernel (ctx_kernel.cuh), bit for bit; only
// the grid differs.  There every CTA takes one unit (sequence, KV head, block
// of 64 queries) and leaves; a unit of n KV tiles costs about 0.75 n us plus a
// fixed ~4-7 us for the CTA's start (tables, barriers, TMEM, the first
// page and Q loads, pipeline fill) and end (pipeline drain, output).  On a
// workload of short units (q_len = kv_len = 2048: 16.5 tiles per unit on
// average) that fixed part is a third of the time.  Here one CTA per SM walks
// its units in turn:
//  * Unit order: a snake over the longest-first order (CTA c of G takes in
//    round k the unit k G + c, or k G + G - 1 - c in odd rounds), which evens
//    out the CTAs' loads as well as the hardware's dynamic assignment does.
//  * Warp 0 (producer) writes each unit's descriptor into a ring of 8 that
//    the other 15 warps read, then loads the unit's Q (two TMA boxes, into
//    one of two buffers, once the S products of the unit two back have read
//    it) and its pages.  Every ring and buffer counter runs on across units,
//    so the next unit's Q, pages, dequantised tiles and first S products are
//    made while the current unit's last tiles and output are finished.
//  * A unit's first P V overwrites O_T: the softmax warps read the previous
//    unit's O_T (their epilogue) before they write the P it waits for.
//  * The epilogue stages each softmax warp's 32 output rows in the finished
//    unit's Q buffer and stores them query by query (512 contiguous bytes per
//    instruction instead of 32 partial lines); the softmax warps, not the S
//    issuers, then release the buffer to the producer.
// The same loop structure run over one long unit computes a tile ~8 % slower
// than ctx_nvfp4_kernel (measured on GB300, outputs byte-identical), so the
// launch plan takes this kernel only for calls of short units (see plan_ctx).
#pragma once
#include "ctx_kernel.cuh"

namespace gqa {
namespace ctx {

constexpr size_t kMaxSmemPerBlock = 232448;

// Units a CTA's producer may describe ahead of the consumers.
constexpr int kUnitRing = 8;

// Arrive `count` times at once on an mbarrier.
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// A softmax warp's 32 output rows (8 queries x 4 heads, 128 bytes each),
// staged in the warp's quarter of the unit's Q buffer (of its M-tile).
constexpr int kOStage = 32 * kD;

// One work unit as the producer describes it to the other roles.
struct Unit {
  int64_t qo;          // first output row of the sequence
  int b;               // sequence, or -1: this CTA has no further unit
  int g;               // KV head
  int q0;              // first query of the block, within the sequence
  int q_len, kv_len;   // clamped lengths of the sequence
  int n_tiles;         // KV tiles of the unit
};

template <int kNP, int kNK, int kQBuf>
struct PSmem {
  uint8_t q[kQBuf][2][kQTile];      // [unit % kQBuf][M-tile] Q (128B-swizzled, K-major A operand)
  uint8_t k[kNK][kKVTile];          // E4M3 K tiles (128B-swizzled, K-major B operand of S = Q K^T)
  uint8_t v[kNK][2 * kVHalf];       // V tiles as F16 (128B-swizzled, MN-major B operand of O += P V)
  uint8_t pk[kNP][2][kPackedPage];  // [stage][K=0,V=1][slot*64 + byte]
  uint8_t sf[kNP][2][kScalePage];   // [stage][K,V][slot*8 + block]
  uint64_t pk_full[kNP], pk_empty[kNP];
  uint64_t kv_ready[kNK], kv_free[kNK];   // dequantised K and V of a slot written / slot consumed
  uint64_t s_full[2][2];                  // [M-tile][buffer]: S computed
  uint64_t p_full[2][2], p_free[2][2];    // [M-tile][buffer]: P written / the P V that read it completed
  uint64_t o_final[2];                    // [M-tile]: every MMA of the unit's M-tile complete
  uint64_t q_ready[kQBuf], q_free[kQBuf];  // Q of a buffer loaded / free (the unit's output, staged there, stored)
  uint64_t unit_full[kUnitRing], unit_empty[kUnitRing];  // descriptor written / read by all 15 consumer warps
  uint64_t drain[3];                // teardown after an expired wait: MMAs of issuer warps 1..3 complete
  Unit unit[kUnitRing];
  uint2 ktab[256];                  // E4M3 magnitudes of the 8 E2M1 codes for every scale byte (K and V)
  uint32_t tmem_base;
};

// Q buffers of an instance: two (the next unit's Q loads while the current
// unit runs) where they fit beside the rings, else one.
template <int kNP, int kNK>
constexpr int q_buffers() {
  return sizeof(PSmem<kNP, kNK, 2>) + 1024 <= kMaxSmemPerBlock ? 2 : 1;
}

template <int kNP, int kNK>
using PSmemOf = PSmem<kNP, kNK, q_buffers<kNP, kNK>()>;

template <int kNP, int kNK>
constexpr size_t psmem_bytes() {
  return sizeof(PSmemOf<kNP, kNK>) + 1024;  // + alignment slack
}

// The k-th unit of this CTA (warp-collective: every lane gets the same
// descriptor; b = -1 once there is none).  CTA c of G takes in round k the
// unit k G + c (k even) or k G + G - 1 - c (k odd): a snake over the
// longest-first order, which evens out the CTAs' loads.  Unit index i is
// (find_unit's entry i / 8, KV head i % 8).
static __device__ Unit unit_of(const CtxArgs& a, int k) {
  Unit w;
  w.qo = 0;
  w.b = -1;
  w.g = w.q0 = w.q_len = w.kv_len = w.n_tiles = 0;
  const int64_t G = gridDim.x, c = blockIdx.x;
  const int64_t idx = (int64_t)k * G + ((k & 1) ? G - 1 - c : c);
  if (idx > 0x7fffffffLL) return w;
  int b, qb;
  find_unit(a.qo_indptr, (int)a.batch, a.total_q, (int)(idx / kHkv), b, qb);
  if (b < 0) return w;
  w.b = b;
  w.g = (int)(idx % kHkv);
  w.qo = a.qo_indptr[b];
  w.q_len = q_len_of(a.qo_indptr, b, a.total_q);
  const int kv_cap = (int)(a.max_pages_per_seq * kPage);
  const int kv_len = a.kv_lens[b];
  w.kv_len = kv_len < 0 ? 0 : (kv_len > kv_cap ? kv_cap : kv_len);
  w.q0 = qb * kQB;
  const int q_last = min(w.q0 + kQB, w.q_len) - 1;
  const int n_keys = min(w.kv_len, w.kv_len - w.q_len + q_last + 1);
  w.n_tiles = n_keys > 0 ? (n_keys + kKT - 1) / kKT : 0;
  return w;
}

template <int kNP, int kNK>
__global__ void __launch_bounds__(kThreads, 1)
    ctx_nvfp4_persistent_kernel(const __grid_constant__ CtxArgs a, const __grid_constant__ CUtensorMap q_map,
                                const float scale_log2, const float inv_out_scale) {
  static_assert(kNK >= 2 && kNP >= 2, "rings need at least two slots");
  constexpr int kQBuf = q_buffers<kNP, kNK>();
  using SM = PSmemOf<kNP, kNK>;
  extern __shared__ uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = (int)a.batch;

  if (warp == 2) {
    // Metadata check: CTA x checks sequences 32 x + 32 G i + lane (G CTAs,
    // i = 0, 1, ...), CTA 0 also the ends.
    bool bad = false;
    for (int64_t bq = (int64_t)blockIdx.x * 32 + lane; bq < B; bq += (int64_t)gridDim.x * 32)
      bad |= a.qo_indptr[bq + 1] < a.qo_indptr[bq];
    if (blockIdx.x == 0 && lane == 0) bad |= a.qo_indptr[0] != 0 || (int64_t)a.qo_indptr[B] != a.total_q;
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&g_ctx_err, kErrBadIndptr);
  } else if (warp == 3 && blockIdx.x == 0) {
    // Rows past the last offset belong to no unit: they are written as zeros
    // (only when qo_indptr is invalid).
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
    for (int i = 0; i < kQBuf; ++i) {
      mbar_init(smem_u32(&sm.q_ready[i]), 1);
      mbar_init(smem_u32(&sm.q_free[i]), 8);  // the softmax warps of both M-tiles, after their epilogue
    }
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(smem_u32(&sm.unit_full[i]), 1);
      mbar_init(smem_u32(&sm.unit_empty[i]), 15);  // every warp but the producer
    }
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&sm.drain[i]), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
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
  // The k-th unit's descriptor, as the producer wrote it (warp-collective).
  auto next_unit = [&](int k, Unit& w) {
    const int us = k % kUnitRing;
    if (!wait_all(&sm.unit_full[us], (k / kUnitRing) & 1)) return false;
    w = sm.unit[us];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.unit_empty[us]));
    return true;
  };
  // Every role walks the same sequence of units and numbers the KV tiles of
  // the CTA continuously (gt): the packed-page and K/V rings, and the S/P
  // buffers of each M-tile (counted over the tiles that M-tile computes),
  // run on across unit boundaries, so the next unit's pages and S start while
  // the current unit's last tiles and its output are finished.
  int issued = 0;       // producer: pages whose copies were issued
  int q_issued = 0;     // producer: Q loads issued
  bool failed = false;  // a wait of this thread's role expired

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Per unit: its descriptor into the unit ring; then (if it has tiles) Q
    // into buffer u % kQBuf -- two TMA boxes, one per M-tile, [32 queries][4
    // heads][128 d] = rows r = 4*query + head, 128-byte swizzled by the
    // tensor map, once the S products of the unit kQBuf back have read that
    // buffer; then one page per KV tile: packed K and V codes (4 KB each) and
    // their scales (512 B each) through the block table.  Q rows past
    // total_q read as zero; rows of the next sequence are computed but never
    // stored.  (With an invalid qo_indptr the box may start anywhere: loads
    // out of range read zeros, and the coordinate is kept where no int
    // overflow occurs.)  The page numbers are read 32 at a time by the whole
    // warp, one chunk ahead of use; lane 0 issues the copies.  (a.starve: a
    // test of the bounded waits -- no copy is issued, so every consumer's
    // wait expires.)
    const uint64_t pol = policy_evict_last();  // pages are re-read by the other query blocks
    int gt = 0;
    for (int k = 0;; ++k) {
      const Unit w = unit_of(a, k);
      const int us = k % kUnitRing;
      if (k >= kUnitRing && !wait_all(&sm.unit_empty[us], ((k / kUnitRing) - 1) & 1)) {
        failed = true;
        break;
      }
      if (lane == 0) {
        sm.unit[us] = w;
        mbar_arrive(smem_u32(&sm.unit_full[us]));
      }
      __syncwarp();
      if (w.b < 0) break;
      if (w.n_tiles == 0 || a.starve) continue;
      const int qbuf = q_issued % kQBuf;
      if (q_issued >= kQBuf && !wait_all(&sm.q_free[qbuf], ((q_issued / kQBuf) - 1) & 1)) {
        failed = true;
        break;
      }
      if (lane == 0) {
        const int64_t z0 = w.qo + w.q0;
        const int z = (z0 >= 0 && z0 < a.total_q) ? (int)z0 : (int)a.total_q;
        const uint32_t qb_ = smem_u32(&sm.q_ready[qbuf]);
        mbar_arrive_expect_tx(qb_, 2u * kQTile);
        tma_load_3d(smem_u32(sm.q[qbuf][0]), &q_map, 0, w.g * kGroup, z, qb_);
        tma_load_3d(smem_u32(sm.q[qbuf][1]), &q_map, 0, w.g * kGroup, z + kQT, qb_);
      }
      q_issued++;
      __syncwarp();
      const int n = w.n_tiles;
      const int32_t* bt = a.block_table + (int64_t)w.b * a.max_pages_per_seq;
      int cur = lane < n ? bt[lane] : 0;
      int nxt = 32 + lane < n ? bt[32 + lane] : 0;
      for (int j = 0; j < n; ++j) {
        if (j > 0 && (j & 31) == 0) {
          cur = nxt;
          nxt = j + 32 + lane < n ? bt[j + 32 + lane] : 0;
        }
        int phys = __shfl_sync(0xffffffffu, cur, j & 31);
        const int st = gt % kNP;
        if (gt >= kNP && !wait_all(&sm.pk_empty[st], ((gt / kNP) - 1) & 1)) {
          failed = true;
          break;
        }
        if (lane == 0) {
          if (phys < 0 || phys >= a.num_pages) {
            atomicOr(&g_ctx_err, kErrBadIndex);
            phys = 0;
          }
          const int64_t row = ((int64_t)phys * kHkv + w.g) * kPage;
          const uint32_t fb = smem_u32(&sm.pk_full[st]);
          mbar_arrive_expect_tx(fb, 2u * (kPackedPage + kScalePage));
          bulk_g2s_hint(smem_u32(sm.pk[st][0]), a.k_fp4 + row * (kD / 2), kPackedPage, fb, pol);
          bulk_g2s_hint(smem_u32(sm.sf[st][0]), a.k_sf + row * (kD / 16), kScalePage, fb, pol);
          bulk_g2s_hint(smem_u32(sm.pk[st][1]), a.v_fp4 + row * (kD / 2), kPackedPage, fb, pol);
          bulk_g2s_hint(smem_u32(sm.sf[st][1]), a.v_sf + row * (kD / 16), kScalePage, fb, pol);
        }
        issued = ++gt;
        __syncwarp();
      }
      if (failed) break;
    }
  } else if (warp == 1 || warp == 3) {
    // -------------------------------------------------------- S issuers
    // Warp 1 issues S = Q K^T of M-tile 0, warp 3 that of M-tile 1: S_T(c)
    // (c = the M-tile's tile count) into buffer c & 1 once K/V of the tile
    // are dequantised and P V_T(c-2), which read P_T(c-2) from that buffer,
    // has completed (p_free), so S of the next tile -- of this unit or the
    // next -- is computed while the softmax works on this one.  Waiting for
    // that P V also orders this S after the softmax's reads of S_T(c-2) and
    // its writes of P_T(c-2).  tcgen05.mma issue blocks while the tensor pipe
    // is busy, so S and P V have separate issuing warps and an S is never
    // queued behind a P V the softmax is not waiting for.  The whole warp
    // runs this code (descriptor arithmetic stays warp-uniform, which keeps
    // it in the uniform datapath the MMA reads); one elected lane issues each
    // MMA and commit.  (The unit's Q buffer is released by the softmax warps,
    // which stage the unit's output there.)  M-tile 1 holds queries q0 + 32
    // .. q0 + 63; when none of them exists (a sequence's last block of at most
    // 32 queries) it is not computed: its issuer only releases the K/V slots.
    const int T = warp == 1 ? 0 : 1;
    constexpr uint32_t idS = tc::idesc_e4m3_f32(128, kKT, false);  // B = K tile, K-major
    const uint64_t dk0 = tc::sw128_desc(smem_u32(sm.k[0]));
    const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0) + (uint32_t)T * kTmemPerTile;
    int gt = 0, sc = 0, qk = 0;  // tiles of the CTA, S tiles of this M-tile, units with tiles
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit w;
      ok = next_unit(k, w);
      if (!ok || w.b < 0) break;
      if (w.n_tiles == 0) continue;
      const int qbuf = qk % kQBuf;
      ok = wait_all(&sm.q_ready[qbuf], (qk / kQBuf) & 1);
      ++qk;
      if (!ok) break;
      if (T == 1 && !(w.q0 + kQT < w.q_len)) {
        for (int j = 0; ok && j < w.n_tiles; ++j, ++gt) {
          ok = wait_all(&sm.kv_ready[gt % kNK], (gt / kNK) & 1);
          if (ok && lane == 0) mbar_arrive(smem_u32(&sm.kv_free[gt % kNK]));
        }
      } else {
        const uint64_t dq = tc::sw128_desc(smem_u32(sm.q[qbuf][T]));
        for (int j = 0; j < w.n_tiles; ++j, ++gt, ++sc) {
          ok = wait_all(&sm.kv_ready[gt % kNK], (gt / kNK) & 1) &&
               (sc < 2 || wait_all(&sm.p_free[T][sc & 1], ((sc >> 1) - 1) & 1));
          if (!ok) break;
          tc::fence_after_thread_sync();
          const uint64_t dk = dk0 + (uint64_t)((gt % kNK) * (kKVTile >> 4));
          const uint32_t ts = tm + (uint32_t)(sc & 1) * kTmemSP;
          if (tc::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) tc::mma_e4m3(ts, dq + 2 * kk, dk + 2 * kk, idS, kk > 0);
            tc::commit(smem_u32(&sm.s_full[T][sc & 1]));
            tc::commit(smem_u32(&sm.kv_free[gt % kNK]));
          }
          __syncwarp();
        }
      }
    }
    if (!ok) failed = true;
  } else if (warp == 2) {
    // ------------------------------------------------------- P V issuer
    // O_T += P_T(c) V for T = 0, 1 in tile order, once the softmax has
    // written P_T(c) (p_full).  P_T(c) is in buffer c & 1 of M-tile T; the
    // commit on p_free tells the S issuer when that buffer may take
    // S_T(c+2) (and the softmax when O_T holds every P V up to that tile).
    // A unit's first P V overwrites O_T: the softmax warps read the previous
    // unit's O_T before they write the P it waits for.  After the unit's
    // last P V, o_final[T] tells the softmax warps that O_T is complete.
    // The V tile was published with K (kv_ready) before S; the wait below is
    // already satisfied.
    constexpr uint32_t idO = tc::idesc_f16_f32(128, 128, true);  // B = V tile (F16), MN-major
    const uint64_t dv0 = tc::sw128_desc_lbo(smem_u32(sm.v[0]), kVHalf);
    const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
    int gt = 0, pc0 = 0, pc1 = 0;  // tiles of the CTA, P V products of M-tile 0 / 1
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit w;
      ok = next_unit(k, w);
      if (!ok || w.b < 0) break;
      if (w.n_tiles == 0) continue;
      const int n_mt = w.q0 + kQT < w.q_len ? 2 : 1;  // M-tiles computed
      for (int j = 0; ok && j < w.n_tiles; ++j, ++gt) {
        ok = wait_all(&sm.kv_ready[gt % kNK], (gt / kNK) & 1);
        const uint64_t dv = dv0 + (uint64_t)((gt % kNK) * ((2 * kVHalf) >> 4));
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (t >= n_mt) break;
          const int c = t == 0 ? pc0 : pc1;
          ok = ok && wait_all(&sm.p_full[t][c & 1], (c >> 1) & 1);
          if (!ok) break;
          tc::fence_after_thread_sync();
          const uint32_t tt = tm + (uint32_t)t * kTmemPerTile;
          const uint32_t pa = tt + (uint32_t)(c & 1) * kTmemSP;
          if (tc::elect_one()) {
            // K = 16 keys per MMA: 8 TMEM columns of P, 16 rows (2048 B) of V
#pragma unroll
            for (int kk = 0; kk < kKT / 16; ++kk)
              tc::mma_f16_tmem_a(tt + kTmemO, pa + 8 * kk, dv + 128 * kk, idO, (j > 0 || kk > 0) ? 1u : 0u);
            tc::commit(smem_u32(&sm.p_free[t][c & 1]));
            if (t == n_mt - 1) tc::commit(smem_u32(&sm.kv_free[gt % kNK]));
          }
          __syncwarp();
          if (t == 0) ++pc0; else ++pc1;
        }
      }
      if (ok && tc::elect_one()) {
        tc::commit(smem_u32(&sm.o_final[0]));
        if (n_mt == 2) tc::commit(smem_u32(&sm.o_final[1]));
      }
      __syncwarp();
    }
    if (!ok) failed = true;
  } else if (warp < 12) {
    // -------------------------------------------------------------- softmax
    const int T = (warp - 4) >> 2;
    const int sub = warp & 3;
    const int r = 32 * sub + lane;  // TMEM lane = row of M-tile T
    const int hh = r & 3;
    const uint32_t lane_off = (uint32_t)(32 * sub) << 16;
    const uint32_t tT = tmem + lane_off + (uint32_t)T * kTmemPerTile;
    const uint32_t tO = tT + kTmemO;
    const bool neg_scale = scale_log2 < 0.f;
    int sc = 0, oc = 0, qk = 0;  // S tiles of this M-tile, units whose O_T was completed, units with tiles
    bool ok = true;
    for (int k = 0; ok; ++k) {
      // Only what the tile loop needs is read here; the epilogue reads the
      // output coordinates from the descriptor again (the slot is released
      // after it), which keeps the loop's live registers to a minimum.
      const int us = k % kUnitRing;
      if (!wait_all(&sm.unit_full[us], (k / kUnitRing) & 1)) {
        ok = false;
        break;
      }
      const Unit& wd = sm.unit[us];
      if (wd.b < 0) break;
      const int q_len = wd.q_len, kv_len = wd.kv_len;
      const int qrow = wd.q0 + T * kQT + (r >> 2);
      int lim_key = kv_len - q_len + qrow;  // last visible key (inclusive)
      if (lim_key > kv_len - 1) lim_key = kv_len - 1;
      float m_used = -INFINITY;
      float l = 0.f;
      const int n_mine = (T == 1 && !(wd.q0 + kQT < q_len)) ? 0 : wd.n_tiles;  // tiles this M-tile computes
      for (int j = 0; j < n_mine; ++j, ++sc) {
        // warp-uniform outcome: the TMEM accesses below are warp-collective
        if (!wait_all(&sm.s_full[T][sc & 1], (sc >> 1) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_thread_sync();
        // buffer sc & 1: S of the tile, then P over its first 32 columns (the
        // P V that read the buffer's previous P completed before this S was
        // issued)
        const uint32_t tS = tT + (uint32_t)(sc & 1) * kTmemSP;
        const uint32_t tP = tS;
        const int kbase = j * kKT;
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
        // 2^kRescaleLog2 (rescaling O and l), and computes P again.  The
        // optimistic pass is skipped where it is bound to fail: a row whose
        // m_used is still -inf and which sees a key of this tile gets an
        // infinite weight (the same P results either way).
        float lsum = INFINITY;
        if (!__any_sync(0xffffffffu, m_used == -INFINITY && kbase <= lim_key))
          lsum = mask_warp ? pass_p(std::true_type{}) : pass_p(std::false_type{});
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
            if (!wait_all(&sm.p_free[T][(sc - 1) & 1], ((sc - 1) >> 1) & 1)) {
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
        if (lane == 0) mbar_arrive(smem_u32(&sm.p_full[T][sc & 1]));
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      // output row qo + qrow; rows outside the sequence or outside [0, total_q) are computed, never stored
      const int64_t qo = *reinterpret_cast<const volatile int64_t*>(&wd.qo);
      const int g = *reinterpret_cast<const volatile int*>(&wd.g);
      const bool row_ok = qrow < q_len && qo + qrow >= 0 && qo + qrow < a.total_q;
      bool have_o = false;
      if (n_mine > 0) {
        have_o = wait_all(&sm.o_final[T], oc & 1);
        ++oc;
        if (!have_o) {
          ok = false;
          break;
        }
        tc::fence_after_thread_sync();
      }
      const float inv = (l > 0.f) ? inv_out_scale / l : 0.f;
      uint8_t* dst = a.out + ((qo + qrow) * kHq + g * kGroup + hh) * kD;
      // The warp's rows are 8 consecutive queries x the group's 4 heads (lane
      // L: query L / 4, head L % 4), i.e. eight 512-byte spans of the output,
      // one per query.  When all 32 are rows of this sequence within
      // [0, total_q) and the unit had tiles, they are staged in the unit's Q
      // buffer -- every S product that read it has completed (o_final, or no
      // product of this M-tile) -- row L at 128 L, 16-byte chunk i at chunk
      // i ^ (L % 8) (no bank conflicts either way), then read back so that
      // each store instruction writes one query's 512 bytes; otherwise every
      // row that is stored at all is stored by its thread (32 partial lines
      // per instruction).  The Q buffer goes back to the producer (q_free)
      // after the read-back: eight arrivals, one per warp of each computed
      // M-tile -- M-tile 0's warps arrive twice when M-tile 1 was not
      // computed, since M-tile 1's warps then wait for nothing and could
      // otherwise arrive for a later unit's use of the buffer first.
      const bool q_held = *reinterpret_cast<const volatile int*>(&wd.n_tiles) > 0;
      const int qbuf = qk % kQBuf;
      const bool staged = __all_sync(0xffffffffu, row_ok) && q_held;
      uint8_t* stage = sm.q[qbuf][T] + kOStage * sub;
      const int z = (int)(qo + qrow) - (lane >> 2);  // first query of the warp's rows (valid when staged)
      // Four rounds of 32 columns; round c + 1's TMEM load is in flight while
      // round c is converted and staged.
      auto emit = [&](const uint32_t (&o)[32], int c) {
        uint32_t pk[8];
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 x = __fmul2_rn(make_float2(u2f(o[4 * i]), u2f(o[4 * i + 1])), inv2);
          const float2 y = __fmul2_rn(make_float2(u2f(o[4 * i + 2]), u2f(o[4 * i + 3])), inv2);
          pk[i] = f4_to_e4m3x4(x.x, x.y, y.x, y.y);
        }
        if (staged) {
#pragma unroll
          for (int i = 0; i < 2; ++i)
            *reinterpret_cast<uint4*>(stage + 128 * lane + 16 * ((2 * c + i) ^ (lane & 7))) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        } else if (row_ok) {
#pragma unroll
          for (int i = 0; i < 2; ++i)
            *reinterpret_cast<uint4*>(dst + 32 * c + 16 * i) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      };
      uint32_t oa[32], ob[32];
      if (have_o) {
        tc::ld32(tO, oa);
        tc::ld_wait();
        tc::ld32(tO + 32, ob);
        emit(oa, 0);
        tc::ld_wait();
        tc::ld32(tO + 64, oa);
        emit(ob, 1);
        tc::ld_wait();
        tc::ld32(tO + 96, ob);
        emit(oa, 2);
        tc::ld_wait();
        emit(ob, 3);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) oa[i] = 0u;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) emit(oa, c);
      }
      if (staged) {
        // read back query by query (lane L: head L / 8, 16-byte chunk L % 8)
        // and store each query's 512 contiguous bytes with one instruction
        __syncwarp();
        const int hr = lane >> 3, ch = lane & 7;
        uint8_t* gb = a.out + ((int64_t)z * kHq + g * kGroup + hr) * kD + 16 * ch;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = 4 * i + hr;
          const uint4 v = *reinterpret_cast<const uint4*>(stage + 128 * row + 16 * (ch ^ (row & 7)));
          *reinterpret_cast<uint4*>(gb + (int64_t)i * kHq * kD) = v;
        }
      }
      if (q_held) {
        __syncwarp();
        if (lane == 0 && (T == 0 || n_mine > 0))
          mbar_arrive_n(smem_u32(&sm.q_free[qbuf]), (T == 0 && !(wd.q0 + kQT < q_len)) ? 2u : 1u);
        ++qk;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.unit_empty[us]));
    }
    if (!ok) failed = true;
  } else {
    // ---------------------------------------------------------- dequantisers
    // Tile j (64 keys): K then V, each 256 items of (key, pair of adjacent
    // 16-element blocks), 2 of each per thread: one 16-byte load of codes,
    // one 2-byte load of scales and two scale-table entries per 32 elements.
    // All of a tile's loads -- codes, scales and both scale tables -- are
    // issued before the wait for the K/V slot (they only need the packed
    // stage), so their latencies overlap one another and the wait; K and V
    // are then written and published together.  Keys past kv_len (only in a
    // sequence's last tile) read as zero.  (Waits are warp-collective, so a
    // wait that expires ends the warp's loops together.)
    const int dt = threadIdx.x - 384;
    const int key0 = dt >> 2;  // items dt + 128 it: key = key0 + 32 it, block pair pb = dt & 3
    const int pb = dt & 3;
    // V: blocks 2 pb and 2 pb + 1 are d = 32 pb .. 32 pb + 31, i.e. half pb / 2,
    // 16-byte chunks 4 (pb % 2) .. 4 (pb % 2) + 3
    const int vc0 = 4 * (pb & 1);
    int gt = 0;  // tiles of the CTA
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit w;
      ok = next_unit(k, w);
      if (!ok || w.b < 0) break;
      for (int j = 0; j < w.n_tiles; ++j, ++gt) {
        const int st = gt % kNP;
        const int slot = gt % kNK;
        if (!wait_all(&sm.pk_full[st], (gt / kNP) & 1)) {
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
        if (gt >= kNK && !wait_all(&sm.kv_free[slot], ((gt / kNK) - 1) & 1)) {
          ok = false;
          break;
        }
        if ((j + 1) * kKT > w.kv_len) {
          // last tile: zero the codes of keys past kv_len (code 0 dequantises to +0)
#pragma unroll
          for (int kv = 0; kv < 2; ++kv)
#pragma unroll
            for (int it = 0; it < 2; ++it)
              if (j * kKT + key0 + 32 * it >= w.kv_len) packed[kv][it] = make_uint4(0u, 0u, 0u, 0u);
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
      for (int qq = max(0, q_issued - kQBuf); qq < q_issued; ++qq)
        mbar_wait(smem_u32(&sm.q_ready[qq % kQBuf]), (qq / kQBuf) & 1, &g_ctx_err);
    }
    tc::fence_before_thread_sync();
    __syncthreads();
  }
  if (warp == 1) {
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Launch of the persistent kernel: min(units, SMs) CTAs.  units = the
// launched-unit bound (8 KV heads x query blocks); the CTAs find the real
// units themselves.
template <int kNP, int kNK>
static cudaError_t launch_persistent(const CtxArgs& a, const CUtensorMap& q_map, int64_t units, float scale_log2,
                                     float inv_out_scale, cudaStream_t stream) {
  static std::atomic<uint64_t> ready{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  constexpr size_t smem = psmem_bytes<kNP, kNK>();
  static_assert(smem <= kMaxSmemPerBlock, "shared memory of this ring depth exceeds the per-block maximum");
  if (!(ready.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(ctx_nvfp4_persistent_kernel<kNP, kNK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    ready.fetch_or(bit, std::memory_order_acq_rel);
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (units < 1 || sms < 1) return cudaErrorInvalidConfiguration;
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  ctx_nvfp4_persistent_kernel<kNP, kNK><<<grid, kThreads, smem, stream>>>(a, q_map, scale_log2, inv_out_scale);
  return cudaGetLastError();
}

}  // namespace ctx
}  // namespace gqa
