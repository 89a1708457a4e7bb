// ctx_decode.cuh -- the decode-shaped form of the NVFP4 paged context
// attention (sm_103a): for calls whose sequences bring only a few new
// queries each (q_len of 1 to a few), as in decoding against an NVFP4 KV
// cache.
//
// Operation: that of ctx_nvfp4_kernel (ctx_kernel.cuh; "GB300 NVFP4 Context
// Attention: scale slot 조기 반납과 8단 packed K/V ring", introduction):
// E4M3 Q, NVFP4 K/V pages dequantised to E4M3, bottom-right causal,
// O = softmax(q K^T * q_scale / sqrt(128)) V.  Results are written as
// split-KV partials (unnormalised O and (m, l) in the exp2 domain) that
// ctx_merge_kernel combines and writes as E4M3(O / out_scale).
//
// Why a second shape: the prefill kernel stacks 32 queries x 4 heads into
// the MMA's M dimension.  A unit of one query uses 4 of those 128 rows, yet
// its softmax warps work on all 128 rows of every tile.  Here the product is
// computed transposed:
//   S^T = K Q^T   M = 128 keys (two pages), N = kN query rows (4 heads x
//                 kN/4 queries), K = 128 head dims: kind::f8f6f4, A = the
//                 K tile (K-major), B = the unit's Q rows (K-major)
//   O^T += V^T P^T M = 128 head dims, N = kN rows, K = 16 keys per MMA:
//                 kind::f16, A = the V tile as F16 (MN-major: the same layout
//                 the prefill kernel uses as its B operand), B = P^T in
//                 shared memory (K-major, keys along K)
// so one softmax thread holds one key's kN logits, and the softmax costs
// kN values per key instead of 128.
//
// Measured against ctx_nvfp4_kernel on 64 sequences x 1 query x 8192 keys:
// 1.06x (outputs within the same parity bar).  K and V tiles recycle through
// separate rings: a K slot is free once S^T has read it, a V slot once O^T
// has (three shared K/V slots: 1.05x; two: 0.80x).  Timing probes (invalid
// output): the page copies alone take 0.63 of the kernel's time (4 page
// stages, ~37 KB in flight per SM), the work on the pages alone 0.88; a third
// dequantiser group, a deeper page ring or one O^T product per tile gain
// little or nothing.
//
// Work unit: (sequence b, chunk of kN/4 queries, KV head g, KV range);
// grid.x = 8 KV heads x a bound on the (sequence, chunk) pairs from
// host-known sizes (CTAs past the last unit leave at once), grid.y = KV
// ranges of tiles_per_range 128-key tiles.
// Warp roles (16 warps): 0 producer of packed pages (one page per stage, 4 stages),
// 1 issuer of S^T, 2 issuer of O^T, 3 Q loader, 4-7 softmax (TMEM lane =
// key of the tile) and epilogue (TMEM lane = head dim), 8-11 and 12-15
// dequantisers of a tile's first and second page.
// TMEM: two S^T buffers (kN columns each), then O^T (kN columns).  Shared
// memory: 3 K slots (16 KB), 4 V slots (32 KB), 4 page stages (9 KB).
// Every wait is bounded (2 s); the teardown drains as in ctx_nvfp4_kernel.
#pragma once
#include "ctx_kernel.cuh"

namespace gqa {
namespace ctx {

constexpr int kDecKT = 128;                  // keys per tile: two pages
constexpr int kDecKTile = kDecKT * kD;       // E4M3 K tile: 16 KB
constexpr int kDecVHalf = kDecKT * 64 * 2;   // one 64-dim half of the F16 V tile: 16 KB
constexpr int kDecNP = 4;                    // packed-page stages (pages)
constexpr int kDecNKk = 3;                   // dequantised K tile slots (16 KB each): free once S^T completes
constexpr int kDecNKv = 4;                   // dequantised V tile slots (32 KB each): free once O^T completes

template <int kN>
struct DecSmem {
  uint8_t k[kDecNKk][kDecKTile];            // K tiles: 128 keys x 128 B, 128B-swizzled (K-major A of S^T)
  uint8_t v[kDecNKv][2 * kDecVHalf];        // V tiles: [half][128 keys][128 B] F16, 128B-swizzled (MN-major A of O^T)
  uint8_t pk[kDecNP][2][kPackedPage];       // [stage][K=0,V=1][slot*64 + byte]
  uint8_t sf[kDecNP][2][kScalePage];        // [stage][K,V][slot*8 + block]
  uint8_t q[kN * 128];                      // Q rows r = 4*query + head, 128B-swizzled (K-major B of S^T)
  uint8_t p[2][2][kN * 128];                // P^T [buffer][keys 0-63 | 64-127][row][128 B] F16, 128B-swizzled
  uint64_t pk_full[kDecNP], pk_empty[kDecNP];
  uint64_t kv_ready[kDecNKv], k_free[kDecNKk], v_free[kDecNKv];  // tile j: K slot j % 3, V slot j % 4
  uint64_t s_full[2], s_free[2], p_full[2], p_free[2];
  uint64_t q_ready, o_final, drain[2];
  uint2 ktab[256];
  float red[4][kN];                         // per-warp row maxima / row sums of the softmax warps
  float mrow[kN];                           // the rows' final maxima (epilogue)
  float alpha[kN];                          // the rows' rescaling factors of a tile's slow path
  uint32_t tmem_base;
  int unit_b, unit_c;
};

template <int kN>
constexpr size_t dec_smem_bytes() {
  return sizeof(DecSmem<kN>) + 1024;
}

// Chunk t of the calls' (sequence, query chunk) pairs in sequence order
// (warp-collective; every lane gets the same answer): b = -1 past the last.
// A sequence of q_len queries has ceil(q_len / chunk) chunks.
__device__ __forceinline__ void find_chunk(const int32_t* __restrict__ qo, int B, int64_t total_q, int chunk,
                                           int t, int& out_b, int& out_c) {
  const int lane = threadIdx.x & 31;
  out_b = -1;
  out_c = -1;
  int base = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    const int n = b < B ? (q_len_of(qo, b, total_q) + chunk - 1) / chunk : 0;
    int incl = n;  // inclusive prefix sum over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (t < base + total) {
      const unsigned hit = __ballot_sync(0xffffffffu, t < base + incl);
      const int src = __ffs(hit) - 1;
      const int before = __shfl_sync(0xffffffffu, incl - n, src);
      out_b = b0 + src;
      out_c = t - base - before;
      return;
    }
    base += total;
  }
}

// Order-preserving map of a float to a signed int (max of the ints = max of the floats).
__device__ __forceinline__ int f2ord(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7fffffff);
}
__device__ __forceinline__ float ord2f(int i) { return __int_as_float(i >= 0 ? i : (i ^ 0x7fffffff)); }

__device__ __forceinline__ int warp_max_i32(int v) {
  int r;
  asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// OR of a predicate over the 128 threads of named barrier 1 (the softmax warps).
__device__ __forceinline__ bool softmax_bar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void softmax_bar() { asm volatile("barrier.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ uint16_t f2h_bits(float x) {
  const __half h = __float2half_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}
__device__ __forceinline__ float h_bits2f(uint16_t b) { return __half2float(*reinterpret_cast<const __half*>(&b)); }

// tcgen05.ld of kN columns (16 or 32) of this warp's 32 lanes.
template <int kN>
__device__ __forceinline__ void ld_cols(uint32_t taddr, uint32_t (&r)[kN]) {
  if constexpr (kN == 32) {
    tc::ld32(taddr, r);
  } else {
    tc::ld16(taddr, r);
  }
}
template <int kN>
__device__ __forceinline__ void st_cols(uint32_t taddr, const uint32_t (&r)[kN]) {
  if constexpr (kN == 32) {
    uint32_t a[16], b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      a[i] = r[i];
      b[i] = r[16 + i];
    }
    tc::st16(taddr, a);
    tc::st16(taddr + 16, b);
  } else {
    tc::st16(taddr, r);
  }
}

template <int kN>
__global__ void __launch_bounds__(kThreads, 1)
    ctx_nvfp4_decode_kernel(const __grid_constant__ CtxArgs a, const float scale_log2, const int tiles_per_range,
                            float* __restrict__ part_o, float2* __restrict__ part_ml) {
  static_assert(kN == 16, "16 query rows per unit (4 queries x 4 heads)");
  constexpr int kChunk = kN / 4;  // queries per unit
  using SM = DecSmem<kN>;
  extern __shared__ uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.x % kHkv;
  const int B = (int)a.batch;

  if (warp == 0) {
    int ub, uc;
    find_chunk(a.qo_indptr, B, a.total_q, kChunk, (int)(blockIdx.x / kHkv), ub, uc);
    if (lane == 0) {
      sm.unit_b = ub;
      sm.unit_c = uc;
    }
  } else if (warp == 2 && blockIdx.y == 0) {
    // metadata check: sequences 32 x + 32 G i + lane, CTA 0 also the ends
    bool bad = false;
    for (int64_t bq = (int64_t)blockIdx.x * 32 + lane; bq < B; bq += (int64_t)gridDim.x * 32)
      bad |= a.qo_indptr[bq + 1] < a.qo_indptr[bq];
    if (blockIdx.x == 0 && lane == 0) bad |= a.qo_indptr[0] != 0 || (int64_t)a.qo_indptr[B] != a.total_q;
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&g_ctx_err, kErrBadIndptr);
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) sm.ktab[i] = nvfp4_scale_table((uint32_t)i);
  if (threadIdx.x == 32) {
    for (int i = 0; i < kDecNP; ++i) {
      mbar_init(smem_u32(&sm.pk_full[i]), 1);
      mbar_init(smem_u32(&sm.pk_empty[i]), 4);
    }
    for (int i = 0; i < kDecNKv; ++i) {
      mbar_init(smem_u32(&sm.kv_ready[i]), 8);  // both dequantiser groups
      mbar_init(smem_u32(&sm.v_free[i]), 1);    // the O^T product
    }
    for (int i = 0; i < kDecNKk; ++i) mbar_init(smem_u32(&sm.k_free[i]), 1);  // the S^T product
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.s_full[i]), 1);
      mbar_init(smem_u32(&sm.s_free[i]), 4);
      mbar_init(smem_u32(&sm.p_full[i]), 4);
      mbar_init(smem_u32(&sm.p_free[i]), 1);
      mbar_init(smem_u32(&sm.drain[i]), 1);
    }
    mbar_init(smem_u32(&sm.q_ready), 1);
    mbar_init(smem_u32(&sm.o_final), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int b = sm.unit_b;
  if (b < 0) return;  // past the last unit
  const int q0 = sm.unit_c * kChunk;
  const int64_t qo = a.qo_indptr[b];
  const int q_len = q_len_of(a.qo_indptr, b, a.total_q);
  int kv_len = a.kv_lens[b];
  const int kv_cap = (int)(a.max_pages_per_seq * kPage);
  kv_len = kv_len < 0 ? 0 : (kv_len > kv_cap ? kv_cap : kv_len);
  const int q_last = min(q0 + kChunk, q_len) - 1;
  const int n_keys = min(kv_len, kv_len - q_len + q_last + 1);  // keys any row of the chunk sees
  const int unit_tiles = n_keys > 0 ? (n_keys + kDecKT - 1) / kDecKT : 0;
  const int t_begin = (int)blockIdx.y * tiles_per_range;
  const int n_tiles = max(0, min(unit_tiles - t_begin, tiles_per_range));
  const int key_begin = t_begin * kDecKT;
  // pages of this range that hold keys below n_keys
  const int n_pages = n_tiles > 0 ? min(2 * n_tiles, (n_keys - key_begin + kPage - 1) / kPage) : 0;

  if (warp == 1) {
    __syncwarp();
    tc::tmem_alloc(smem_u32(&sm.tmem_base), 128);
    tc::tmem_relinquish();
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const uint32_t tmem = sm.tmem_base;
  auto wait_all = [](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, &g_ctx_err));
  };
  int issued = 0;
  bool failed = false;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (n_pages > 0 && !a.starve) {
      const uint64_t pol = policy_evict_first();  // every page is read once
      const int32_t* bt = a.block_table + (int64_t)b * a.max_pages_per_seq + (int64_t)t_begin * 2;
      int cur = lane < n_pages ? bt[lane] : 0;
      int nxt = 32 + lane < n_pages ? bt[32 + lane] : 0;
      for (int pg = 0; pg < n_pages; ++pg) {
        if (pg > 0 && (pg & 31) == 0) {
          cur = nxt;
          nxt = pg + 32 + lane < n_pages ? bt[pg + 32 + lane] : 0;
        }
        int phys = __shfl_sync(0xffffffffu, cur, pg & 31);
        const int st = pg % kDecNP;
        if (pg >= kDecNP && !wait_all(&sm.pk_empty[st], ((pg / kDecNP) - 1) & 1)) {
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
        issued = pg + 1;
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- S^T = K Q^T issuer
    if (n_tiles > 0) {
      constexpr uint32_t idS = tc::idesc_e4m3_f32(128, kN, false);
      const uint64_t dq = tc::sw128_desc(smem_u32(sm.q));
      const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
      bool ok = wait_all(&sm.q_ready, 0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int ks = j % kDecNKk;
        ok = wait_all(&sm.kv_ready[j % kDecNKv], (j / kDecNKv) & 1) &&
             (j < 2 || wait_all(&sm.s_free[j & 1], ((j >> 1) - 1) & 1));
        if (!ok) break;
        tc::fence_after_thread_sync();
        const uint64_t dk = tc::sw128_desc(smem_u32(sm.k[ks]));
        if (tc::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) tc::mma_e4m3(tm + (uint32_t)(j & 1) * kN, dk + 2 * kk, dq + 2 * kk, idS, kk > 0);
          tc::commit(smem_u32(&sm.s_full[j & 1]));
          tc::commit(smem_u32(&sm.k_free[ks]));
        }
        __syncwarp();
      }
      if (!ok) failed = true;
    }
  } else if (warp == 2) {
    // -------------------------------------------------- O^T += V^T P^T issuer
    if (n_tiles > 0) {
      constexpr uint32_t idO = tc::idesc_f16_f32_ab(128, kN, true, false);  // A = V tile MN-major, B = P^T K-major
      const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0) + 2 * kN;
      bool ok = true;
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int vs = j % kDecNKv;
        ok = wait_all(&sm.kv_ready[vs], (j / kDecNKv) & 1) && wait_all(&sm.p_full[j & 1], (j >> 1) & 1);
        if (!ok) break;
        tc::fence_after_thread_sync();
        const uint64_t dv = tc::sw128_desc_lbo(smem_u32(sm.v[vs]), kDecVHalf);
        const uint64_t dp = tc::sw128_desc(smem_u32(sm.p[j & 1][0]));
        if (tc::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kDecKT / 16; ++kk) {
            // 16 keys: 16 rows (2 KB) of each V half; 32 B of each P^T row, the
            // second 64 keys in the next block of kN rows
            const uint64_t a_d = dv + (uint64_t)(kk * (2048 >> 4));
            const uint64_t b_d = dp + (uint64_t)((kk >> 2) * ((kN * 128) >> 4) + (kk & 3) * 2);
            tc::mma_f16(tm, a_d, b_d, idO, (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc::commit(smem_u32(&sm.p_free[j & 1]));
          tc::commit(smem_u32(&sm.v_free[vs]));
        }
        __syncwarp();
      }
      if (ok && tc::elect_one()) tc::commit(smem_u32(&sm.o_final));
      __syncwarp();
      if (!ok) failed = true;
    }
  } else if (warp == 3) {
    // --------------------------------------------------------- Q loader
    // row r = 4 * query + head of the chunk; rows of queries outside the
    // sequence or past total_q are zero
    if (lane < kN) {
      const int qi = lane >> 2, h = lane & 3;
      const int64_t tok = qo + q0 + qi;
      const bool valid = q0 + qi < q_len && tok >= 0 && tok < a.total_q;
      const uint4* src = reinterpret_cast<const uint4*>(a.q + (tok * kHq + g * kGroup + h) * kD);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sm.q + swz(lane, c)) = v;
      }
    }
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.q_ready));
  } else if (warp < 8) {
    // ----------------------------------------------------- softmax, epilogue
    const int k = 32 * (warp - 4) + lane;  // key of the tile (S^T lane) / head dim (O^T lane)
    const uint32_t lane_off = (uint32_t)(32 * (warp - 4)) << 16;
    float m[kN], l[kN];
#pragma unroll
    for (int r = 0; r < kN; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
    }
    // query qi of the chunk sees key j iff j < kv_len and j - lim0 <= qi
    const int lim0 = kv_len - q_len + q0;
    // The four softmax warps meet at named barriers (barrier 1) in every
    // tile, so none of them may leave the loop early: after an expired wait a
    // warp records it, skips its later waits and arrivals and keeps running
    // the (harmless) rest of each iteration, and every wait is bounded, so the
    // others finish too.
    bool ok = true;
    // P^T of key k: byte offset in a [kN rows][128 B] block
    const int kb = k >> 6, kc = (k & 63) >> 3, kw = (k & 7) * 2;
    for (int j = 0; j < n_tiles; ++j) {
      if (ok) ok = wait_all(&sm.s_full[j & 1], (j >> 1) & 1);
      tc::fence_after_thread_sync();
      uint32_t sv[kN];
      ld_cols<kN>(tmem + lane_off + (uint32_t)(j & 1) * kN, sv);
      tc::ld_wait();
      tc::fence_before_thread_sync();
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(smem_u32(&sm.s_free[j & 1]));
      const int key = key_begin + j * kDecKT + k;
      const int dk = key < kv_len ? key - lim0 : 0x7fffffff;
      float* x = reinterpret_cast<float*>(sv);  // the logits, in place
      bool over = false;
#pragma unroll
      for (int r = 0; r < kN; ++r) {
        x[r] = dk <= (r >> 2) ? __uint_as_float(sv[r]) * scale_log2 : -INFINITY;
        over |= x[r] - m[r] > 15.f;  // (false for a masked key: NaN or -inf)
      }
      bool rescale = false;
      if (softmax_bar_or(over)) {
        // some weight could exceed 2^15 with the maxima as they stand: take
        // the tile's row maxima and raise m where they grew by more than 2^8
        // (also for the first finite maximum), scaling l and, below, O^T by
        // alpha = 2^(m_old - m_new), as the prefill kernel does; every thread
        // computes the same values
#pragma unroll
        for (int r = 0; r < kN; ++r) {
          const int mx = warp_max_i32(f2ord(x[r]));
          if (lane == 0) sm.red[warp - 4][r] = ord2f(mx);
        }
        softmax_bar();
        bool any_raise = false;
#pragma unroll
        for (int r = 0; r < kN; ++r) {
          const float tmx = fmaxf(fmaxf(sm.red[0][r], sm.red[1][r]), fmaxf(sm.red[2][r], sm.red[3][r]));
          float al = 1.f;
          if (tmx > m[r] + 8.f) {
            al = fast_exp2(m[r] - tmx);  // 0 when m was -inf
            l[r] *= al;
            m[r] = tmx;
            any_raise = true;
          }
          if (warp == 4 && lane == 0) sm.alpha[r] = al;
        }
        rescale = any_raise && j > 0;
        if (rescale) softmax_bar();  // sm.alpha visible to the four warps
      }
      // P^T buffer j & 1 was last read by the O^T product of tile j - 2
      if (ok && j >= 2) ok = wait_all(&sm.p_free[j & 1], ((j >> 1) - 1) & 1);
      uint8_t* pb = sm.p[j & 1][kb];
#pragma unroll
      for (int r = 0; r < kN; ++r) {
        const float pv = x[r] == -INFINITY || m[r] == -INFINITY ? 0.f : fast_exp2(x[r] - m[r]);
        const uint16_t h = f2h_bits(pv);
        l[r] += h_bits2f(h);
        *reinterpret_cast<uint16_t*>(pb + (r >> 3) * 1024 + (r & 7) * 128 + ((kc ^ (r & 7)) << 4) + kw) = h;
      }
      if (rescale) {
        // O^T must hold the products of every earlier tile before it is
        // rescaled (this tile's product waits for the P published below)
        if (ok) ok = wait_all(&sm.p_free[(j - 1) & 1], ((j - 1) >> 1) & 1);
        tc::fence_after_thread_sync();
        uint32_t o[kN];
        ld_cols<kN>(tmem + lane_off + 2 * kN, o);
        tc::ld_wait();
#pragma unroll
        for (int r = 0; r < kN; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * sm.alpha[r]);
        st_cols<kN>(tmem + lane_off + 2 * kN, o);
        tc::st_wait();
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_thread_sync();
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(smem_u32(&sm.p_full[j & 1]));
    }
    if (!ok) failed = true;
    // -------------------------------------------------------------- epilogue
    // row sums over the 128 key threads, then this range's partial rows
    bool have_o = false;
    if (ok && n_tiles > 0) {
      have_o = wait_all(&sm.o_final, 0);
      if (!have_o) failed = true;
    }
    tc::fence_after_thread_sync();
    // (every thread holds the same maxima; one warp parks them in shared memory)
    if (warp == 4 && lane == 0) {
#pragma unroll
      for (int r = 0; r < kN; ++r) sm.mrow[r] = m[r];
    }
    softmax_bar();  // every warp has read the last tile's maxima from red
#pragma unroll
    for (int r = 0; r < kN; ++r) {
      float sum = l[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) sm.red[warp - 4][r] = sum;
    }
    softmax_bar();
    uint32_t ov[kN];
    if (have_o) {
      ld_cols<kN>(tmem + lane_off + 2 * kN, ov);
      tc::ld_wait();
    } else {
#pragma unroll
      for (int r = 0; r < kN; ++r) ov[r] = 0u;
    }
    // row r = 4 qi + h of the chunk -> partial row (range, token qo + q0 + qi, head 4 g + h)
    const int64_t prow0 = ((int64_t)blockIdx.y * a.total_q + qo + q0) * kHq + g * kGroup;
    float* po = part_o + prow0 * kD + k;
    const int64_t tok0 = qo + q0;
#pragma unroll
    for (int r = 0; r < kN; ++r) {
      const int qi = r >> 2, h = r & 3;
      if (q0 + qi < q_len && tok0 + qi >= 0 && tok0 + qi < a.total_q) {
        po[(qi * kHq + h) * kD] = have_o ? __uint_as_float(ov[r]) : 0.f;
        if (k == 0) {
          const float lt = sm.red[0][r] + sm.red[1][r] + sm.red[2][r] + sm.red[3][r];
          part_ml[prow0 + qi * kHq + h] = make_float2(have_o && lt > 0.f ? sm.mrow[r] : -INFINITY, have_o ? lt : 0.f);
        }
      }
    }
  } else {
    // ---------------------------------------------------------- dequantisers
    // Group 0 (warps 8-11) writes keys 0-63 of each tile from its first page,
    // group 1 (warps 12-15) keys 64-127 from its second; a page past the
    // range's keys is written as zeros without a copy.  Per thread two keys
    // x one pair of 16-element blocks of K and V, as in the prefill kernel.
    const int grp = warp >= 12 ? 1 : 0;
    const int dt = threadIdx.x & 127;
    const int key0 = dt >> 2;
    const int pb = dt & 3;
    const int vc0 = 4 * (pb & 1);
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int pg = 2 * j + grp;  // page of the range
      const bool have = pg < n_pages;
      const int st = pg % kDecNP;
      const int ks = j % kDecNKk, vs = j % kDecNKv;
      uint4 packed[2][2];
      uint2 ktab[2][2], vtab[2][2];
      if (have) {
        if (!wait_all(&sm.pk_full[st], (pg / kDecNP) & 1)) {
          ok = false;
          break;
        }
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
      } else {
#pragma unroll
        for (int it = 0; it < 2; ++it) {
          packed[0][it] = packed[1][it] = make_uint4(0u, 0u, 0u, 0u);
          ktab[it][0] = ktab[it][1] = vtab[it][0] = vtab[it][1] = sm.ktab[0];
        }
      }
      if ((j >= kDecNKk && !wait_all(&sm.k_free[ks], ((j / kDecNKk) - 1) & 1)) ||
          (j >= kDecNKv && !wait_all(&sm.v_free[vs], ((j / kDecNKv) - 1) & 1))) {
        ok = false;
        break;
      }
      // keys past the sequence's visible range read as zero (code 0 -> +0)
#pragma unroll
      for (int kv = 0; kv < 2; ++kv)
#pragma unroll
        for (int it = 0; it < 2; ++it)
          if (key_begin + j * kDecKT + 64 * grp + key0 + 32 * it >= kv_len) packed[kv][it] = make_uint4(0u, 0u, 0u, 0u);
      uint8_t* kt = sm.k[ks];
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int row = 64 * grp + key0 + 32 * it;
        *reinterpret_cast<uint4*>(kt + swz(row, 2 * pb)) =
            dequant16_e4m3(make_uint2(packed[0][it].x, packed[0][it].y), ktab[it][0]);
        *reinterpret_cast<uint4*>(kt + swz(row, 2 * pb + 1)) =
            dequant16_e4m3(make_uint2(packed[0][it].z, packed[0][it].w), ktab[it][1]);
      }
      uint8_t* half = sm.v[vs] + (pb >> 1) * kDecVHalf;
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int row = 64 * grp + key0 + 32 * it;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t w0 = hh == 0 ? packed[1][it].x : packed[1][it].z;
          const uint32_t w1 = hh == 0 ? packed[1][it].y : packed[1][it].w;
          *reinterpret_cast<uint4*>(half + swz(row, vc0 + 2 * hh)) = nvfp4_to_f16_8(w0, vtab[it][hh]);
          *reinterpret_cast<uint4*>(half + swz(row, vc0 + 2 * hh + 1)) = nvfp4_to_f16_8(w1, vtab[it][hh]);
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.kv_ready[vs]));
        if (have) mbar_arrive(smem_u32(&sm.pk_empty[st]));
      }
    }
    if (!ok) failed = true;
  }

  // ---------------------------------------------------------------- teardown
  tc::fence_before_thread_sync();
  if (__syncthreads_or(failed)) {
    if (warp == 1 || warp == 2) {
      if (tc::elect_one()) tc::commit(smem_u32(&sm.drain[warp - 1]));
      __syncwarp();
      mbar_wait(smem_u32(&sm.drain[warp - 1]), 0, &g_ctx_err);
    } else if (warp == 0) {
      for (int jj = max(0, issued - kDecNP); jj < issued; ++jj)
        mbar_wait(smem_u32(&sm.pk_full[jj % kDecNP]), (jj / kDecNP) & 1, &g_ctx_err);
    }
    tc::fence_before_thread_sync();
    __syncthreads();
  }
  asm volatile("griddepcontrol.launch_dependents;");
  if (warp == 1) {
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, 128);
  }
}

template <int kN>
static cudaError_t launch_decode_shaped(const CtxArgs& a, unsigned units, int n_ranges, float scale_log2,
                                        int tiles_per_range, float* part_o, float2* part_ml, cudaStream_t stream) {
  static std::atomic<uint64_t> ready{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  constexpr size_t smem = dec_smem_bytes<kN>();
  static_assert(smem <= 232448, "shared memory exceeds the per-block maximum");
  if (!(ready.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(ctx_nvfp4_decode_kernel<kN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ready.fetch_or(bit, std::memory_order_acq_rel);
  }
  ctx_nvfp4_decode_kernel<kN><<<dim3(units, (unsigned)n_ranges), kThreads, smem, stream>>>(a, scale_log2,
                                                                                          tiles_per_range, part_o,
                                                                                          part_ml);
  return cudaGetLastError();
}

}  // namespace ctx
}  // namespace gqa
