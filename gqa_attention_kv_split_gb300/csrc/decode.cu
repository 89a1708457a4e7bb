// decode.cu -- FP16 grouped-query single-token decode, split-KV, for sm_103a.
//
// Operation ("NVIDIA SM110 GPU를 위한 실험적인 FP16 GQA 디코드 커널 추가",
// section 1, the sm110_gqa_decode docstring, and section 3, the SDPA
// comparator with enable_gqa=True):
//   for every batch b and query head h (KV head g = h / 4),
//   out[b,h,:] = softmax_t( q[b,h,:] . K[b,g,t,:] * q_scale / sqrt(128) ) V[b,g,t,:]
//   over t < sequence_lengths[b], with K = kv[b,0], V = kv[b,1].
//
// Design (GB300 first; the page's 256/384-thread SM110 kernels are prior art
// only):
//  * Split kernel, grid (splits, 8 KV heads, batch).  Each CTA streams one
//    chunk of tokens of one (b, g) slab.  A producer warp moves 16-token K and
//    V tiles (4 KB each, contiguous in HBM) into an 8-stage shared-memory ring
//    with 1-D bulk copies (TMA), completion tracked by mbarriers; the copies
//    carry an L2 evict-first hint because every K/V byte is read exactly once.
//  * Four consumer warps take whole stages round robin.  Each lane owns 8
//    head-dim elements of one token (16-byte shared loads), computes the 4
//    query heads' partial dot products, and a 16-lane reduce-scatter with
//    shuffles leaves each lane two complete logits.  Online softmax runs in
//    the exp2 domain (log2 e folded into the query scale), P is broadcast
//    through shared memory, and PV accumulates in fp32 registers.
//  * The four warps merge in shared memory and write one partial
//    (m, l, o[128]) per (b, h, split); a second tiny kernel merges the splits
//    by log-sum-exp.  When one split covers the capacity, the split kernel
//    normalises and writes fp16 directly and no merge is launched.
#include <cuda.h>  // CUcontext and the cuCtxGetCurrent prototype (resolved at run time)
#include <cuda_fp16.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace gqa {
namespace {

constexpr int kStageTok = 16;                         // tokens per ring stage
constexpr int kStagesDefault = 8;                     // ring depth of the production instances
constexpr int kComputeWarps = 4;                      // consumer warps
constexpr int kThreads = (kComputeWarps + 1) * 32;    // + one producer warp
constexpr int kRowBytes = kD * 2;                     // one token of one head: 256 B
constexpr int kStageBytes = kStageTok * kRowBytes;    // 4 KB of K (and of V)
constexpr int kChunkQuantum = kStageTok * kComputeWarps;  // 64 tokens
// Consumer warp w takes ring positions w, w + kComputeWarps, ...; with a ring
// depth that is a multiple of the warp count every stage belongs to one warp,
// so no warp can wait on a stage's barrier a phase ahead of the data (checked
// in the kernel template for every depth instantiated).

__device__ uint32_t g_decode_err;

template <int kStages>
struct DecodeSmem {
  alignas(1024) uint8_t k[kStages][kStageBytes];
  alignas(128) uint8_t v[kStages][kStageBytes];
  alignas(16) float p[kComputeWarps][kStageTok][kGroup];  // softmax weights, per warp
  alignas(16) float o[kComputeWarps][kGroup][kD];         // per-warp partial outputs
  float m[kComputeWarps][kGroup];
  float l[kComputeWarps][kGroup];
  alignas(8) uint64_t full[kStages];
  alignas(8) uint64_t empty[kStages];
};

// Producer epilogue: wait (bounded) until the copies of the last `issued`
// stages have landed, so that none lands after the CTA has exited.  In a
// normal run these phases completed long ago; after an expired wait the
// consumers may have stopped before consuming them.
template <int kStages>
__device__ __forceinline__ void drain_stages(DecodeSmem<kStages>& sm, int issued) {
  for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
    mbar_wait(smem_u32(&sm.full[i % kStages]), (i / kStages) & 1, &g_decode_err);
}

__device__ __forceinline__ void h8_to_f8(const uint4& u, float f[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __half22float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// kPaged: K/V come from 64-token HND pages through a block table (pages;
// kv unused); otherwise from the stacked cache kv [B, 2, 8, cap, 128].
template <bool kPaged, int kStages>
__global__ void __launch_bounds__(kThreads, 3)
    decode_split_kernel(const __half* __restrict__ q, const __half* __restrict__ kv, const DecodePages pages,
                        const int32_t* __restrict__ seq_lens, float* __restrict__ part_o,
                        float2* __restrict__ part_ml, __half* __restrict__ out, int64_t cap, int chunk,
                        int n_splits, float scale_log2, const int starve) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  static_assert(kStages % kComputeWarps == 0, "each ring stage must be owned by one consumer warp");
  DecodeSmem<kStages>& sm = *reinterpret_cast<DecodeSmem<kStages>*>(smem_raw);
  const int s = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int64_t len = seq_lens[b];
  len = len < 0 ? 0 : (len > cap ? cap : len);
  const int64_t t0 = (int64_t)s * chunk;
  const bool direct = (n_splits == 1);

  if (t0 >= len) {
    // Nothing to read.  In direct mode (single split) this is an empty
    // sequence: its output rows are zero.  Otherwise the merge covers it.
    if (direct && warp < kComputeWarps) {
      __half* dst = out + ((int64_t)b * kHq + g * kGroup + warp) * kD;
      reinterpret_cast<uint2*>(dst)[lane] = make_uint2(0u, 0u);
    }
    return;
  }
  const int n_tok = (int)((len < t0 + chunk ? len : t0 + chunk) - t0);
  const int n_st = (n_tok + kStageTok - 1) / kStageTok;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&sm.full[i]), 1);
      mbar_init(smem_u32(&sm.empty[i]), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kComputeWarps && kPaged) {
    // ---------------- producer (paged): a 16-token stage lies inside one
    // 64-token page (t0 is a multiple of 64).  The whole warp reads the
    // chunk's page numbers 32 at a time, one group ahead; lane 0 issues the
    // copies of each stage from (page, g, token % 64).
    const uint64_t pol = policy_evict_first();
    const int32_t* bt = pages.block_table + (int64_t)b * pages.max_pages_per_seq + t0 / kPage;
    const int n_pg = (n_tok + kPage - 1) / kPage;
    int cur = lane < n_pg ? bt[lane] : 0;
    int nxt = 32 + lane < n_pg ? bt[32 + lane] : 0;
    const __half* kp = static_cast<const __half*>(pages.k_pages);
    const __half* vp = static_cast<const __half*>(pages.v_pages);
    int issued = 0;
    for (int i = 0; i < (starve ? 0 : n_st); ++i) {
      const int pi = i / (kPage / kStageTok);  // page of this stage within the chunk
      if (pi > 0 && (pi & 31) == 0 && i % (kPage / kStageTok) == 0) {
        cur = nxt;
        nxt = pi + 32 + lane < n_pg ? bt[pi + 32 + lane] : 0;
      }
      int page = __shfl_sync(0xffffffffu, cur, pi & 31);
      const int st = i % kStages;
      if (i >= kStages &&
          !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.empty[st]), ((i / kStages) - 1) & 1, &g_decode_err)))
        break;
      if (lane == 0) {
        if (page < 0 || page >= pages.num_pages) {
          atomicOr(&g_decode_err, kErrBadIndex);
          page = 0;
        }
        const int nt = min(kStageTok, n_tok - i * kStageTok);
        const uint32_t bytes = (uint32_t)nt * kRowBytes;
        const int64_t off = (((int64_t)page * kHkv + g) * kPage + (i % (kPage / kStageTok)) * kStageTok) * kD;
        const uint32_t fb = smem_u32(&sm.full[st]);
        mbar_arrive_expect_tx(fb, 2 * bytes);
        bulk_g2s_hint(smem_u32(sm.k[st]), kp + off, bytes, fb, pol);
        bulk_g2s_hint(smem_u32(sm.v[st]), vp + off, bytes, fb, pol);
      }
      issued = i + 1;
      __syncwarp();
    }
    // No copy may land after the CTA exits (the consumers stop early when a
    // wait expires): wait for the last issued stages.
    if (lane == 0) drain_stages(sm, issued);
    return;
  }
  if (warp == kComputeWarps) {
    // ---------------- producer: bulk copies of K and V tiles --------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const __half* kbase = kv + (((int64_t)b * 2 + 0) * kHkv + g) * cap * kD + t0 * kD;
      const __half* vbase = kv + (((int64_t)b * 2 + 1) * kHkv + g) * cap * kD + t0 * kD;
      int issued = 0;
      for (int i = 0; i < (starve ? 0 : n_st); ++i) {
        const int st = i % kStages;
        if (i >= kStages && !mbar_wait(smem_u32(&sm.empty[st]), ((i / kStages) - 1) & 1, &g_decode_err)) break;
        const int nt = min(kStageTok, n_tok - i * kStageTok);
        const uint32_t bytes = (uint32_t)nt * kRowBytes;
        const uint32_t fb = smem_u32(&sm.full[st]);
        mbar_arrive_expect_tx(fb, 2 * bytes);
        bulk_g2s_hint(smem_u32(sm.k[st]), kbase + (int64_t)i * kStageTok * kD, bytes, fb, pol);
        bulk_g2s_hint(smem_u32(sm.v[st]), vbase + (int64_t)i * kStageTok * kD, bytes, fb, pol);
        issued = i + 1;
      }
      drain_stages(sm, issued);
    }
    return;
  }

  // ---------------- consumers ------------------------------------------------
  const int hw = lane >> 4;  // which token of a pair this half-warp reads
  const int j = lane & 15;   // head-dim slice [8j, 8j+8)
  const int jt = j >> 1;     // token-pair permutation used by the reduce-scatter
  const int jh = (j & 1) << 1;  // head permutation used by the reduce-scatter

  // Query slice, pre-scaled into the exp2 domain.  Position h holds head
  // (h ^ jh) so that every reduce-scatter step keeps its low half.
  float qf[kGroup][8];
#pragma unroll
  for (int h = 0; h < kGroup; ++h) {
    const uint4 u = *reinterpret_cast<const uint4*>(q + ((int64_t)b * kHq + g * kGroup + (h ^ jh)) * kD + 8 * j);
    h8_to_f8(u, qf[h]);
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[h][e] *= scale_log2;
  }

  float o[kGroup][8];
#pragma unroll
  for (int h = 0; h < kGroup; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) o[h][e] = 0.f;
  float m[kGroup] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  float lsum0 = 0.f, lsum1 = 0.f;  // running sums for heads jh, jh+1 (this lane's share)

  bool ok = true;
  for (int i = warp; i < n_st; i += kComputeWarps) {
    const int st = i % kStages;
    if (!mbar_wait(smem_u32(&sm.full[st]), (i / kStages) & 1, &g_decode_err)) {
      ok = false;
      break;
    }
    const int nt = min(kStageTok, n_tok - i * kStageTok);
    const uint8_t* ks = sm.k[st];
    const uint8_t* vs = sm.v[st];

    // ---- S = q K^T: 8 tokens x 4 heads of partial sums per lane.
    float part[32];
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) {
      const int tl = 2 * (ii ^ jt) + hw;
      float kf[8];
      h8_to_f8(*reinterpret_cast<const uint4*>(ks + tl * kRowBytes + 16 * j), kf);
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
        float acc = qf[h][0] * kf[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) acc = fmaf(qf[h][e], kf[e], acc);
        part[ii * kGroup + h] = acc;
      }
    }
    // Reduce-scatter over the 16 lanes of the half-warp: keep low half, send
    // high half.  Afterwards part[0..1] = full logits of token
    // 2*jt + hw for heads jh, jh+1.
#pragma unroll
    for (int k = 0; k < 16; ++k) part[k] += __shfl_xor_sync(0xffffffffu, part[k + 16], 8);
#pragma unroll
    for (int k = 0; k < 8; ++k) part[k] += __shfl_xor_sync(0xffffffffu, part[k + 8], 4);
#pragma unroll
    for (int k = 0; k < 4; ++k) part[k] += __shfl_xor_sync(0xffffffffu, part[k + 4], 2);
#pragma unroll
    for (int k = 0; k < 2; ++k) part[k] += __shfl_xor_sync(0xffffffffu, part[k + 2], 1);

    const int tok = 2 * jt + hw;
    float s0 = tok < nt ? part[0] : -INFINITY;
    float s1 = tok < nt ? part[1] : -INFINITY;

    // ---- tile maxima per head: the 16 lanes sharing jh, then swap pairs.
    float t0m = s0, t1m = s1;
#pragma unroll
    for (int mask = 2; mask <= 16; mask <<= 1) {
      t0m = fmaxf(t0m, __shfl_xor_sync(0xffffffffu, t0m, mask));
      t1m = fmaxf(t1m, __shfl_xor_sync(0xffffffffu, t1m, mask));
    }
    const float o0m = __shfl_xor_sync(0xffffffffu, t0m, 1);
    const float o1m = __shfl_xor_sync(0xffffffffu, t1m, 1);
    const bool lo_pair = (jh == 0);
    float tmax[kGroup];
    tmax[0] = lo_pair ? t0m : o0m;
    tmax[1] = lo_pair ? t1m : o1m;
    tmax[2] = lo_pair ? o0m : t0m;
    tmax[3] = lo_pair ? o1m : t1m;

    float mnew[kGroup], alpha[kGroup];
    bool rescale = false;
#pragma unroll
    for (int h = 0; h < kGroup; ++h) {
      mnew[h] = fmaxf(m[h], tmax[h]);
      rescale |= (mnew[h] != m[h]);
      alpha[h] = fast_exp2(m[h] - mnew[h]);
    }
    const float p0 = fast_exp2(s0 - (lo_pair ? mnew[0] : mnew[2]));
    const float p1 = fast_exp2(s1 - (lo_pair ? mnew[1] : mnew[3]));
    lsum0 = fmaf(lsum0, lo_pair ? alpha[0] : alpha[2], p0);
    lsum1 = fmaf(lsum1, lo_pair ? alpha[1] : alpha[3], p1);
    *reinterpret_cast<float2*>(&sm.p[warp][tok][jh]) = make_float2(p0, p1);
    __syncwarp();

    if (rescale) {
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] *= alpha[h];
        m[h] = mnew[h];
      }
    }

    // ---- O += P V over this lane's 8 tokens.
    if (nt == kStageTok) {
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        const int tl = 2 * ii + hw;
        const float4 pp = *reinterpret_cast<const float4*>(&sm.p[warp][tl][0]);
        float vf[8];
        h8_to_f8(*reinterpret_cast<const uint4*>(vs + tl * kRowBytes + 16 * j), vf);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          o[0][e] = fmaf(pp.x, vf[e], o[0][e]);
          o[1][e] = fmaf(pp.y, vf[e], o[1][e]);
          o[2][e] = fmaf(pp.z, vf[e], o[2][e]);
          o[3][e] = fmaf(pp.w, vf[e], o[3][e]);
        }
      }
    } else {
      for (int ii = 0; ii < 8; ++ii) {
        const int tl = 2 * ii + hw;
        if (tl >= nt) continue;  // rows past the copied tokens hold stale data
        const float4 pp = *reinterpret_cast<const float4*>(&sm.p[warp][tl][0]);
        float vf[8];
        h8_to_f8(*reinterpret_cast<const uint4*>(vs + tl * kRowBytes + 16 * j), vf);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          o[0][e] = fmaf(pp.x, vf[e], o[0][e]);
          o[1][e] = fmaf(pp.y, vf[e], o[1][e]);
          o[2][e] = fmaf(pp.z, vf[e], o[2][e]);
          o[3][e] = fmaf(pp.w, vf[e], o[3][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));
  }

  // ---- per-warp finalisation: full row sums, fold the two half-warps.
#pragma unroll
  for (int mask = 2; mask <= 16; mask <<= 1) {
    lsum0 += __shfl_xor_sync(0xffffffffu, lsum0, mask);
    lsum1 += __shfl_xor_sync(0xffffffffu, lsum1, mask);
  }
  const float l_o0 = __shfl_xor_sync(0xffffffffu, lsum0, 1);
  const float l_o1 = __shfl_xor_sync(0xffffffffu, lsum1, 1);
#pragma unroll
  for (int h = 0; h < kGroup; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], 16);
  if (hw == 0) {
#pragma unroll
    for (int h = 0; h < kGroup; ++h) {
      *reinterpret_cast<float4*>(&sm.o[warp][h][8 * j]) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
      *reinterpret_cast<float4*>(&sm.o[warp][h][8 * j + 4]) = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
    }
  }
  if (lane == 0) {  // lane 0 has jh = 0
#pragma unroll
    for (int h = 0; h < kGroup; ++h) sm.m[warp][h] = m[h];
    sm.l[warp][0] = lsum0;
    sm.l[warp][1] = lsum1;
    sm.l[warp][2] = l_o0;
    sm.l[warp][3] = l_o1;
  }
  named_bar_sync(1, kComputeWarps * 32);
  if (!ok) return;

  // ---- merge the four warps; warp w finishes head w of the group.
  const int h = warp;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, sm.m[w][h]);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < kComputeWarps; ++w) {
    const float f = fast_exp2(sm.m[w][h] - M);  // 0 for a warp that saw no token
    L = fmaf(sm.l[w][h], f, L);
    const float4 ow = *reinterpret_cast<const float4*>(&sm.o[w][h][4 * lane]);
    acc.x = fmaf(ow.x, f, acc.x);
    acc.y = fmaf(ow.y, f, acc.y);
    acc.z = fmaf(ow.z, f, acc.z);
    acc.w = fmaf(ow.w, f, acc.w);
  }
  const int64_t row = (int64_t)b * kHq + g * kGroup + h;
  if (direct) {
    const float inv = 1.f / L;
    __half2 lo = __floats2half2_rn(acc.x * inv, acc.y * inv);
    __half2 hi = __floats2half2_rn(acc.z * inv, acc.w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(out + row * kD)[lane] = pk;
  } else {
    reinterpret_cast<float4*>(part_o + (row * n_splits + s) * kD)[lane] = acc;
    if (lane == 0) part_ml[row * n_splits + s] = make_float2(M, L);
    // the partials are written: the merge grid may be launched (it waits for
    // this grid's completion before it reads them)
    asm volatile("griddepcontrol.launch_dependents;");
  }
}

// Log-sum-exp merge of the per-split partials.  One CTA of 4 warps per
// (b, h); warp w folds splits w, w+4, ...; lane owns 4 head-dim elements.
__global__ void __launch_bounds__(128)
    decode_merge_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                        const int32_t* __restrict__ seq_lens, __half* __restrict__ out, int64_t cap, int chunk,
                        int n_splits) {
  __shared__ float4 so[4][32];
  __shared__ float sm_m[4], sm_l[4];
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int64_t len = seq_lens[b];
  len = len < 0 ? 0 : (len > cap ? cap : len);
  const int nv = (int)((len + chunk - 1) / chunk);  // splits holding data
  const int64_t row = (int64_t)b * kHq + h;
  if (nv == 0) {
    if (warp == 0) reinterpret_cast<uint2*>(out + row * kD)[lane] = make_uint2(0u, 0u);
    return;
  }
  // Launched as a programmatic dependent of the split kernel: wait until that
  // grid has completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float2* ml = part_ml + row * n_splits;
  float M = -INFINITY;
  for (int s = warp; s < nv; s += 4) M = fmaxf(M, ml[s].x);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = warp; s < nv; s += 4) {
    const float2 v = ml[s];
    const float f = fast_exp2(v.x - M);
    L = fmaf(v.y, f, L);
    const float4 ov = reinterpret_cast<const float4*>(part_o + (row * n_splits + s) * kD)[lane];
    acc.x = fmaf(ov.x, f, acc.x);
    acc.y = fmaf(ov.y, f, acc.y);
    acc.z = fmaf(ov.z, f, acc.z);
    acc.w = fmaf(ov.w, f, acc.w);
  }
  so[warp][lane] = acc;
  if (lane == 0) {
    sm_m[warp] = M;
    sm_l[warp] = L;
  }
  __syncthreads();
  if (warp != 0) return;
  float MM = fmaxf(fmaxf(sm_m[0], sm_m[1]), fmaxf(sm_m[2], sm_m[3]));
  float LL = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float f = fast_exp2(sm_m[w] - MM);  // 0 for a warp with no split
    LL = fmaf(sm_l[w], f, LL);
    a.x = fmaf(so[w][lane].x, f, a.x);
    a.y = fmaf(so[w][lane].y, f, a.y);
    a.z = fmaf(so[w][lane].z, f, a.z);
    a.w = fmaf(so[w][lane].w, f, a.w);
  }
  const float inv = 1.f / LL;
  __half2 lo = __floats2half2_rn(a.x * inv, a.y * inv);
  __half2 hi = __floats2half2_rn(a.z * inv, a.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(out + row * kD)[lane] = pk;
}

// Launch of one instance of the split kernel; the dynamic-shared-memory
// opt-in is made once per device and instance (cached bitmask).
template <bool kPaged, int kStages>
cudaError_t launch_split(dim3 grid, cudaStream_t stream, const __half* q, const __half* kv, const DecodePages& pages,
                         const int32_t* seq_lens, float* part_o, float2* part_ml, __half* out, int64_t cap, int chunk,
                         int n_splits, float scale_log2, int starve) {
  static std::atomic<uint64_t> ready{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  constexpr size_t smem = sizeof(DecodeSmem<kStages>);
  if (!(ready.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(decode_split_kernel<kPaged, kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    ready.fetch_or(bit, std::memory_order_acq_rel);
  }
  decode_split_kernel<kPaged, kStages><<<grid, kThreads, smem, stream>>>(q, kv, pages, seq_lens, part_o, part_ml,
                                                                        out, cap, chunk, n_splits, scale_log2, starve);
  return cudaGetLastError();
}

}  // namespace

bool decode_schedule_supported(int stages) {
  return stages == 0 || stages == 4 || stages == kStagesDefault || stages == 12 || stages == 16;
}

DecodePlan plan_decode(int64_t batch, int64_t capacity) {
  DecodePlan p;
  // A split is a whole number of 64-token quanta (4 warps x 16-token stages).
  // Aim for about 4096 split CTAs over the whole capacity (many waves of 2
  // CTAs per SM on 152 SMs, so ragged lengths balance), with a power-of-two
  // split between 256 and 4096 tokens: larger splits cut the per-CTA prologue
  // and the partial-result traffic, smaller ones balance better.
  const double per_split = (double)batch * kHkv * (double)capacity / 4096.0;
  int chunk = 256;
  while (chunk < 4096 && chunk < per_split) chunk *= 2;
  const int64_t cap_q = (capacity + kChunkQuantum - 1) / kChunkQuantum * kChunkQuantum;
  if (cap_q <= chunk) chunk = (int)(cap_q > 0 ? cap_q : kChunkQuantum);
  p.chunk = chunk;
  p.n_splits = (int)((capacity + chunk - 1) / chunk);
  if (p.n_splits < 1) p.n_splits = 1;
  return p;
}

size_t decode_workspace_bytes(int64_t batch, const DecodePlan& plan) {
  if (plan.n_splits <= 1) return 0;
  const size_t rows = (size_t)batch * kHq * (size_t)plan.n_splits;
  return rows * kD * sizeof(float) + rows * sizeof(float2);
}

namespace {
cudaError_t launch_decode_any(const void* q, const void* kv, const DecodePages* pages, const int32_t* seq_lens,
                              void* out, int64_t batch, int64_t capacity, float q_scale, const DecodePlan& plan,
                              void* workspace, cudaStream_t stream) {
  cudaError_t e;
  const float scale_log2 = q_scale / sqrtf((float)kD) * 1.4426950408889634f;
  const int starve = starve_producers();
  float* part_o = nullptr;
  float2* part_ml = nullptr;
  if (plan.n_splits > 1) {
    const size_t rows = (size_t)batch * kHq * (size_t)plan.n_splits;
    part_o = static_cast<float*>(workspace);
    part_ml = reinterpret_cast<float2*>(part_o + rows * kD);
  }
  dim3 grid((unsigned)plan.n_splits, kHkv, (unsigned)batch);
  const __half* qh = static_cast<const __half*>(q);
  __half* oh = static_cast<__half*>(out);
  if (pages) {
    e = launch_split<true, kStagesDefault>(grid, stream, qh, nullptr, *pages, seq_lens, part_o, part_ml, oh, capacity,
                                           plan.chunk, plan.n_splits, scale_log2, starve);
  } else {
    const __half* kvh = static_cast<const __half*>(kv);
    const DecodePages none{};
    // ring depth: the production depth, or another instantiated depth chosen for a study (gqa_set_schedule)
    switch (schedule_decode_stages()) {
      case 4:
        e = launch_split<false, 4>(grid, stream, qh, kvh, none, seq_lens, part_o, part_ml, oh, capacity, plan.chunk,
                                   plan.n_splits, scale_log2, starve);
        break;
      case 12:
        e = launch_split<false, 12>(grid, stream, qh, kvh, none, seq_lens, part_o, part_ml, oh, capacity, plan.chunk,
                                    plan.n_splits, scale_log2, starve);
        break;
      case 16:
        e = launch_split<false, 16>(grid, stream, qh, kvh, none, seq_lens, part_o, part_ml, oh, capacity, plan.chunk,
                                    plan.n_splits, scale_log2, starve);
        break;
      default:
        e = launch_split<false, kStagesDefault>(grid, stream, qh, kvh, none, seq_lens, part_o, part_ml, oh, capacity,
                                                plan.chunk, plan.n_splits, scale_log2, starve);
    }
  }
  if (e != cudaSuccess) return e;
  if (plan.n_splits > 1) {
    // programmatic dependent launch: the merge's launch and its seq_lens read
    // overlap the split kernel's last CTAs (griddepcontrol.wait orders the rest)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kHq, (unsigned)batch);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, decode_merge_kernel, (const float*)part_o, (const float2*)part_ml, seq_lens,
                                static_cast<__half*>(out), (int64_t)capacity, (int)plan.chunk,
                                (int)plan.n_splits)) != cudaSuccess)
      return e;
  }
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_decode(const void* q, const void* kv, const int32_t* seq_lens, void* out, int64_t batch,
                          int64_t capacity, float q_scale, const DecodePlan& plan, void* workspace,
                          cudaStream_t stream) {
  return launch_decode_any(q, kv, nullptr, seq_lens, out, batch, capacity, q_scale, plan, workspace, stream);
}

cudaError_t launch_decode_paged(const void* q, const DecodePages& pages, const int32_t* seq_lens, void* out,
                                int64_t batch, float q_scale, const DecodePlan& plan, void* workspace,
                                cudaStream_t stream) {
  return launch_decode_any(q, nullptr, &pages, seq_lens, out, batch, pages.max_pages_per_seq * kPage, q_scale,
                           plan, workspace, stream);
}

// ---- bounded-wait check ---------------------------------------------------
//
// One thread waits on an mbarrier that nothing completes, through the same
// bounded wait every kernel here uses: after kWaitNs it records
// kErrWaitTimeout in the error word and returns.  No trap, no fault; the
// context stays usable.
namespace {
__global__ void wait_expiry_kernel() {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    mbar_wait(smem_u32(&bar), 0, &g_decode_err);  // phase 0 never completes
  }
}
}  // namespace

cudaError_t launch_wait_expiry(cudaStream_t stream) {
  wait_expiry_kernel<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

// ---- allocation-free variant ---------------------------------------------
//
// Scratch for gqa_decode_noalloc: the per-split partials live in this
// file-scope device array instead of a cudaMalloc'd workspace.  Every GPU
// that loads the library holds it until the process exits.  In host code the
// name g_static_scratch is only a stand-in for the symbol, never a device
// address: the address is looked up by cudaGetSymbolAddress (with the device
// current) and cached per device together with the CUDA context it belongs
// to.  A device reset destroys the primary context and reloads the module
// at a possibly different address, so a call that finds another context
// current looks the address up again.
static __device__ __align__(256) uint8_t g_static_scratch[kDecodeStaticScratchBytes];

namespace {
std::mutex g_static_mu;
struct StaticScratchAddr {
  void* addr = nullptr;
  CUcontext ctx = nullptr;
};
StaticScratchAddr g_static_addr[64];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
std::once_flag g_ctx_fn_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;

// The calling thread's current CUDA context (nullptr if the driver entry
// point is unavailable: the cache is then keyed by device alone).
CUcontext current_context() {
  std::call_once(g_ctx_fn_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  });
  CUcontext c = nullptr;
  if (g_ctx_get_current && g_ctx_get_current(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}
}  // namespace

cudaError_t launch_decode_static_scratch(const void* q, const void* kv, const int32_t* seq_lens, void* out,
                                         int64_t batch, int64_t capacity, float q_scale, const DecodePlan& plan,
                                         cudaStream_t stream) {
  if (decode_workspace_bytes(batch, plan) > kDecodeStaticScratchBytes) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_static_mu);
    const CUcontext ctx = current_context();
    StaticScratchAddr& c = g_static_addr[dev];
    if (c.addr == nullptr || c.ctx != ctx) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess) return e;
      c.addr = p;
      c.ctx = current_context();  // the lookup may have created the primary context
    }
    scratch = c.addr;
  }
  // The partials need no clearing: the merge reads only the splits that the
  // split kernel of this same call has written.
  return launch_decode(q, kv, seq_lens, out, batch, capacity, q_scale, plan, scratch, stream);
}

cudaError_t decode_read_errors(uint32_t* word) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  uint32_t zero = 0;
  if ((e = cudaMemcpyFromSymbol(word, g_decode_err, sizeof(uint32_t))) != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_decode_err, &zero, sizeof(uint32_t));
}

}  // namespace gqa
