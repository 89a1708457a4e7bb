// ctx_nvfp4.cu -- host side of the NVFP4 paged context attention for
// sm_103a: split-KV planning, launch of the attention kernel (ctx_kernel.cuh)
// at the production ring depths and of its split-KV merge, and the test
// export of the dequantisation.  (Other ring depths: ctx_study.cu.)
//
// Operation ("GB300 NVFP4 Context Attention: scale slot 조기 반납과 8단 packed
// K/V ring", introduction): see ctx_kernel.cuh.
#include <cuda.h>  // CUtensorMap and the cuTensorMapEncodeTiled prototype (resolved at run time)
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "ctx_kernel.cuh"
#include "ctx_decode.cuh"
#include "ctx_persistent.cuh"

namespace gqa {
using namespace ctx;
namespace {

// ---------------------------------------------------------------------------
// Debug export: dense gather of dequantised tokens, one thread per (token,
// KV head, 16-element block), through the attention kernel's own routines:
// the E4M3 bytes of the K path are written out, and the f16 values of the V
// path are checked on the device to be the same numbers (kErrSelfCheck when
// not), so a bit-exact test of the output covers both.
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
      const uint32_t sfb = sf[row * (kD / 16) + blk];
      const uint2 tab = nvfp4_scale_table(sfb);
      r = dequant16_e4m3(packed, tab);
      if ((sfb & 0x7fu) != 0x7fu) {  // (a NaN scale has no numbers to compare)
        const uint4 vt = nvfp4_f16_table(tab);
        const uint4 h0 = nvfp4_to_f16_8(packed.x, tab), h1 = nvfp4_to_f16_8(packed.y, tab);
        const uint4 t0 = nvfp4_to_f16_8_tables(packed.x, vt), t1 = nvfp4_to_f16_8_tables(packed.y, vt);
        const uint32_t e[4] = {f16x2_to_e4m3x2(h0.x) | (f16x2_to_e4m3x2(h0.y) << 16),
                               f16x2_to_e4m3x2(h0.z) | (f16x2_to_e4m3x2(h0.w) << 16),
                               f16x2_to_e4m3x2(h1.x) | (f16x2_to_e4m3x2(h1.y) << 16),
                               f16x2_to_e4m3x2(h1.z) | (f16x2_to_e4m3x2(h1.w) << 16)};
        const bool same = h0.x == t0.x && h0.y == t0.y && h0.z == t0.z && h0.w == t0.w && h1.x == t1.x &&
                          h1.y == t1.y && h1.z == t1.z && h1.w == t1.w;
        if (!same || e[0] != r.x || e[1] != r.y || e[2] != r.z || e[3] != r.w) atomicOr(&g_ctx_err, kErrSelfCheck);
      }
    } else {
      atomicOr(&g_ctx_err, kErrBadIndex);
    }
  }
  *reinterpret_cast<uint4*>(out + (((int64_t)b * max_kv + t) * kHkv + g) * kD + blk * 16) = r;
}

// ---------------------------------------------------------------------------
// Split-KV merge: one warp per (query row, head), lane l holding head-dim
// elements 4l .. 4l+3.  With M the largest m of the ranges that saw a key,
//   out = E4M3( sum_s 2^(m_s - M) O_s / (sum_s 2^(m_s - M) l_s) / out_scale ),
// and zeros when no range saw one (the same result as one unsplit pass, up
// to f32 rounding order).  Rows past qo_indptr[batch] belong to no unit
// (only with an invalid qo_indptr) and are written as zeros.
// ---------------------------------------------------------------------------
constexpr int kMergeWarps = 8;
constexpr int kCtxSplitTargetCtas = 152;  // one wave: one CTA per SM
constexpr int kMinTilesPerSplit = 8;      // a split amortises the CTA's start-up over >= 512 keys
// The persistent grid pays when units are short: it saves ~3 us of CTA start
// and end per unit and computes a tile ~8 % (~0.06 us) slower, so it breaks
// even near 47 tiles per unit.  Taken when every unit has at most 48 tiles
// (max_pages_per_seq <= 48) and there are at least two units per SM.
constexpr int64_t kPersistentMaxPages = 48;
constexpr int64_t kPersistentMinUnits = 2 * kCtxSplitTargetCtas;
constexpr int64_t kDecodeShapedMinPages = 16;

__global__ void __launch_bounds__(32 * kMergeWarps)
    ctx_merge_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml, uint8_t* __restrict__ out,
                     int64_t rows, int n_splits, float inv_out_scale, const int32_t* __restrict__ qo_indptr,
                     int64_t batch) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);  // token * 32 + head
  const int64_t last = qo_indptr[batch];
  // Launched as a programmatic dependent of the attention kernel: wait until
  // that grid has completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (row >= rows) return;
  if (row / kHq >= last) {
    reinterpret_cast<uint32_t*>(out + row * kD)[lane] = 0u;
    return;
  }
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

// The merge of the split partials, launched as a programmatic dependent grid:
// its launch overlaps the attention kernel's tail (it waits for that kernel
// with griddepcontrol.wait before it reads).
cudaError_t launch_merge(const float* part_o, const float2* part_ml, const CtxArgs& a, int64_t rows, int n_splits,
                         float inv_out_scale, cudaStream_t stream) {
  const int64_t mblocks = (rows + kMergeWarps - 1) / kMergeWarps;
  if (mblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
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
  return cudaLaunchKernelEx(&cfg, ctx_merge_kernel, part_o, part_ml, a.out, rows, n_splits, inv_out_scale,
                            a.qo_indptr, a.batch);
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

// Upper bound on the number of (sequence, 64-query block) units without
// reading qo_indptr on the host: sum_b ceil(q_b / 64) = sum_b floor((q_b + 63)
// / 64) <= floor((total_q + 63 batch) / 64).
static int64_t max_query_blocks(int64_t batch, int64_t total_q) {
  return (total_q + (int64_t)(kQB - 1) * batch) / kQB;
}

// Decode-shaped plan: units of rows/4 queries per (sequence, KV head), their
// KV ranges sized so that the units x ranges fill about four waves of the SMs
// (fewer waves leave a costly tail, more pay the CTA start-up more often) with
// at least 4 tiles (512 keys) per range.
static CtxPlan plan_decode_shaped(int64_t batch, int64_t total_q, int64_t max_pages_per_seq, int rows) {
  CtxPlan p{0, 1, 0, rows};
  const int64_t chunk = rows / 4;
  const int64_t units = (total_q + (chunk - 1) * batch) / chunk * kHkv;
  const int64_t tiles = (max_pages_per_seq + 1) / 2;
  int64_t ranges = (4 * kCtxSplitTargetCtas + units - 1) / units;
  const int64_t by_len = tiles / 4 > 0 ? tiles / 4 : 1;
  if (ranges > by_len) ranges = by_len;
  if (ranges > 32) ranges = 32;  // the merge holds one range per lane
  if (ranges < 1) ranges = 1;
  const int64_t tpr = (tiles + ranges - 1) / ranges;
  p.tiles_per_split = (int)tpr;
  p.n_splits = (int)((tiles + tpr - 1) / tpr);
  return p;
}

CtxPlan plan_ctx(int64_t batch, int64_t total_q, int64_t max_pages_per_seq) {
  CtxPlan p{0, 1, 0, 0};
  if (batch < 1 || total_q < 1 || max_pages_per_seq < 1) return p;
  // Decode-shaped calls (at most one query per sequence on average, over at
  // least 16 pages) take the transposed kernel, where it measured faster; a
  // test switch forces it, and a ring-depth study keeps the prefill kernel.
  const int mode = schedule_ctx_grid();
  const bool study = schedule_ctx_stages() || schedule_ctx_slots();
  if (mode == 3 || (mode == 0 && !study && total_q <= batch && max_pages_per_seq >= kDecodeShapedMinPages))
    return plan_decode_shaped(batch, total_q, max_pages_per_seq, 16);
  // Launched units (an upper bound on the real ones, as the grid below).
  const int64_t units = max_query_blocks(batch, total_q) * kHkv;
  p.persistent = units >= kPersistentMinUnits && max_pages_per_seq <= kPersistentMaxPages;
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
  if (plan.n_splits <= 1 && !plan.decode_rows) return 0;
  return (size_t)plan.n_splits * (size_t)total_q * kHq * (kD * sizeof(float) + sizeof(float2));
}

cudaError_t launch_ctx(const CtxArgs& a, const CtxPlan& plan, void* workspace, cudaStream_t stream) {
  const int64_t grid = max_query_blocks(a.batch, a.total_q) * kHkv;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const float scale_log2 = a.q_scale / sqrtf((float)kD) * 1.4426950408889634f;
  const float inv_out_scale = 1.f / a.out_scale;
  alignas(64) CUtensorMap q_map;
  cudaError_t e = make_q_map(a.q, a.total_q, &q_map);
  if (e != cudaSuccess) return e;
  const int64_t rows = a.total_q * kHq;
  if (plan.decode_rows) {
    if (!workspace || plan.tiles_per_split < 1 || plan.n_splits < 1 || plan.n_splits > 32)
      return cudaErrorInvalidValue;
    const int64_t chunk = plan.decode_rows / 4;
    const int64_t units = (a.total_q + (chunk - 1) * a.batch) / chunk * kHkv;
    if (units <= 0 || units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    float* part_o = static_cast<float*>(workspace);
    float2* part_ml = reinterpret_cast<float2*>(part_o + (size_t)plan.n_splits * rows * kD);
    if (plan.decode_rows != 16) return cudaErrorInvalidValue;
    e = launch_decode_shaped<16>(a, (unsigned)units, plan.n_splits, scale_log2, plan.tiles_per_split, part_o, part_ml,
                                 stream);
    if (e != cudaSuccess) return e;
    return launch_merge(part_o, part_ml, a, rows, plan.n_splits, inv_out_scale, stream);
  }
  if (plan.n_splits <= 1) {
    const int st = schedule_ctx_stages(), sl = schedule_ctx_slots();
    if ((st && st != kCtxStagesDefault) || (sl && sl != kCtxSlotsDefault))
      return launch_ctx_study(a, q_map, (unsigned)grid, scale_log2, inv_out_scale, st ? st : kCtxStagesDefault,
                              sl ? sl : kCtxSlotsDefault, stream);
    const int mode = schedule_ctx_grid();
    if (mode == 2 || (mode == 0 && plan.persistent))
      return launch_persistent<kCtxStagesPersistent, kCtxSlotsDefault>(a, q_map, grid, scale_log2, inv_out_scale,
                                                                          stream);
    return launch_attention<false, kCtxStagesDefault, kCtxSlotsDefault>(
        a, q_map, dim3((unsigned)grid, 1), scale_log2, inv_out_scale, 0, nullptr, nullptr, stream);
  }
  // the merge holds one range per lane
  if (!workspace || plan.tiles_per_split < 1 || plan.n_splits > 32) return cudaErrorInvalidValue;
  float* part_o = static_cast<float*>(workspace);
  float2* part_ml = reinterpret_cast<float2*>(part_o + (size_t)plan.n_splits * rows * kD);
  e = launch_attention<true, kCtxStagesSplit, kCtxSlotsDefault>(
      a, q_map, dim3((unsigned)grid, (unsigned)plan.n_splits), scale_log2, inv_out_scale, plan.tiles_per_split,
      part_o, part_ml, stream);
  if (e != cudaSuccess) return e;
  return launch_merge(part_o, part_ml, a, rows, plan.n_splits, inv_out_scale, stream);
}

cudaError_t ctx_read_errors(uint32_t* word) { return read_ctx_error_word(word); }

}  // namespace gqa
