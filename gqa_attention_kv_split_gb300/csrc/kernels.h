// kernels.h -- internal launch interface between the C-ABI layer (api.cpp)
// and the CUDA translation units.  Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>  // CUtensorMap
#include <cuda_runtime.h>

namespace gqa {

// Limit of every bounded wait in the kernels: 2 s.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

// Process-wide test switch of the bounded-wait machinery (set by
// gqa_debug_starve_producers): the kernels' producers issue no copies, so
// every consumer's wait expires.
int starve_producers();

// Ring depths used by the next launches (set by gqa_set_schedule for
// studies; 0 = the production depth).  Only the instantiated depths are
// accepted: see gqa_set_schedule in include/gqa.h.
int schedule_ctx_stages();
int schedule_ctx_slots();
int schedule_decode_stages();
// Grid of unsplit context calls: 0 = as planned, 1 = one CTA per unit, 2 = persistent.
int schedule_ctx_grid();
bool ctx_schedule_supported(int stages, int slots);
bool decode_schedule_supported(int stages);

// ---- FP16 split-KV decode -------------------------------------------------

struct DecodePlan {
  int chunk;     // tokens per split (multiple of 64)
  int n_splits;  // splits per sequence = ceil(capacity / chunk)
};

// Split planning from the capacity and batch only (sequence lengths live on
// the device and are never read by the host).
DecodePlan plan_decode(int64_t batch, int64_t capacity);

// Bytes of scratch the decode needs for its per-split partial results
// (0 when a single split covers the capacity).
size_t decode_workspace_bytes(int64_t batch, const DecodePlan& plan);

// Paged K/V for the decode: 64-token pages in HND order, one block table row
// per sequence (the same page layout as the context attention's NVFP4
// pages, with fp16 values).
struct DecodePages {
  const void* k_pages;         // [num_pages, 8, 64, 128] f16
  const void* v_pages;         // [num_pages, 8, 64, 128] f16
  const int32_t* block_table;  // [batch, max_pages_per_seq]
  int64_t num_pages;
  int64_t max_pages_per_seq;   // capacity = 64 * max_pages_per_seq
};

// The paged decode: the same split-KV kernels, K/V tiles gathered through
// the block table (capacity = 64 * pages.max_pages_per_seq).
cudaError_t launch_decode_paged(const void* q, const DecodePages& pages, const int32_t* seq_lens, void* out,
                                int64_t batch, float q_scale, const DecodePlan& plan, void* workspace,
                                cudaStream_t stream);

cudaError_t launch_decode(const void* q, const void* kv, const int32_t* seq_lens, void* out, int64_t batch,
                          int64_t capacity, float q_scale, const DecodePlan& plan, void* workspace,
                          cudaStream_t stream);

// Size of the file-scope device array that gqa_decode_noalloc uses for the
// per-split partials (16 MiB per GPU that loads the library).
constexpr size_t kDecodeStaticScratchBytes = size_t(16) << 20;

// launch_decode with the partials in that static array.  On the first call
// on a device (which must be current) it looks up the array's device address
// with cudaGetSymbolAddress and caches it.  Returns cudaErrorInvalidValue if
// the plan needs more than kDecodeStaticScratchBytes.  Allocates nothing.
cudaError_t launch_decode_static_scratch(const void* q, const void* kv, const int32_t* seq_lens, void* out,
                                         int64_t batch, int64_t capacity, float q_scale, const DecodePlan& plan,
                                         cudaStream_t stream);

// Test export: one CTA whose single wait never completes; its bounded wait
// expires after kWaitNs and sets kErrWaitTimeout in the decode error word.
cudaError_t launch_wait_expiry(cudaStream_t stream);

// Reads and clears the decode kernels' device error word on the current
// device (synchronises the device).
cudaError_t decode_read_errors(uint32_t* word);

// ---- NVFP4 paged context attention --------------------------------------

struct CtxArgs {
  const uint8_t* q;            // [total_q, 32, 128] E4M3
  const uint8_t* k_fp4;        // [num_pages, 8, 64, 64]
  const uint8_t* k_sf;         // [num_pages, 8, 64, 8]
  const uint8_t* v_fp4;
  const uint8_t* v_sf;
  const int32_t* block_table;  // [batch, max_pages_per_seq]
  const int32_t* qo_indptr;    // [batch + 1]
  const int32_t* kv_lens;      // [batch]
  uint8_t* out;                // [total_q, 32, 128] E4M3
  float q_scale;
  float out_scale;
  int64_t batch;
  int64_t total_q;
  int64_t num_pages;
  int64_t max_pages_per_seq;
  int starve;                  // test switch: the producer issues no copies
};

// Split-KV plan of the context attention, from host-known sizes only: when
// the (sequence, 64-query block, KV head) units cannot fill the GPU (short
// query lengths: decode-like and few-sequence calls), each unit's KV tiles
// are divided into n_splits contiguous ranges of tiles_per_split tiles, one
// CTA each, and a merge kernel combines the ranges' partial results.
struct CtxPlan {
  int tiles_per_split;  // 64-key tiles per split CTA (0 when n_splits == 1)
  int n_splits;         // 1: the attention kernel writes the output itself
  int persistent;       // unsplit calls of short units: the persistent grid (one CTA per SM walks its units)
  int decode_rows;      // decode-shaped calls: query rows per unit of the transposed kernel (16 or 32), else 0;
                        // then n_splits KV ranges of tiles_per_split 128-key tiles, always merged
};

CtxPlan plan_ctx(int64_t batch, int64_t total_q, int64_t max_pages_per_seq);

// Bytes of scratch for the split partials (0 when n_splits == 1):
// n_splits * total_q * 32 heads * (128 f32 of O + f32 m + f32 l).
size_t ctx_workspace_bytes(int64_t total_q, const CtxPlan& plan);

cudaError_t launch_ctx(const CtxArgs& a, const CtxPlan& plan, void* workspace, cudaStream_t stream);

cudaError_t launch_dequant_pages(const uint8_t* fp4, const uint8_t* sf, const int32_t* block_table,
                                 const int32_t* kv_lens, uint8_t* out, int64_t batch, int64_t num_pages,
                                 int64_t max_pages_per_seq, int64_t max_kv, cudaStream_t stream);

cudaError_t ctx_read_errors(uint32_t* word);

// The unsplit attention kernel at ring depths other than the production ones
// (a separate translation unit); cudaErrorNotSupported for a combination that
// is not instantiated.
cudaError_t launch_ctx_study(const CtxArgs& a, const CUtensorMap& q_map, unsigned grid, float scale_log2,
                             float inv_out_scale, int stages, int slots, cudaStream_t stream);
cudaError_t ctx_study_read_errors(uint32_t* word);

}  // namespace gqa
