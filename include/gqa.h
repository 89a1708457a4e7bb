/*
 * gqa.h -- C ABI of libgqa: grouped-query attention kernels for NVIDIA GB300
 * (sm_103a), head_dim 128, 32 query heads over 8 KV heads (4 query heads per
 * KV head).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every tensor argument is a plain pointer to a dense, row-major
 * (C-contiguous) array with the shape stated below.  All tensor pointers of
 * one call must be either
 *   - device memory of one and the same CUDA device (cudaMalloc'd, managed,
 *     or a PyTorch CUDA tensor's data pointer): the call enqueues its kernels
 *     on `stream` and returns without synchronising; or
 *   - host memory (pageable or pinned): the call stages the inputs into a
 *     library-owned device buffer on the calling thread's current device,
 *     runs the same kernels on `stream`, copies the output back, and
 *     synchronises `stream` before returning.
 * Mixing host and device pointers, or device pointers of two devices, is
 * rejected with GQA_ERR_DEVICE_MISMATCH.  Device pointers must be 16-byte
 * aligned (GQA_ERR_INVALID_ARG otherwise).
 *
 * Device selection.  For device pointers the call switches to the pointers'
 * device for its duration and restores the caller's current device on
 * return; the caller's current device need not match.  (The launcher
 * conventions of "FlashInfer NVFP4 QKV GEMM 최적화: SM103a Epilogue 통합 및 CUDA
 * 런처 개선", section 2: all tensors on one device, scoped device switch, no
 * current-device check, positive launch grid.)
 *
 * Ownership.  The caller owns every tensor.  The library owns a grow-only
 * scratch workspace per (device, stream), released by
 * gqa_release_workspace().  Two calls on the same stream are ordered by the
 * stream; calls on different streams use different workspaces.
 *
 * Errors.  Every entry point returns a gqa_status; GQA_OK means the work was
 * validated and enqueued (device pointers) or completed (host pointers).  On
 * any other status nothing was launched, and gqa_last_error() returns a
 * thread-local message.  No C++ exception crosses this boundary.
 */
#ifndef GQA_H_
#define GQA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA runtime headers; 0 is the legacy
 * default stream. */
typedef struct CUstream_st* gqa_stream_t;

typedef enum gqa_status {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = 1,        /* null pointer, bad size, dtype or strides, misalignment */
  GQA_ERR_UNSUPPORTED = 2,        /* shape outside what the kernels handle */
  GQA_ERR_UNSUPPORTED_SHAPE = 2,  /* (the same code, by the name the descriptor entry points use) */
  GQA_ERR_DEVICE_MISMATCH = 3,    /* pointers on different devices / host+device mix */
  GQA_ERR_CUDA = 4,               /* a CUDA runtime call failed */
  GQA_ERR_OOM = 5,                /* workspace allocation failed */
  GQA_ERR_TIMEOUT = 6             /* a kernel's bounded wait expired (see gqa_check_device_errors) */
} gqa_status;

/*
 * Tensor descriptor of the *_t entry points below: the pointer entry points'
 * arguments plus what a C caller would otherwise have to get right unaided --
 * element type, placement, shape and strides -- so that the library can
 * check them (a DLPack-like record of our own).
 *
 *   data     first element (device or host memory)
 *   dtype    a gqa_dtype
 *   device   CUDA device ordinal of `data`, or -1 for host memory; checked
 *            against where the memory really is
 *   ndim     number of dimensions (<= 6)
 *   shape    extents; strides in elements, dense row-major required (a
 *            dimension of extent 1 may carry any stride)
 */
typedef enum gqa_dtype {
  GQA_F16 = 1,   /* IEEE binary16 */
  GQA_E4M3 = 2,  /* OCP FP8 E4M3 ("fn") bytes */
  GQA_U8 = 3,    /* bytes: packed E2M1 pairs, or E4M3 codes given as raw bytes */
  GQA_I32 = 4,
  GQA_F32 = 5
} gqa_dtype;

typedef struct gqa_tensor {
  void* data;
  int32_t dtype;
  int32_t device;
  int32_t ndim;
  int64_t shape[6];
  int64_t strides[6];
} gqa_tensor;

/* Message for the last non-OK status returned on this thread. */
const char* gqa_last_error(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int gqa_version(void);

/*
 * gqa_decode -- FP16 grouped-query attention for one new token per sequence.
 *
 * Defined by "NVIDIA SM110 GPU를 위한 실험적인 FP16 GQA 디코드 커널 추가",
 * section 1 (the sm110_gqa_decode API and its docstring) and section 3 (the
 * scaled_dot_product_attention comparator with enable_gqa=True):
 *
 *   out[b,h,:] = sum_t softmax_t(s) * V[b,g,t,:],   g = h / 4,
 *   s_t = (q[b,h,:] . K[b,g,t,:]) * q_scale / sqrt(128),   0 <= t < len_b,
 *   K = kv[b,0,...], V = kv[b,1,...],  len_b = clamp(seq_lens[b], 0, capacity).
 *
 *   q         [batch, 32, 128]                 float16
 *   kv        [batch, 2, 8, capacity, 128]     float16 (K stacked over V)
 *   seq_lens  [batch]                          int32 (read by the kernels)
 *   out       [batch, 32, 128]                 float16, written; caller-owned
 *   batch     1 .. 65535
 *   capacity  1 .. 2^31 - 1 tokens per sequence
 *   q_scale   finite; multiplies the standard 1/sqrt(128) scale
 *
 * A sequence of length 0 produces a zero row.  Element offsets are computed
 * in 64-bit, so kv may hold 2^31 or more elements.
 */
gqa_status gqa_decode(const void* q, const void* kv, const int32_t* seq_lens, void* out, int64_t batch,
                      int64_t capacity, float q_scale, gqa_stream_t stream);

/*
 * gqa_decode_noalloc -- gqa_decode that allocates no memory.  (An addition
 * of this library; the pages have no counterpart.)
 *
 * Same operation, arguments, layouts and results as gqa_decode, for callers
 * that cannot allocate device memory at call time: engines that reserve
 * nearly all of HBM up front for their KV cache and own every byte through
 * their own allocator (a late cudaMalloc would fail or fragment it), and
 * latency-critical loops that must not block in cudaMalloc/cudaFree, which
 * can synchronise the device.  The split partials go to a file-scope device
 * array of 16 MiB instead of the library workspace; every GPU that loads
 * libgqa holds that array until the process exits.
 *
 *   - Device pointers only (host buffers would need staging memory):
 *     GQA_ERR_UNSUPPORTED otherwise.
 *   - Rejects, with GQA_ERR_UNSUPPORTED and a message naming the sizes, a
 *     (batch, capacity) whose partials exceed 16 MiB: batch * 32 * splits *
 *     520 bytes, splits as reported by gqa_decode_plan.  The benchmark shapes
 *     (64 x 8192, 8 x 131072) need 8.5 MB.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and caches it with the device's current CUDA
 *     context; a call that finds another context current (after
 *     cudaDeviceReset, which reloads the library's device code) looks it up
 *     again.  Make the first call on a device, and the first after a reset,
 *     before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind (nothing in it needs to start at zero).  Calls whose kernels
 *     overlap on the GPU -- on different streams, without ordering -- race on
 *     it; order them on one stream or with events.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
gqa_status gqa_decode_noalloc(const void* q, const void* kv, const int32_t* seq_lens, void* out, int64_t batch,
                              int64_t capacity, float q_scale, gqa_stream_t stream);

/*
 * gqa_decode_paged -- the operation of gqa_decode over a paged K/V cache:
 * the same split-KV kernels, each 16-token K/V tile gathered through the
 * block table ("NVIDIA SM110 GPU를 위한 실험적인 FP16 GQA 디코드 커널 추가",
 * section 1, for the operation; the page layout is the one the context
 * attention uses, "GB300 NVFP4 Context Attention: scale slot 조기 반납과 8단
 * packed K/V ring", introduction, with fp16 values).
 *
 *   q            [batch, 32, 128]                 fp16
 *   k_pages      [num_pages, 8, 64, 128]          fp16, HND: page p, KV head g,
 *   v_pages      [num_pages, 8, 64, 128]          slot s holds token 64*p' + s
 *                of the sequence whose block_table row maps logical page p'
 *                to p
 *   block_table  [batch, max_pages_per_seq]       int32; entries for logical
 *                pages < ceil(len_b / 64) must be in [0, num_pages)
 *   seq_lens     [batch]                          int32, read on the device,
 *                clamped to [0, 64 * max_pages_per_seq]
 *   out          [batch, 32, 128]                 fp16, written
 *
 * Splits as gqa_decode_plan(batch, 64 * max_pages_per_seq) reports.  Same
 * placement rules as gqa_decode (one device, or all host buffers: staged,
 * synchronous, table entries checked on the host).  A page index outside
 * [0, num_pages) met on the device is not read: page 0 is used instead and
 * bit 1 of the error word (gqa_check_device_errors) is set.  Errors:
 * GQA_ERR_UNSUPPORTED for batch outside [1, 65535], GQA_ERR_INVALID_ARG for
 * bad sizes, NULL or misaligned pointers, a non-finite q_scale.
 */
gqa_status gqa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                            const int32_t* seq_lens, void* out, int64_t batch, int64_t num_pages,
                            int64_t max_pages_per_seq, float q_scale, gqa_stream_t stream);

/*
 * Descriptor forms of gqa_decode, gqa_decode_paged and nvfp4_paged_ctx_attn:
 * the same operations, with every tensor given as a gqa_tensor.  Before any
 * CUDA work they check each descriptor's dtype, rank, shape (including the
 * extents the tensors share: batch, pages, total_q), dense row-major strides
 * and non-null data -- GQA_ERR_INVALID_ARG, or GQA_ERR_UNSUPPORTED_SHAPE for
 * an extent the kernels do not handle (32 query heads, 8 KV heads, head dim
 * 128, 64-token pages) -- then that all tensors share one `device` field and
 * that the memory really is there (GQA_ERR_DEVICE_MISMATCH); then they call
 * the pointer form with the sizes read from the shapes.  Accepted dtypes:
 * q/kv/out/pages of the decodes GQA_F16; q_fp8, k_sf, v_sf, out_fp8 GQA_E4M3
 * or GQA_U8; k_fp4, v_fp4 GQA_U8; seq_lens, block_table, qo_indptr, kv_lens
 * GQA_I32.  Shapes as in the pointer forms' comments.
 */
gqa_status gqa_decode_t(const gqa_tensor* q, const gqa_tensor* kv, const gqa_tensor* seq_lens, gqa_tensor* out,
                        float q_scale, gqa_stream_t stream);
gqa_status gqa_decode_paged_t(const gqa_tensor* q, const gqa_tensor* k_pages, const gqa_tensor* v_pages,
                              const gqa_tensor* block_table, const gqa_tensor* seq_lens, gqa_tensor* out,
                              float q_scale, gqa_stream_t stream);
gqa_status nvfp4_paged_ctx_attn_t(const gqa_tensor* q_fp8, float q_scale, const gqa_tensor* k_fp4,
                                  const gqa_tensor* k_sf, const gqa_tensor* v_fp4, const gqa_tensor* v_sf,
                                  const gqa_tensor* block_table, const gqa_tensor* qo_indptr,
                                  const gqa_tensor* kv_lens, gqa_tensor* out_fp8, float out_scale,
                                  gqa_stream_t stream);

/*
 * gqa_decode_plan -- how gqa_decode splits the KV sequence for a given batch
 * and capacity (chosen from these two only; the lengths stay on the device):
 * *tokens_per_split tokens per split CTA, *num_splits splits per sequence,
 * *num_launches kernels per call (1 when one split covers the capacity: the
 * split kernel then writes the output itself; 2 otherwise: split + merge).
 * Any output pointer may be NULL.
 */
gqa_status gqa_decode_plan(int64_t batch, int64_t capacity, int32_t* tokens_per_split, int32_t* num_splits,
                           int32_t* num_launches);

/*
 * nvfp4_paged_ctx_attn -- paged context (prefill) attention with FP8-E4M3
 * query and output and NVFP4 K/V pages, bottom-right causal.
 *
 * Defined by "GB300 NVFP4 Context Attention: scale slot 조기 반납과 8단 packed
 * K/V ring", introduction: FP8 (E4M3) query/output, NVFP4 K/V pages with
 * E4M3 block scales, dequantised to E4M3 in shared memory, head dim 128,
 * bottom-right causal mask, HND page layout.  For sequence b with
 * q_len_b = qo_indptr[b+1] - qo_indptr[b] and kv_len_b = kv_lens[b], query i
 * (row qo_indptr[b] + i) sees key j iff j <= kv_len_b - q_len_b + i, and
 *
 *   Kq[b,g,j,d] = E4M3_rne_sat( e2m1(code) * e4m3(scale) )   (same for Vq)
 *   s_j  = (q[row,h,:] . Kq[b,g,j,:]) * q_scale / sqrt(128),  g = h / 4
 *   out[row,h,:] = E4M3_rne_sat( (sum_j softmax_j(s) Vq[b,g,j,:]) / out_scale )
 *
 *   q_fp8        [total_q, 32, 128]                E4M3 bytes
 *   k_fp4, v_fp4 [num_pages, 8, 64, 64]            uint8, two E2M1 codes per
 *                byte, head-dim element 2i in the low nibble of byte i;
 *                page p, KV head g, slot s holds token 64*p' + s of the
 *                sequence whose block_table row maps logical page p' to p
 *   k_sf, v_sf   [num_pages, 8, 64, 8]             E4M3 scale per 16 head-dim
 *                elements (element d uses scale d / 16)
 *   block_table  [batch, max_pages_per_seq]        int32 physical page ids;
 *                entries for logical pages < ceil(kv_len_b / 64) must be in
 *                [0, num_pages)
 *   qo_indptr    [batch + 1]                       int32, qo_indptr[0] = 0,
 *                non-decreasing, qo_indptr[batch] = total_q
 *   kv_lens      [batch]                           int32, 0 <= kv_len_b <=
 *                64 * max_pages_per_seq
 *   out_fp8      [total_q, 32, 128]                E4M3 bytes, written
 *   q_scale, out_scale  finite, out_scale > 0
 *
 * qo_indptr and kv_lens are read on the device only.  A query row that sees
 * no key (q_len_b > kv_len_b) is written as zeros.  The kernels check
 * qo_indptr on the device: when it does not run non-decreasing from 0 to
 * total_q they set bit 2 of the error word (gqa_check_device_errors), write
 * rows past qo_indptr[batch] as zeros, and never read or write a row outside
 * [0, total_q); the other rows are then unspecified.  (With host buffers the
 * library checks qo_indptr, kv_lens and the used block-table entries before
 * staging and returns GQA_ERR_INVALID_ARG.)  The softmax numerators P
 * enter the P*V product as f16 (V's dequantised E4M3 values widened to f16
 * exactly), so the result matches the exact value to within the output's
 * E4M3 rounding.
 *
 * Work is split by (sequence, block of 64 queries, KV head).  When those
 * units cannot fill the GPU (short query lengths: decode-like calls, few
 * sequences), each unit's KV range is also split, as gqa_ctx_plan reports,
 * and a second kernel merges the ranges; the partials live in the library's
 * workspace for (device, stream) (n_splits * total_q * 32 * 520 bytes).
 */
gqa_status nvfp4_paged_ctx_attn(const void* q_fp8, float q_scale, const void* k_fp4, const void* k_sf,
                                const void* v_fp4, const void* v_sf, const int32_t* block_table,
                                const int32_t* qo_indptr, const int32_t* kv_lens, void* out_fp8,
                                float out_scale, int64_t batch, int64_t total_q, int64_t num_pages,
                                int64_t max_pages_per_seq, gqa_stream_t stream);

/*
 * gqa_ctx_plan -- how nvfp4_paged_ctx_attn divides the KV range of each work
 * unit, chosen from batch, total_q and max_pages_per_seq only (qo_indptr and
 * kv_lens stay on the device): *tiles_per_split 64-key tiles per split CTA
 * (0 when unsplit), *num_splits ranges per unit, *num_launches kernels per
 * call (0 when total_q = 0; 1 unsplit; 2 with the merge).  The split is used
 * when at most 76 units (8 KV heads x floor((total_q + 63 * batch) / 64), a
 * bound on the (sequence, 64-query block) pairs) can be launched and every
 * range keeps at least 8 tiles.  *persistent = 1 when an unsplit call runs
 * the persistent grid (one CTA per SM walks a share of the units; same
 * result, bit for bit): at least 304 units and max_pages_per_seq <= 48, i.e.
 * short units, whose per-CTA start and end it saves.  *decode_shaped = 1 when
 * the call runs the decode-shaped kernel instead (total_q <= batch, i.e. at
 * most one query per sequence on average, and max_pages_per_seq >= 16): S and
 * P V computed transposed (keys on the MMA's M dimension, 4 queries x 4 heads
 * on N), always as KV ranges (*num_splits of *tiles_per_split 128-key tiles)
 * that the merge combines (*num_launches = 2); its outputs meet the same
 * parity bar but are not bit-identical to the other kernels'.  Any output
 * pointer may be NULL.
 */
gqa_status gqa_ctx_plan(int64_t batch, int64_t total_q, int64_t max_pages_per_seq, int32_t* tiles_per_split,
                        int32_t* num_splits, int32_t* num_launches, int32_t* persistent, int32_t* decode_shaped);

/*
 * gqa_set_ctx_grid -- test switch: the grid of later unsplit
 * nvfp4_paged_ctx_attn calls (all devices, all threads; process-wide).
 * GQA_CTX_GRID_PLANNED (0) = as gqa_ctx_plan reports; GQA_CTX_GRID_PER_UNIT
 * (1) = one CTA per work unit; GQA_CTX_GRID_PERSISTENT (2) = the persistent
 * grid; GQA_CTX_GRID_DECODE_SHAPED (3) = the decode-shaped kernel for every
 * call.  The first two compute the same result, bit for bit; split-KV calls
 * and the ring-depth study instances (gqa_set_schedule) always run one CTA
 * per unit.  Modes 1 and 2 keep calls off the decode-shaped kernel.
 * GQA_ERR_INVALID_ARG for another mode (nothing changes).
 */
enum { GQA_CTX_GRID_PLANNED = 0, GQA_CTX_GRID_PER_UNIT = 1, GQA_CTX_GRID_PERSISTENT = 2, GQA_CTX_GRID_DECODE_SHAPED = 3 };
gqa_status gqa_set_ctx_grid(int mode);

/*
 * gqa_debug_dequant_pages -- test export of the context kernel's NVFP4 ->
 * E4M3 dequantisation (same device routine), gathered through the block
 * table into a dense array.
 *
 *   fp4          [num_pages, 8, 64, 64]   uint8 (as k_fp4 above)
 *   sf           [num_pages, 8, 64, 8]    E4M3 (as k_sf above)
 *   block_table  [batch, max_pages_per_seq] int32
 *   kv_lens      [batch] int32 (device-read)
 *   out_e4m3     [batch, max_kv, 8, 128]  E4M3 bytes: token t of sequence b
 *                for t < min(kv_lens[b], max_kv); zero bytes beyond
 */
gqa_status gqa_debug_dequant_pages(const void* fp4, const void* sf, const int32_t* block_table,
                                   const int32_t* kv_lens, void* out_e4m3, int64_t batch, int64_t num_pages,
                                   int64_t max_pages_per_seq, int64_t max_kv, gqa_stream_t stream);

/*
 * gqa_check_device_errors -- synchronise `device` and return (then clear)
 * the kernels' device error word in *word: bit 0 = a bounded wait expired,
 * bit 1 = an out-of-range page index was skipped, bit 2 = qo_indptr was not
 * non-decreasing from 0 to total_q, bit 3 = the dequantisation export's
 * self-check failed.  Returns GQA_ERR_TIMEOUT when bit 0 is set,
 * GQA_ERR_INVALID_ARG when another bit is set, GQA_OK when the word is 0.
 * After a timeout the outputs of the affected call are unspecified; every
 * kernel waits for the tensor-core operations and copies it started before
 * it releases its resources, so later calls are unaffected.
 */
gqa_status gqa_check_device_errors(int device, uint32_t* word);

/*
 * gqa_debug_wait_expiry -- test export of the kernels' failure detection: on
 * `device`, one CTA waits on an mbarrier that nothing completes, through the
 * bounded wait every kernel of the library uses.  After about 2 s the wait
 * gives up, sets bit 0 of the error word and the kernel returns; a following
 * gqa_check_device_errors reports GQA_ERR_TIMEOUT.  No trap and no fault: the
 * context stays usable.  Asynchronous on `stream`.
 */
gqa_status gqa_debug_wait_expiry(int device, gqa_stream_t stream);

/*
 * gqa_set_schedule -- study switch: ring depths of later launches (all
 * devices, all threads; process-wide).  Every depth computes the same
 * result, bit for bit -- the invariant "GB300 NVFP4 Context Attention: scale
 * slot 조기 반납과 8단 packed K/V ring" checks for its ring changes (section 2
 * and its results section) -- so a schedule changes only speed.
 *
 *   ctx_packed_stages, ctx_kv_slots  packed NVFP4 page stages and dequantised
 *       K/V tile slots of the one-CTA-per-unit context attention kernel of
 *       unsplit calls; 0 = its production depth (4 stages, 4 slots).
 *       Instantiated (stages, slots): (4,4) (6,4) (8,4) (10,4) (6,3) (12,3)
 *       (6,5) (6,2).  A non-production depth runs every unsplit call on the
 *       one-CTA-per-unit grid; split-KV calls and the persistent grid always
 *       run their production depths (6 stages, 4 slots).
 *   decode_stages  16-token K/V stages of the decode ring (stacked cache);
 *       0 = the production depth 8; also 4, 12, 16.  The paged decode always
 *       runs depth 8.
 *
 * GQA_ERR_UNSUPPORTED for a depth that is not instantiated (nothing changes).
 */
gqa_status gqa_set_schedule(int ctx_packed_stages, int ctx_kv_slots, int decode_stages);

/*
 * gqa_debug_starve_producers -- test switch of the failure detection.  With
 * enable != 0, every later launch (all devices, all threads) runs its
 * kernels with producers that issue no copies: each consumer's bounded wait
 * expires after about 2 s, every role leaves its loop, the CTA drains what it
 * started, frees its tensor memory and exits, and gqa_check_device_errors
 * reports GQA_ERR_TIMEOUT.  enable = 0 restores normal operation.  Not for
 * concurrent use with real work: the setting is process-wide.
 */
gqa_status gqa_debug_starve_producers(int enable);

/* Free every workspace the library holds (all devices and streams).  The
 * caller must ensure no libgqa work is still running. */
gqa_status gqa_release_workspace(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_H_ */
