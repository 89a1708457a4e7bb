// api.cpp -- the C ABI of libgqa (include/gqa.h): argument validation,
// device scoping, workspace ownership, host-buffer staging and launch.
//
// Launcher conventions follow "FlashInfer NVFP4 QKV GEMM 최적화: SM103a
// Epilogue 통합 및 CUDA 런처 개선", section 2: every tensor must sit on one
// device (checked per pointer), the call switches to that device and
// restores the caller's (no current-device check), and a launch grid must be
// positive.  Nothing here computes attention; every step of the path runs in
// the kernels of decode.cu and ctx_nvfp4.cu.
#include "../../include/gqa.h"

#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <initializer_list>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "kernels.h"

namespace {

thread_local std::string t_last_error;

gqa_status fail(gqa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

gqa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GQA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

#define GQA_CUDA_TRY(expr, what)                   \
  do {                                             \
    cudaError_t _e = (expr);                       \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

// Switches to `dev` for the lifetime of the object; restores the previous
// current device afterwards.
class ScopedDevice {
 public:
  explicit ScopedDevice(int dev) {
    if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
    if (prev_ != dev) ok_ = (cudaSetDevice(dev) == cudaSuccess);
    switched_ = (prev_ != dev) && ok_;
  }
  ~ScopedDevice() {
    if (switched_ && prev_ >= 0) cudaSetDevice(prev_);
  }
  bool ok() const { return ok_; }

 private:
  int prev_ = -1;
  bool ok_ = true;
  bool switched_ = false;
};

// Where a pointer lives.
struct Where {
  bool host;
  int device;
};

gqa_status classify(const void* p, const char* name, Where* w) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "cudaPointerGetAttributes");
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    w->host = false;
    w->device = a.device;
  } else {
    w->host = true;
    w->device = -1;
  }
  (void)name;
  return GQA_OK;
}

struct Arg {
  const void* p;
  const char* name;
  size_t align;
};

constexpr int kAnyDevice = -1000;  // no expectation from a descriptor

// All pointers on one side: either the same device or all host; when
// `expect` is a descriptor's device field (-1 = host), the memory must be
// there.
gqa_status locate(const std::vector<Arg>& args, Where* out, int expect = kAnyDevice) {
  for (const Arg& a : args)
    if (a.p == nullptr) return fail(GQA_ERR_INVALID_ARG, "%s is a null pointer", a.name);
  Where first{};
  for (size_t i = 0; i < args.size(); ++i) {
    Where w;
    gqa_status st = classify(args[i].p, args[i].name, &w);
    if (st != GQA_OK) return st;
    if (i == 0) {
      first = w;
    } else if (w.host != first.host || w.device != first.device) {
      return fail(GQA_ERR_DEVICE_MISMATCH, "%s is on %s %d but %s is on %s %d", args[i].name,
                  w.host ? "host" : "device", w.device, args[0].name, first.host ? "host" : "device",
                  first.device);
    }
    if (!w.host && (reinterpret_cast<uintptr_t>(args[i].p) % args[i].align) != 0)
      return fail(GQA_ERR_INVALID_ARG, "%s is not %zu-byte aligned", args[i].name, args[i].align);
  }
  const int real = first.host ? -1 : first.device;
  if (expect != kAnyDevice && real != expect)
    return fail(GQA_ERR_DEVICE_MISMATCH, "the descriptors say device %d but the memory is on %s %d", expect,
                first.host ? "host" : "device", first.device);
  *out = first;
  return GQA_OK;
}

// Grow-only device scratch per (device, stream).
struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;

gqa_status workspace(int dev, cudaStream_t stream, size_t bytes, void** out) {
  *out = nullptr;
  if (bytes == 0) return GQA_OK;
  std::lock_guard<std::mutex> lk(g_ws_mu);
  Workspace& w = g_ws[{dev, reinterpret_cast<uintptr_t>(stream)}];
  if (w.bytes < bytes) {
    if (w.ptr) {
      // Work queued on this stream may still use the old buffer.
      cudaError_t e = cudaStreamSynchronize(stream);
      if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
      cudaFree(w.ptr);
      w.ptr = nullptr;
      w.bytes = 0;
    }
    size_t grow = bytes + bytes / 8;
    cudaError_t e = cudaMalloc(&w.ptr, grow);
    if (e != cudaSuccess) {
      cudaGetLastError();
      w.ptr = nullptr;
      e = cudaMalloc(&w.ptr, bytes);
      if (e != cudaSuccess) {
        cudaGetLastError();
        w.ptr = nullptr;
        return fail(GQA_ERR_OOM, "workspace of %zu bytes: %s", bytes, cudaGetErrorString(e));
      }
      grow = bytes;
    }
    w.bytes = grow;
  }
  *out = w.ptr;
  return GQA_OK;
}

// Carves 256-byte aligned sub-buffers out of one allocation.
struct Carver {
  size_t off = 0;
  size_t take(size_t bytes) {
    size_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  }
};

// ---- tensor descriptors (gqa_tensor) ---------------------------------------

const char* dtype_name(int32_t d) {
  switch (d) {
    case GQA_F16: return "f16";
    case GQA_E4M3: return "e4m3";
    case GQA_U8: return "u8";
    case GQA_I32: return "i32";
    case GQA_F32: return "f32";
    default: return "unknown";
  }
}

// Structural check of one descriptor: non-null, an accepted dtype, the rank
// and shape asked for (-1 = any extent, returned in got[]), dense row-major
// strides (in elements; a dimension of extent 1 may carry any stride).  No
// CUDA call: it runs before anything touches the device.
gqa_status check_desc(const gqa_tensor* t, const char* name, std::initializer_list<int32_t> dtypes,
                      std::initializer_list<int64_t> shape, int64_t* got = nullptr) {
  if (!t) return fail(GQA_ERR_INVALID_ARG, "%s: null descriptor", name);
  if (!t->data) return fail(GQA_ERR_INVALID_ARG, "%s is a null pointer", name);
  bool dt_ok = false;
  for (int32_t d : dtypes) dt_ok |= (t->dtype == d);
  if (!dt_ok) {
    std::string want;
    for (int32_t d : dtypes) want += std::string(want.empty() ? "" : " or ") + dtype_name(d);
    return fail(GQA_ERR_INVALID_ARG, "%s has dtype %s; expected %s", name, dtype_name(t->dtype), want.c_str());
  }
  const int nd = (int)shape.size();
  if (t->ndim != nd) return fail(GQA_ERR_INVALID_ARG, "%s has %d dimensions; expected %d", name, t->ndim, nd);
  int i = 0;
  for (int64_t want : shape) {
    const int64_t have = t->shape[i];
    if (have < 0) return fail(GQA_ERR_INVALID_ARG, "%s: negative extent in dimension %d", name, i);
    if (want >= 0 && have != want)
      return fail(GQA_ERR_UNSUPPORTED_SHAPE, "%s has extent %lld in dimension %d; expected %lld", name,
                  (long long)have, i, (long long)want);
    if (got) got[i] = have;
    ++i;
  }
  int64_t expect = 1;
  for (int d = nd - 1; d >= 0; --d) {
    if (t->shape[d] != 1 && t->strides[d] != expect)
      return fail(GQA_ERR_INVALID_ARG, "%s is not dense row-major (stride %lld in dimension %d; expected %lld)", name,
                  (long long)t->strides[d], d, (long long)expect);
    expect *= t->shape[d];
  }
  return GQA_OK;
}

// Every descriptor names the same device (or all host memory, device -1).
// (Where the memory really is, is checked once per pointer by locate().)
gqa_status check_devices(std::initializer_list<std::pair<const gqa_tensor*, const char*>> ts) {
  const gqa_tensor* first = ts.begin()->first;
  for (const auto& t : ts)
    if (t.first->device != first->device)
      return fail(GQA_ERR_DEVICE_MISMATCH, "%s is on device %d but %s is on device %d", t.second, t.first->device,
                  ts.begin()->second, first->device);
  return GQA_OK;
}

#define GQA_TRY(expr)                  \
  do {                                 \
    gqa_status _s = (expr);            \
    if (_s != GQA_OK) return _s;       \
  } while (0)

std::atomic<int> g_starve{0};
std::atomic<int> g_ctx_stages{0}, g_ctx_slots{0}, g_decode_stages{0}, g_ctx_grid{0};

}  // namespace

namespace gqa {
int starve_producers() { return g_starve.load(std::memory_order_relaxed); }
int schedule_ctx_stages() { return g_ctx_stages.load(std::memory_order_relaxed); }
int schedule_ctx_slots() { return g_ctx_slots.load(std::memory_order_relaxed); }
int schedule_decode_stages() { return g_decode_stages.load(std::memory_order_relaxed); }
int schedule_ctx_grid() { return g_ctx_grid.load(std::memory_order_relaxed); }
}  // namespace gqa

extern "C" {

const char* gqa_last_error(void) { return t_last_error.c_str(); }

int gqa_version(void) { return 302; }  // 0.3.2: decode-shaped context kernel, gqa_ctx_plan(decode_shaped)

namespace {
gqa_status decode_impl(const void* q, const void* kv, const int32_t* seq_lens, void* out, int64_t batch,
                       int64_t capacity, float q_scale, gqa_stream_t stream_, int expect) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (batch < 1 || batch > 65535) return fail(GQA_ERR_UNSUPPORTED, "batch %lld outside [1, 65535]", (long long)batch);
  if (capacity < 1 || capacity > 2147483647LL)
    return fail(GQA_ERR_UNSUPPORTED, "capacity %lld outside [1, 2^31-1]", (long long)capacity);
  if (!std::isfinite(q_scale)) return fail(GQA_ERR_INVALID_ARG, "q_scale is not finite");
  Where where;
  gqa_status st =
      locate({{q, "q", 16}, {kv, "kv", 16}, {seq_lens, "seq_lens", 4}, {out, "out", 16}}, &where, expect);
  if (st != GQA_OK) return st;

  const gqa::DecodePlan plan = gqa::plan_decode(batch, capacity);
  if (plan.n_splits < 1) return fail(GQA_ERR_INVALID_ARG, "launch grid must be positive");
  const size_t part_bytes = gqa::decode_workspace_bytes(batch, plan);

  if (!where.host) {
    ScopedDevice sd(where.device);
    if (!sd.ok()) return fail(GQA_ERR_CUDA, "cannot switch to device %d", where.device);
    void* ws = nullptr;
    if ((st = workspace(where.device, stream, part_bytes, &ws)) != GQA_OK) return st;
    GQA_CUDA_TRY(gqa::launch_decode(q, kv, seq_lens, out, batch, capacity, q_scale, plan, ws, stream),
                 "decode launch");
    return GQA_OK;
  }

  // Host buffers: stage the bytes the kernels read, run, copy the result back.
  int dev = 0;
  GQA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  const size_t q_bytes = (size_t)batch * 32 * 128 * 2;
  const size_t slab = (size_t)capacity * 128 * 2;  // one (b, K|V, g) slab
  const size_t kv_bytes = (size_t)batch * 2 * 8 * slab;
  Carver c;
  const size_t o_q = c.take(q_bytes), o_kv = c.take(kv_bytes), o_len = c.take((size_t)batch * 4),
               o_out = c.take(q_bytes), o_part = c.take(part_bytes);
  void* ws = nullptr;
  if ((st = workspace(dev, stream, c.off, &ws)) != GQA_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(ws);
  GQA_CUDA_TRY(cudaMemcpyAsync(base + o_q, q, q_bytes, cudaMemcpyHostToDevice, stream), "copy q");
  GQA_CUDA_TRY(cudaMemcpyAsync(base + o_len, seq_lens, (size_t)batch * 4, cudaMemcpyHostToDevice, stream),
               "copy seq_lens");
  for (int64_t b = 0; b < batch; ++b) {
    int64_t len = seq_lens[b];
    len = len < 0 ? 0 : (len > capacity ? capacity : len);
    if (len == 0) continue;
    // 16 slabs (K and V of 8 heads), each with its first len tokens.
    const uint8_t* src = static_cast<const uint8_t*>(kv) + (size_t)b * 16 * slab;
    GQA_CUDA_TRY(cudaMemcpy2DAsync(base + o_kv + (size_t)b * 16 * slab, slab, src, slab, (size_t)len * 256, 16,
                                   cudaMemcpyHostToDevice, stream),
                 "copy kv");
  }
  GQA_CUDA_TRY(gqa::launch_decode(base + o_q, base + o_kv, reinterpret_cast<const int32_t*>(base + o_len),
                                  base + o_out, batch, capacity, q_scale, plan,
                                  part_bytes ? base + o_part : nullptr, stream),
               "decode launch");
  GQA_CUDA_TRY(cudaMemcpyAsync(out, base + o_out, q_bytes, cudaMemcpyDeviceToHost, stream), "copy out");
  GQA_CUDA_TRY(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
  return GQA_OK;
}

gqa_status decode_paged_impl(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                             const int32_t* seq_lens, void* out, int64_t batch, int64_t num_pages,
                             int64_t max_pages_per_seq, float q_scale, gqa_stream_t stream_, int expect) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (batch < 1 || batch > 65535) return fail(GQA_ERR_UNSUPPORTED, "batch %lld outside [1, 65535]", (long long)batch);
  if (num_pages < 1 || num_pages > 2147483647LL)
    return fail(GQA_ERR_INVALID_ARG, "num_pages %lld out of range", (long long)num_pages);
  if (max_pages_per_seq < 1 || max_pages_per_seq > (2147483647LL / 64))
    return fail(GQA_ERR_INVALID_ARG, "max_pages_per_seq %lld out of range", (long long)max_pages_per_seq);
  if (!std::isfinite(q_scale)) return fail(GQA_ERR_INVALID_ARG, "q_scale is not finite");
  Where where;
  gqa_status st = locate({{q, "q", 16},
                          {k_pages, "k_pages", 16},
                          {v_pages, "v_pages", 16},
                          {block_table, "block_table", 4},
                          {seq_lens, "seq_lens", 4},
                          {out, "out", 16}},
                         &where, expect);
  if (st != GQA_OK) return st;
  const int64_t capacity = max_pages_per_seq * 64;
  const gqa::DecodePlan plan = gqa::plan_decode(batch, capacity);
  if (plan.n_splits < 1) return fail(GQA_ERR_INVALID_ARG, "launch grid must be positive");
  const size_t part_bytes = gqa::decode_workspace_bytes(batch, plan);
  gqa::DecodePages pg;
  pg.num_pages = num_pages;
  pg.max_pages_per_seq = max_pages_per_seq;

  if (!where.host) {
    ScopedDevice sd(where.device);
    if (!sd.ok()) return fail(GQA_ERR_CUDA, "cannot switch to device %d", where.device);
    void* ws = nullptr;
    if ((st = workspace(where.device, stream, part_bytes, &ws)) != GQA_OK) return st;
    pg.k_pages = k_pages;
    pg.v_pages = v_pages;
    pg.block_table = block_table;
    GQA_CUDA_TRY(gqa::launch_decode_paged(q, pg, seq_lens, out, batch, q_scale, plan, ws, stream),
                 "paged decode launch");
    return GQA_OK;
  }

  // Host buffers: the host can read the lengths and the table, so check the
  // pages a sequence uses, then stage everything and run.
  for (int64_t b = 0; b < batch; ++b) {
    int64_t len = seq_lens[b];
    len = len < 0 ? 0 : (len > capacity ? capacity : len);
    for (int64_t p = 0; p < (len + 63) / 64; ++p) {
      const int32_t pgid = block_table[b * max_pages_per_seq + p];
      if (pgid < 0 || pgid >= num_pages)
        return fail(GQA_ERR_INVALID_ARG, "block_table[%lld][%lld] = %d outside [0, num_pages)", (long long)b,
                    (long long)p, pgid);
    }
  }
  int dev = 0;
  GQA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  const size_t q_bytes = (size_t)batch * 32 * 128 * 2;
  const size_t page_bytes = (size_t)num_pages * 8 * 64 * 128 * 2;
  const size_t bt_bytes = (size_t)batch * max_pages_per_seq * 4;
  Carver c;
  const size_t o_q = c.take(q_bytes), o_k = c.take(page_bytes), o_v = c.take(page_bytes), o_bt = c.take(bt_bytes),
               o_len = c.take((size_t)batch * 4), o_out = c.take(q_bytes), o_part = c.take(part_bytes);
  void* ws = nullptr;
  if ((st = workspace(dev, stream, c.off, &ws)) != GQA_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(ws);
  const std::pair<size_t, std::pair<const void*, size_t>> copies[] = {
      {o_q, {q, q_bytes}},       {o_k, {k_pages, page_bytes}},        {o_v, {v_pages, page_bytes}},
      {o_bt, {block_table, bt_bytes}}, {o_len, {seq_lens, (size_t)batch * 4}}};
  for (const auto& cp : copies)
    GQA_CUDA_TRY(cudaMemcpyAsync(base + cp.first, cp.second.first, cp.second.second, cudaMemcpyHostToDevice, stream),
                 "stage input");
  pg.k_pages = base + o_k;
  pg.v_pages = base + o_v;
  pg.block_table = reinterpret_cast<const int32_t*>(base + o_bt);
  GQA_CUDA_TRY(gqa::launch_decode_paged(base + o_q, pg, reinterpret_cast<const int32_t*>(base + o_len), base + o_out,
                                        batch, q_scale, plan, part_bytes ? base + o_part : nullptr, stream),
               "paged decode launch");
  GQA_CUDA_TRY(cudaMemcpyAsync(out, base + o_out, q_bytes, cudaMemcpyDeviceToHost, stream), "copy out");
  GQA_CUDA_TRY(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
  return GQA_OK;
}
}  // namespace

gqa_status gqa_decode(const void* q, const void* kv, const int32_t* seq_lens, void* out, int64_t batch,
                      int64_t capacity, float q_scale, gqa_stream_t stream) {
  return decode_impl(q, kv, seq_lens, out, batch, capacity, q_scale, stream, kAnyDevice);
}

gqa_status gqa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                            const int32_t* seq_lens, void* out, int64_t batch, int64_t num_pages,
                            int64_t max_pages_per_seq, float q_scale, gqa_stream_t stream) {
  return decode_paged_impl(q, k_pages, v_pages, block_table, seq_lens, out, batch, num_pages, max_pages_per_seq,
                           q_scale, stream, kAnyDevice);
}

gqa_status gqa_decode_noalloc(const void* q, const void* kv, const int32_t* seq_lens, void* out, int64_t batch,
                              int64_t capacity, float q_scale, gqa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (batch < 1 || batch > 65535) return fail(GQA_ERR_UNSUPPORTED, "batch %lld outside [1, 65535]", (long long)batch);
  if (capacity < 1 || capacity > 2147483647LL)
    return fail(GQA_ERR_UNSUPPORTED, "capacity %lld outside [1, 2^31-1]", (long long)capacity);
  if (!std::isfinite(q_scale)) return fail(GQA_ERR_INVALID_ARG, "q_scale is not finite");
  Where where;
  gqa_status st = locate({{q, "q", 16}, {kv, "kv", 16}, {seq_lens, "seq_lens", 4}, {out, "out", 16}}, &where);
  if (st != GQA_OK) return st;
  if (where.host)
    return fail(GQA_ERR_UNSUPPORTED,
                "gqa_decode_noalloc takes device pointers only (host buffers would need staging memory)");
  const gqa::DecodePlan plan = gqa::plan_decode(batch, capacity);
  const size_t need = gqa::decode_workspace_bytes(batch, plan);
  if (need > gqa::kDecodeStaticScratchBytes)
    return fail(GQA_ERR_UNSUPPORTED,
                "batch %lld x capacity %lld needs %zu bytes of split partials; the static scratch holds %zu "
                "(use gqa_decode)",
                (long long)batch, (long long)capacity, need, gqa::kDecodeStaticScratchBytes);
  ScopedDevice sd(where.device);
  if (!sd.ok()) return fail(GQA_ERR_CUDA, "cannot switch to device %d", where.device);
  GQA_CUDA_TRY(gqa::launch_decode_static_scratch(q, kv, seq_lens, out, batch, capacity, q_scale, plan, stream),
               "decode launch (static scratch)");
  return GQA_OK;
}

gqa_status gqa_decode_plan(int64_t batch, int64_t capacity, int32_t* tokens_per_split, int32_t* num_splits,
                           int32_t* num_launches) {
  if (batch < 1 || batch > 65535) return fail(GQA_ERR_UNSUPPORTED, "batch %lld outside [1, 65535]", (long long)batch);
  if (capacity < 1 || capacity > 2147483647LL)
    return fail(GQA_ERR_UNSUPPORTED, "capacity %lld outside [1, 2^31-1]", (long long)capacity);
  const gqa::DecodePlan plan = gqa::plan_decode(batch, capacity);
  if (tokens_per_split) *tokens_per_split = plan.chunk;
  if (num_splits) *num_splits = plan.n_splits;
  if (num_launches) *num_launches = plan.n_splits > 1 ? 2 : 1;
  return GQA_OK;
}

gqa_status gqa_ctx_plan(int64_t batch, int64_t total_q, int64_t max_pages_per_seq, int32_t* tiles_per_split,
                        int32_t* num_splits, int32_t* num_launches, int32_t* persistent, int32_t* decode_shaped) {
  if (batch < 1 || batch > (1 << 20)) return fail(GQA_ERR_UNSUPPORTED, "batch %lld outside [1, 2^20]", (long long)batch);
  if (total_q < 0 || total_q > 2147483647LL) return fail(GQA_ERR_INVALID_ARG, "total_q %lld out of range", (long long)total_q);
  if (max_pages_per_seq < 1 || max_pages_per_seq > (2147483647LL / 64))
    return fail(GQA_ERR_INVALID_ARG, "max_pages_per_seq %lld out of range", (long long)max_pages_per_seq);
  const gqa::CtxPlan plan = gqa::plan_ctx(batch, total_q, max_pages_per_seq);
  if (tiles_per_split) *tiles_per_split = plan.tiles_per_split;
  if (num_splits) *num_splits = plan.n_splits;
  if (num_launches) *num_launches = total_q == 0 ? 0 : (plan.n_splits > 1 || plan.decode_rows ? 2 : 1);
  if (persistent) *persistent = total_q > 0 && plan.n_splits == 1 && plan.persistent && !plan.decode_rows ? 1 : 0;
  if (decode_shaped) *decode_shaped = total_q > 0 && plan.decode_rows ? 1 : 0;
  return GQA_OK;
}

namespace {
gqa_status ctx_impl(const void* q_fp8, float q_scale, const void* k_fp4, const void* k_sf, const void* v_fp4,
                    const void* v_sf, const int32_t* block_table, const int32_t* qo_indptr, const int32_t* kv_lens,
                    void* out_fp8, float out_scale, int64_t batch, int64_t total_q, int64_t num_pages,
                    int64_t max_pages_per_seq, gqa_stream_t stream_, int expect) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (batch < 1 || batch > (1 << 20))
    return fail(GQA_ERR_UNSUPPORTED, "batch %lld outside [1, 2^20]", (long long)batch);
  if (total_q < 0 || total_q > 2147483647LL) return fail(GQA_ERR_INVALID_ARG, "total_q %lld out of range", (long long)total_q);
  if (num_pages < 1 || num_pages > 2147483647LL) return fail(GQA_ERR_INVALID_ARG, "num_pages %lld out of range", (long long)num_pages);
  if (max_pages_per_seq < 1 || max_pages_per_seq > (2147483647LL / 64))
    return fail(GQA_ERR_INVALID_ARG, "max_pages_per_seq %lld out of range", (long long)max_pages_per_seq);
  if (!std::isfinite(q_scale)) return fail(GQA_ERR_INVALID_ARG, "q_scale is not finite");
  if (!std::isfinite(out_scale) || !(out_scale > 0.f)) return fail(GQA_ERR_INVALID_ARG, "out_scale must be finite and > 0");
  Where where;
  gqa_status st = locate({{q_fp8, "q_fp8", 16},
                          {k_fp4, "k_fp4", 16},
                          {k_sf, "k_sf", 16},
                          {v_fp4, "v_fp4", 16},
                          {v_sf, "v_sf", 16},
                          {block_table, "block_table", 4},
                          {qo_indptr, "qo_indptr", 4},
                          {kv_lens, "kv_lens", 4},
                          {out_fp8, "out_fp8", 16}},
                         &where, expect);
  if (st != GQA_OK) return st;

  gqa::CtxArgs a;
  a.starve = gqa::starve_producers();
  a.q_scale = q_scale;
  a.out_scale = out_scale;
  a.batch = batch;
  a.total_q = total_q;
  a.num_pages = num_pages;
  a.max_pages_per_seq = max_pages_per_seq;
  const gqa::CtxPlan plan = gqa::plan_ctx(batch, total_q, max_pages_per_seq);
  const size_t part_bytes = gqa::ctx_workspace_bytes(total_q, plan);

  if (!where.host) {
    if (total_q == 0) return GQA_OK;
    ScopedDevice sd(where.device);
    if (!sd.ok()) return fail(GQA_ERR_CUDA, "cannot switch to device %d", where.device);
    void* part = nullptr;
    if (part_bytes && (st = workspace(where.device, stream, part_bytes, &part)) != GQA_OK) return st;
    a.q = static_cast<const uint8_t*>(q_fp8);
    a.k_fp4 = static_cast<const uint8_t*>(k_fp4);
    a.k_sf = static_cast<const uint8_t*>(k_sf);
    a.v_fp4 = static_cast<const uint8_t*>(v_fp4);
    a.v_sf = static_cast<const uint8_t*>(v_sf);
    a.block_table = block_table;
    a.qo_indptr = qo_indptr;
    a.kv_lens = kv_lens;
    a.out = static_cast<uint8_t*>(out_fp8);
    cudaError_t e = gqa::launch_ctx(a, plan, part, stream);
    if (e == cudaErrorNotSupported) return fail(GQA_ERR_UNSUPPORTED, "context kernel not available in this build");
    GQA_CUDA_TRY(e, "ctx launch");
    return GQA_OK;
  }

  // Host buffers: the host can read the metadata, so check it fully.
  if (qo_indptr[0] != 0 || qo_indptr[batch] != total_q)
    return fail(GQA_ERR_INVALID_ARG, "qo_indptr must start at 0 and end at total_q");
  for (int64_t b = 0; b < batch; ++b) {
    if (qo_indptr[b + 1] < qo_indptr[b]) return fail(GQA_ERR_INVALID_ARG, "qo_indptr decreases at %lld", (long long)b);
    if (kv_lens[b] < 0 || (int64_t)kv_lens[b] > 64 * max_pages_per_seq)
      return fail(GQA_ERR_INVALID_ARG, "kv_lens[%lld] = %d out of range", (long long)b, kv_lens[b]);
    const int64_t np = ((int64_t)kv_lens[b] + 63) / 64;
    for (int64_t p = 0; p < np; ++p) {
      const int32_t pg = block_table[b * max_pages_per_seq + p];
      if (pg < 0 || pg >= num_pages)
        return fail(GQA_ERR_INVALID_ARG, "block_table[%lld][%lld] = %d outside [0, num_pages)", (long long)b,
                    (long long)p, pg);
    }
  }
  if (total_q == 0) return GQA_OK;
  int dev = 0;
  GQA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  const size_t q_bytes = (size_t)total_q * 32 * 128;
  const size_t fp4_bytes = (size_t)num_pages * 8 * 64 * 64;
  const size_t sf_bytes = (size_t)num_pages * 8 * 64 * 8;
  const size_t bt_bytes = (size_t)batch * max_pages_per_seq * 4;
  Carver c;
  const size_t o_q = c.take(q_bytes), o_kf = c.take(fp4_bytes), o_ks = c.take(sf_bytes), o_vf = c.take(fp4_bytes),
               o_vs = c.take(sf_bytes), o_bt = c.take(bt_bytes), o_qi = c.take((size_t)(batch + 1) * 4),
               o_kl = c.take((size_t)batch * 4), o_out = c.take(q_bytes), o_part = c.take(part_bytes);
  void* ws = nullptr;
  if ((st = workspace(dev, stream, c.off, &ws)) != GQA_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(ws);
  const std::pair<size_t, std::pair<const void*, size_t>> copies[] = {
      {o_q, {q_fp8, q_bytes}},  {o_kf, {k_fp4, fp4_bytes}}, {o_ks, {k_sf, sf_bytes}},
      {o_vf, {v_fp4, fp4_bytes}}, {o_vs, {v_sf, sf_bytes}},   {o_bt, {block_table, bt_bytes}},
      {o_qi, {qo_indptr, (size_t)(batch + 1) * 4}}, {o_kl, {kv_lens, (size_t)batch * 4}}};
  for (const auto& cp : copies)
    GQA_CUDA_TRY(cudaMemcpyAsync(base + cp.first, cp.second.first, cp.second.second, cudaMemcpyHostToDevice, stream),
                 "stage input");
  a.q = base + o_q;
  a.k_fp4 = base + o_kf;
  a.k_sf = base + o_ks;
  a.v_fp4 = base + o_vf;
  a.v_sf = base + o_vs;
  a.block_table = reinterpret_cast<const int32_t*>(base + o_bt);
  a.qo_indptr = reinterpret_cast<const int32_t*>(base + o_qi);
  a.kv_lens = reinterpret_cast<const int32_t*>(base + o_kl);
  a.out = base + o_out;
  cudaError_t e = gqa::launch_ctx(a, plan, part_bytes ? base + o_part : nullptr, stream);
  if (e == cudaErrorNotSupported) return fail(GQA_ERR_UNSUPPORTED, "context kernel not available in this build");
  GQA_CUDA_TRY(e, "ctx launch");
  GQA_CUDA_TRY(cudaMemcpyAsync(out_fp8, base + o_out, q_bytes, cudaMemcpyDeviceToHost, stream), "copy out");
  GQA_CUDA_TRY(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
  return GQA_OK;
}
}  // namespace

gqa_status nvfp4_paged_ctx_attn(const void* q_fp8, float q_scale, const void* k_fp4, const void* k_sf,
                                const void* v_fp4, const void* v_sf, const int32_t* block_table,
                                const int32_t* qo_indptr, const int32_t* kv_lens, void* out_fp8, float out_scale,
                                int64_t batch, int64_t total_q, int64_t num_pages, int64_t max_pages_per_seq,
                                gqa_stream_t stream) {
  return ctx_impl(q_fp8, q_scale, k_fp4, k_sf, v_fp4, v_sf, block_table, qo_indptr, kv_lens, out_fp8, out_scale,
                  batch, total_q, num_pages, max_pages_per_seq, stream, kAnyDevice);
}

gqa_status gqa_debug_dequant_pages(const void* fp4, const void* sf, const int32_t* block_table,
                                   const int32_t* kv_lens, void* out_e4m3, int64_t batch, int64_t num_pages,
                                   int64_t max_pages_per_seq, int64_t max_kv, gqa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (batch < 1 || batch > 65535) return fail(GQA_ERR_UNSUPPORTED, "batch %lld outside [1, 65535]", (long long)batch);
  if (num_pages < 1 || max_pages_per_seq < 1 || max_kv < 1 || max_kv > 64 * max_pages_per_seq)
    return fail(GQA_ERR_INVALID_ARG, "bad num_pages / max_pages_per_seq / max_kv");
  Where where;
  gqa_status st = locate({{fp4, "fp4", 16}, {sf, "sf", 16}, {block_table, "block_table", 4},
                          {kv_lens, "kv_lens", 4}, {out_e4m3, "out_e4m3", 16}},
                         &where);
  if (st != GQA_OK) return st;
  if (where.host) return fail(GQA_ERR_UNSUPPORTED, "gqa_debug_dequant_pages takes device pointers only");
  ScopedDevice sd(where.device);
  if (!sd.ok()) return fail(GQA_ERR_CUDA, "cannot switch to device %d", where.device);
  GQA_CUDA_TRY(gqa::launch_dequant_pages(static_cast<const uint8_t*>(fp4), static_cast<const uint8_t*>(sf),
                                         block_table, kv_lens, static_cast<uint8_t*>(out_e4m3), batch, num_pages,
                                         max_pages_per_seq, max_kv, stream),
               "dequant launch");
  return GQA_OK;
}

gqa_status gqa_debug_wait_expiry(int device, gqa_stream_t stream) {
  ScopedDevice sd(device);
  if (!sd.ok()) return fail(GQA_ERR_CUDA, "cannot switch to device %d", device);
  GQA_CUDA_TRY(gqa::launch_wait_expiry(reinterpret_cast<cudaStream_t>(stream)), "wait-expiry launch");
  return GQA_OK;
}

gqa_status gqa_set_schedule(int ctx_packed_stages, int ctx_kv_slots, int decode_stages) {
  if (!gqa::ctx_schedule_supported(ctx_packed_stages, ctx_kv_slots))
    return fail(GQA_ERR_UNSUPPORTED,
                "context ring depths (%d packed stages, %d K/V slots) are not instantiated; see gqa.h", ctx_packed_stages,
                ctx_kv_slots);
  if (!gqa::decode_schedule_supported(decode_stages))
    return fail(GQA_ERR_UNSUPPORTED, "decode ring depth %d is not instantiated (0, 4, 8, 12 or 16)", decode_stages);
  g_ctx_stages.store(ctx_packed_stages, std::memory_order_relaxed);
  g_ctx_slots.store(ctx_kv_slots, std::memory_order_relaxed);
  g_decode_stages.store(decode_stages, std::memory_order_relaxed);
  return GQA_OK;
}

gqa_status gqa_set_ctx_grid(int mode) {
  if (mode < GQA_CTX_GRID_PLANNED || mode > GQA_CTX_GRID_DECODE_SHAPED)
    return fail(GQA_ERR_INVALID_ARG, "context grid mode %d is not 0, 1, 2 or 3", mode);
  g_ctx_grid.store(mode, std::memory_order_relaxed);
  return GQA_OK;
}

gqa_status gqa_debug_starve_producers(int enable) {
  g_starve.store(enable ? 1 : 0, std::memory_order_relaxed);
  return GQA_OK;
}

gqa_status gqa_check_device_errors(int device, uint32_t* word) {
  if (!word) return fail(GQA_ERR_INVALID_ARG, "word is a null pointer");
  *word = 0;
  ScopedDevice sd(device);
  if (!sd.ok()) return fail(GQA_ERR_CUDA, "cannot switch to device %d", device);
  uint32_t a = 0, b = 0, c = 0;
  GQA_CUDA_TRY(gqa::decode_read_errors(&a), "read decode error word");
  GQA_CUDA_TRY(gqa::ctx_read_errors(&b), "read ctx error word");
  GQA_CUDA_TRY(gqa::ctx_study_read_errors(&c), "read ctx study error word");
  *word = a | b | c;
  if (*word & 1u) return fail(GQA_ERR_TIMEOUT, "a kernel's bounded wait expired (error word 0x%x)", *word);
  if (*word)
    return fail(GQA_ERR_INVALID_ARG,
                "a kernel met invalid metadata: bit 1 = out-of-range page index skipped, bit 2 = qo_indptr not "
                "non-decreasing from 0 to total_q, bit 3 = dequantisation self-check (error word 0x%x)",
                *word);
  return GQA_OK;
}

// ---- descriptor forms of the three operations --------------------------------

gqa_status gqa_decode_t(const gqa_tensor* q, const gqa_tensor* kv, const gqa_tensor* seq_lens, gqa_tensor* out,
                        float q_scale, gqa_stream_t stream) {
  int64_t qs[3], ks[5];
  GQA_TRY(check_desc(q, "q", {GQA_F16}, {-1, 32, 128}, qs));
  GQA_TRY(check_desc(kv, "kv", {GQA_F16}, {qs[0], 2, 8, -1, 128}, ks));
  GQA_TRY(check_desc(seq_lens, "seq_lens", {GQA_I32}, {qs[0]}));
  GQA_TRY(check_desc(out, "out", {GQA_F16}, {qs[0], 32, 128}));
  GQA_TRY(check_devices({{q, "q"}, {kv, "kv"}, {seq_lens, "seq_lens"}, {out, "out"}}));
  return decode_impl(q->data, kv->data, static_cast<const int32_t*>(seq_lens->data), out->data, qs[0], ks[3], q_scale,
                     stream, q->device);
}

gqa_status gqa_decode_paged_t(const gqa_tensor* q, const gqa_tensor* k_pages, const gqa_tensor* v_pages,
                              const gqa_tensor* block_table, const gqa_tensor* seq_lens, gqa_tensor* out,
                              float q_scale, gqa_stream_t stream) {
  int64_t qs[3], ps[4], bs[2];
  GQA_TRY(check_desc(q, "q", {GQA_F16}, {-1, 32, 128}, qs));
  GQA_TRY(check_desc(k_pages, "k_pages", {GQA_F16}, {-1, 8, 64, 128}, ps));
  GQA_TRY(check_desc(v_pages, "v_pages", {GQA_F16}, {ps[0], 8, 64, 128}));
  GQA_TRY(check_desc(block_table, "block_table", {GQA_I32}, {qs[0], -1}, bs));
  GQA_TRY(check_desc(seq_lens, "seq_lens", {GQA_I32}, {qs[0]}));
  GQA_TRY(check_desc(out, "out", {GQA_F16}, {qs[0], 32, 128}));
  GQA_TRY(check_devices({{q, "q"}, {k_pages, "k_pages"}, {v_pages, "v_pages"}, {block_table, "block_table"},
                         {seq_lens, "seq_lens"}, {out, "out"}}));
  return decode_paged_impl(q->data, k_pages->data, v_pages->data, static_cast<const int32_t*>(block_table->data),
                           static_cast<const int32_t*>(seq_lens->data), out->data, qs[0], ps[0], bs[1], q_scale, stream,
                           q->device);
}

gqa_status nvfp4_paged_ctx_attn_t(const gqa_tensor* q_fp8, float q_scale, const gqa_tensor* k_fp4,
                                  const gqa_tensor* k_sf, const gqa_tensor* v_fp4, const gqa_tensor* v_sf,
                                  const gqa_tensor* block_table, const gqa_tensor* qo_indptr,
                                  const gqa_tensor* kv_lens, gqa_tensor* out_fp8, float out_scale,
                                  gqa_stream_t stream) {
  int64_t qs[3], ps[4], ls[1], bs[2];
  GQA_TRY(check_desc(q_fp8, "q_fp8", {GQA_E4M3, GQA_U8}, {-1, 32, 128}, qs));
  GQA_TRY(check_desc(k_fp4, "k_fp4", {GQA_U8}, {-1, 8, 64, 64}, ps));
  GQA_TRY(check_desc(k_sf, "k_sf", {GQA_E4M3, GQA_U8}, {ps[0], 8, 64, 8}));
  GQA_TRY(check_desc(v_fp4, "v_fp4", {GQA_U8}, {ps[0], 8, 64, 64}));
  GQA_TRY(check_desc(v_sf, "v_sf", {GQA_E4M3, GQA_U8}, {ps[0], 8, 64, 8}));
  GQA_TRY(check_desc(kv_lens, "kv_lens", {GQA_I32}, {-1}, ls));
  GQA_TRY(check_desc(qo_indptr, "qo_indptr", {GQA_I32}, {ls[0] + 1}));
  GQA_TRY(check_desc(block_table, "block_table", {GQA_I32}, {ls[0], -1}, bs));
  GQA_TRY(check_desc(out_fp8, "out_fp8", {GQA_E4M3, GQA_U8}, {qs[0], 32, 128}));
  GQA_TRY(check_devices({{q_fp8, "q_fp8"}, {k_fp4, "k_fp4"}, {k_sf, "k_sf"}, {v_fp4, "v_fp4"}, {v_sf, "v_sf"},
                         {block_table, "block_table"}, {qo_indptr, "qo_indptr"}, {kv_lens, "kv_lens"},
                         {out_fp8, "out_fp8"}}));
  return ctx_impl(q_fp8->data, q_scale, k_fp4->data, k_sf->data, v_fp4->data, v_sf->data,
                  static_cast<const int32_t*>(block_table->data), static_cast<const int32_t*>(qo_indptr->data),
                  static_cast<const int32_t*>(kv_lens->data), out_fp8->data, out_scale, ls[0], qs[0], ps[0], bs[1],
                  stream, q_fp8->device);
}

gqa_status gqa_release_workspace(void) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  int prev = -1;
  cudaGetDevice(&prev);
  for (auto& kv : g_ws) {
    if (kv.second.ptr) {
      cudaSetDevice(kv.first.first);
      cudaFree(kv.second.ptr);
    }
  }
  g_ws.clear();
  if (prev >= 0) cudaSetDevice(prev);
  return GQA_OK;
}

}  // extern "C"
