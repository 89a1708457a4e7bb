// ctx_nvfp4.cu -- NVFP4 paged context attention for sm_103a, and the test
// export of its dequantisation.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "nvfp4.cuh"

namespace gqa {
namespace {

__device__ uint32_t g_ctx_err;

// Dense gather of dequantised tokens: one thread per (token, KV head,
// 16-element block).  Uses the same dequant16 as the attention kernel.
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

cudaError_t launch_ctx(const CtxArgs& a, cudaStream_t stream) {
  (void)a;
  (void)stream;
  return cudaErrorNotSupported;
}

cudaError_t ctx_read_errors(uint32_t* word) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  uint32_t zero = 0;
  if ((e = cudaMemcpyFromSymbol(word, g_ctx_err, sizeof(uint32_t))) != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_ctx_err, &zero, sizeof(uint32_t));
}

}  // namespace gqa
