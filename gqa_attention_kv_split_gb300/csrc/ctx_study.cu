// ctx_study.cu -- the unsplit NVFP4 context attention kernel at ring depths
// other than the production ones, for the ring-depth study of "GB300 NVFP4
// Context Attention: scale slot 조기 반납과 8단 packed K/V ring" (section 2, the
// 8-stage packed K/V ring, and the bit-identity check of its results
// section): every instance computes the same result bit for bit; only the
// number of packed-page stages (kNP) and of dequantised K/V slots (kNK)
// differs.  Selected through gqa_set_schedule; a translation unit of its own
// so that the instances compile in parallel with the production ones.
#include "ctx_kernel.cuh"

namespace gqa {

bool ctx_schedule_supported(int stages, int slots) {
  const int s = stages ? stages : ctx::kCtxStagesDefault, k = slots ? slots : ctx::kCtxSlotsDefault;
  switch (s * 100 + k) {
    case 604: case 404: case 804: case 1004: case 603: case 1203: case 605: case 602:
      return true;
    default:
      return false;
  }
}

cudaError_t launch_ctx_study(const CtxArgs& a, const CUtensorMap& q_map, unsigned grid, float scale_log2,
                             float inv_out_scale, int stages, int slots, cudaStream_t stream) {
  const dim3 g(grid, 1);
  switch (stages * 100 + slots) {
    case 604: return ctx::launch_attention<false, 6, 4>(a, q_map, g, scale_log2, inv_out_scale, 0, nullptr, nullptr, stream);
    case 804: return ctx::launch_attention<false, 8, 4>(a, q_map, g, scale_log2, inv_out_scale, 0, nullptr, nullptr, stream);
    case 1004: return ctx::launch_attention<false, 10, 4>(a, q_map, g, scale_log2, inv_out_scale, 0, nullptr, nullptr, stream);
    case 603: return ctx::launch_attention<false, 6, 3>(a, q_map, g, scale_log2, inv_out_scale, 0, nullptr, nullptr, stream);
    case 1203: return ctx::launch_attention<false, 12, 3>(a, q_map, g, scale_log2, inv_out_scale, 0, nullptr, nullptr, stream);
    case 605: return ctx::launch_attention<false, 6, 5>(a, q_map, g, scale_log2, inv_out_scale, 0, nullptr, nullptr, stream);
    case 602: return ctx::launch_attention<false, 6, 2>(a, q_map, g, scale_log2, inv_out_scale, 0, nullptr, nullptr, stream);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t ctx_study_read_errors(uint32_t* word) { return ctx::read_ctx_error_word(word); }

}  // namespace gqa
