// Per-sequence paged attention kernels, head_dim 128 (decode and verify).
#include "pa_attn.cuh"

namespace pa {

cudaError_t launch_attn_d128(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                            int rows, dim3 grid, cudaStream_t s, bool overlap_previous) {
  return launch_dispatch<128, false>(tk, tv, p, rows, grid, s, overlap_previous);
}

cudaError_t take_error_attn_d128(unsigned* bits) { return take_error_word(bits); }

}  // namespace pa
