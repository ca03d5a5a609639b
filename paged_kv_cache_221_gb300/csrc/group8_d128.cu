// Shared-prefix paged attention kernels over FP8 (E4M3) pages, head_dim 128: one
// CTA reads a group's copy-on-write prefix pages once for all members of the group.
#include "pa_attn.cuh"

namespace pa {

cudaError_t launch_attn_group8_d128(const CUtensorMap& tk, const CUtensorMap& tv,
                                    const AttnParams& p, int rows, dim3 grid, cudaStream_t s) {
  return launch_dispatch<128, true, true>(tk, tv, p, rows, grid, s, false);
}

cudaError_t take_error_group8_d128(unsigned* bits) { return take_error_word(bits); }

}  // namespace pa
