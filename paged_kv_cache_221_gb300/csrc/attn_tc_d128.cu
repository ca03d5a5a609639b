// Tensor-core (tcgen05) attention kernel: head_dim 128, bf16 pages, up to 32
// query rows per kv head.
#include "pa_attn_tc.cuh"

namespace pa {

cudaError_t launch_attn_tc_d128(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                                int rows, dim3 grid, cudaStream_t s, bool overlap_previous) {
  return launch_tc(tk, tv, p, rows, static_cast<int>(grid.x), s, overlap_previous);
}

cudaError_t take_error_attn_tc_d128(unsigned* bits) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_pa_err, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_pa_err, &zero, sizeof(zero));
  *bits |= v;
  return e;
}

}  // namespace pa
