// Persistent decode attention kernels (at most 8 query rows per kv head),
// head_dim 128, bf16 and FP8 pages.
#include "pa_attn_stream.cuh"

namespace pa {

cudaError_t launch_stream_d128(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                             int rows, long long max_units, bool kv8, bool always, cudaStream_t s,
                             bool* launched) {
  return kv8 ? launch_stream<128, true>(tk, tv, p, rows, max_units, true, s, launched)
             : launch_stream<128, false>(tk, tv, p, rows, max_units, always, s, launched);
}

cudaError_t take_error_stream_d128(unsigned* bits) { return take_error_word(bits); }

}  // namespace pa
