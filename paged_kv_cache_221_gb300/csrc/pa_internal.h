// Internal host/device interface between the C ABI (pa_api.cpp) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Bits of the sticky device error word (one word per kernel translation unit).
enum : unsigned { kErrBounds = 1u, kErrTimeout = 2u };

constexpr int kBlockSize = 16;        // tokens per physical block (the only size built)
constexpr int kStages = 8;            // pages in flight per CTA (multiple of every PL)
constexpr int kMaxRows = 64;          // query rows per CTA (8 n-tiles of 8)
constexpr int kStreamMaxSeqs = 256;   // persistent decode kernel: sequences its unit list holds
constexpr int kStreamMaxPpb = 256;    // persistent decode kernel: pages per partition
constexpr int kMaxPartitions = 4096;  // split-KV partitions per sequence (merge smem bound)
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;   // 2 s per wait
constexpr int kMaxSpecVocab = 1 << 19;  // speculative acceptance: largest vocabulary

// Everything an attention launch needs besides the two tensor maps.
struct AttnParams {
  const void* q;                  // bf16 [B, T, Hq, D]
  void* out;                      // bf16 [B, T, Hq, D]
  const int32_t* block_tables;    // [B, mbs]
  const int32_t* context_lens;    // [B]
  const void* new_k;              // bf16 [B, T, Hkv, D] or nullptr: K of the query tokens,
  const void* new_v;              //   written at positions L-T .. L-1 before they are read
  void* k_pool;                   // the pools again, for those writes
  void* v_pool;
  float* part_o;                  // [B*T*Hq, max_parts, D]   (split-KV partials)
  float2* part_ml;                // [B*T*Hq, max_parts]      (reference max in the log2
                                  //   domain, softmax denominator) per partition
  const int32_t* seq_group;       // [B] or nullptr
  const int32_t* group_prefix_blocks;  // [num_groups] or nullptr
  const float* k_scale;           // FP8 pages: [Hkv] dequantisation scales of K and V
  const float* v_scale;           //   (nullptr for bf16 pages)
  int mbs;                        // max_blocks_per_seq
  int max_ctx;                    // bound on context_lens
  int num_seqs, T, Hq, Hkv, G, num_blocks;
  int ppb;                        // pages (blocks) per partition
  int max_parts;                  // partition slots per query row
  int members_per_chunk;          // shared-prefix kernel: group members per CTA
  int num_chunks;                 // shared-prefix kernel: CTAs per group (per partition, head)
  int max_prefix_blocks;          // bound on group_prefix_blocks (launch sizing)
  float scale_log2;               // softmax scale * log2(e)
  int window;                     // sliding window (positions each query sees), 0 = none
  unsigned wcap;                  // window, or 2^31 without one (visibility: lim - j < wcap)
  int wspan;                      // window, or 2^30 without one (interior pages: tok0 +
                                  //   wspan >= context length)
  unsigned long long timeout_ns;  // limit of every pipeline wait
  int* unit_counter;              // tcgen05 kernel: next work unit to claim (zeroed before the
                                  //   launch), or nullptr for a fixed round-robin order
  void* stream_ctl;               // persistent decode kernel: its StreamCtl in the scratch,
                                  //   or nullptr (no scratch: fixed order)
};

// Claim state of the persistent decode kernel, kept in the split-KV scratch:
// a tag and the next unit-list position to hand out.  When the tag is present
// at launch, `next` is zero and CTAs claim positions from it; the split-KV merge
// that follows every such launch sets `next` back to zero and writes the tag.
// Without the tag (scratch not yet used by this kernel, or overwritten since)
// the launch takes positions in a fixed order and leaves `next` untouched.
struct StreamCtl {
  unsigned long long tag;
  int next;
  int pad;
};
constexpr unsigned long long kStreamTag = 0x70615F7374726D31ull;

// The partition size (tokens) a per-sequence call with partition_size 0 uses:
// the library default for this batch, with the FP8-page rule when fp8_pages.
int default_partition_for(int max_context_len, int num_seqs, int num_kv_heads, bool fp8_pages);

// Split-KV scratch bytes a call with these sizes needs (partition_size 0 = the
// library default for this kv-head count).
size_t workspace_for(int num_seqs, int num_q_heads, int num_kv_heads, int num_query_tokens,
                     int max_context_len, int head_dim, int partition_size,
                     int max_prefix_blocks);

// Kernel launchers (one translation unit per head_dim and mode); `rows` is the
// number of query rows one CTA carries (1 .. kMaxRows).
// overlap_previous: launch with programmatic stream serialisation so the kernel may
// run alongside the shared-prefix kernel launched just before it.
cudaError_t launch_attn_d64(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                            int rows, dim3 grid, cudaStream_t s, bool overlap_previous);
cudaError_t launch_attn_d128(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                             int rows, dim3 grid, cudaStream_t s, bool overlap_previous);
cudaError_t launch_attn_group_d64(const CUtensorMap& tk, const CUtensorMap& tv,
                                  const AttnParams& p, int rows, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_group_d128(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const AttnParams& p, int rows, dim3 grid, cudaStream_t s);
// FP8 (E4M3) pages: K [NB, Hkv, 16, D] token-major, V [NB, Hkv, D, 16] per-page transposed.
cudaError_t launch_attn8_d64(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                             int rows, dim3 grid, cudaStream_t s, bool overlap_previous);
cudaError_t launch_attn8_d128(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                              int rows, dim3 grid, cudaStream_t s, bool overlap_previous);
cudaError_t launch_attn_group8_d64(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const AttnParams& p, int rows, dim3 grid, cudaStream_t s);
cudaError_t launch_attn_group8_d128(const CUtensorMap& tk, const CUtensorMap& tv,
                                    const AttnParams& p, int rows, dim3 grid, cudaStream_t s);
// Persistent decode kernel (pa_attn_stream.cuh): per-sequence mode, at most 8
// query rows per kv head, at most kStreamMaxSeqs sequences and kStreamMaxPpb
// pages per partition; `max_units` bounds the work units.  Unless `always`, it
// runs only where it measured faster than the one-CTA-per-unit kernel (FP8
// pages, or at least 4 units per resident CTA); *launched says whether it ran.
cudaError_t launch_stream_d64(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                              int rows, long long max_units, bool kv8, bool always,
                              cudaStream_t s, bool* launched);
cudaError_t launch_stream_d128(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                               int rows, long long max_units, bool kv8, bool always,
                               cudaStream_t s, bool* launched);
// tcgen05 kernel (head_dim 128, bf16 pages, 17-32 query rows per kv head).
cudaError_t launch_attn_tc_d128(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                                int rows, dim3 grid, cudaStream_t s, bool overlap_previous);
cudaError_t launch_reshape_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slots, const float* k_scale, const float* v_scale,
                               int num_tokens, int num_blocks, int hkv, int head_dim,
                               cudaStream_t s);
// Speculative acceptance (pa_spec.cu): one CTA per sequence.
cudaError_t launch_spec_accept(const float* p, const float* q, const int32_t* drafts,
                               const uint32_t* a24, const uint32_t* s32, int num_seqs, int K,
                               int V, bool greedy, int32_t* out_tokens, int32_t* out_kept,
                               cudaStream_t s);
// Graph runner padding: rows [from, to) become a one-block sequence of `len` tokens
// in block `pad_block`.
cudaError_t launch_pad_rows(int32_t* block_tables, int32_t* context_lens, int from, int to,
                            int max_blocks_per_seq, int pad_block, int len, cudaStream_t s);
// Graph runner staging: `bytes` (a multiple of 16; both addresses 16-byte aligned and
// device-addressable) copied by a kernel.
cudaError_t launch_stage_copy(void* dst, const void* src, size_t bytes, cudaStream_t s);
cudaError_t launch_reduce(const AttnParams& p, int head_dim, cudaStream_t s);
cudaError_t launch_reshape(const void* key, const void* value, void* k_cache, void* v_cache,
                           const int64_t* slots, int num_tokens, int num_blocks, int hkv,
                           int head_dim, int block_size, cudaStream_t s);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                               int num_blocks, int hkv, int head_dim, int block_size,
                               cudaStream_t s);
cudaError_t launch_selftest_wait(unsigned long long timeout_ns, cudaStream_t s);

// Read and clear the device error word of each translation unit (synchronous).
cudaError_t take_error_attn_d64(unsigned* bits);
cudaError_t take_error_attn_d128(unsigned* bits);
cudaError_t take_error_group_d64(unsigned* bits);
cudaError_t take_error_group_d128(unsigned* bits);
cudaError_t take_error_attn8_d64(unsigned* bits);
cudaError_t take_error_attn8_d128(unsigned* bits);
cudaError_t take_error_group8_d64(unsigned* bits);
cudaError_t take_error_group8_d128(unsigned* bits);
cudaError_t take_error_spec(unsigned* bits);
cudaError_t take_error_attn_tc_d128(unsigned* bits);
cudaError_t take_error_stream_d64(unsigned* bits);
cudaError_t take_error_stream_d128(unsigned* bits);
cudaError_t take_error_misc(unsigned* bits);

}  // namespace pa
