// C ABI of the paged decode-attention library: argument checks, split-KV
// planning, TMA descriptor encoding and kernel launches on the caller's stream.
// No call allocates device memory or synchronises (pa_get_device_error aside).
#include <cudaTypedefs.h>
#include <stdint.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "paged_attn.h"
#include "pa_internal.h"

using namespace pa;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// The pool [num_blocks, Hkv, 16, D] viewed as a 2-D tensor of rows of D bf16;
// a 16 x 64 box lands in shared memory with the 128-byte swizzle.
bool encode_pool_map(CUtensorMap* map, const void* base, long long rows, int head_dim) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlockSize)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP8 pools.  K [num_blocks, Hkv, 16, D] bytes viewed as rows of D codes; one
// 16 x D box per page (128-byte swizzle at D = 128, none at D = 64).  V
// [num_blocks, Hkv, D, 16] bytes viewed as rows of 128 bytes; one box of D/8
// rows per page, unswizzled.
bool encode_fp8_maps(CUtensorMap* tk, CUtensorMap* tv, const void* k_base, const void* v_base,
                     long long pages, int head_dim) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[2] = {1, 1};
  cuuint64_t kdims[2] = {static_cast<cuuint64_t>(head_dim),
                         static_cast<cuuint64_t>(pages * kBlockSize)};
  cuuint64_t kstr[1] = {static_cast<cuuint64_t>(head_dim)};
  cuuint32_t kbox[2] = {static_cast<cuuint32_t>(head_dim), static_cast<cuuint32_t>(kBlockSize)};
  if (fn(tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(k_base), kdims, kstr, kbox, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE,
         head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  // V page bytes as rows of 128: one box of head_dim/8 rows (few long rows keep the
  // TMA unit's per-row cost low; shared memory sees the same contiguous bytes).
  cuuint64_t vdims[2] = {128, static_cast<cuuint64_t>(pages * head_dim / 8)};
  cuuint64_t vstr[1] = {128};
  cuuint32_t vbox[2] = {128, static_cast<cuuint32_t>(head_dim / 8)};
  return fn(tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(v_base), vdims, vstr, vbox,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The kernel of this host thread's last per-sequence attention launch
// (pa_last_attention_kernel).
thread_local int g_last_kernel = PA_KERNEL_NONE;

// Kernel for multi-query tiles of 17-32 query rows per kv head (speculative
// verify) at head_dim 128 with bf16 pages: the mma.sync kernel, or the tcgen05
// kernel when the environment variable PA_VERIFY_KERNEL is "tcgen05" (read on
// every call, so that a process can compare the two).
bool tensor_core_kernel_enabled() {
  const char* v = std::getenv("PA_VERIFY_KERNEL");
  return v != nullptr && std::strcmp(v, "tcgen05") == 0;
}

// Kernel for at most 8 query rows per kv head: the environment variable
// PA_DECODE_KERNEL = "per_unit" selects the one-CTA-per-unit kernel,
// "persistent" the persistent kernel; unset (or anything else), the library
// chooses (read on every call, so that a process can compare them).
enum StreamMode { kStreamNever = 0, kStreamAuto = 1, kStreamAlways = 2 };
StreamMode stream_kernel_mode() {
  const char* v = std::getenv("PA_DECODE_KERNEL");
  if (v != nullptr && std::strcmp(v, "per_unit") == 0) return kStreamNever;
  if (v != nullptr && std::strcmp(v, "persistent") == 0) return kStreamAlways;
  return kStreamAuto;
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Plan {
  int ppb = 1;           // pages per partition
  int max_parts = 1;     // partition slots per query row
  size_t ws_bytes = 0;   // scratch needed
  size_t off_ml = 0;
  size_t off_counter = 0;  // work-unit counter of the tcgen05 kernel
};

// Partition sizes measured best on GB300: contexts up to 1024 tokens stay
// whole.  Few (sequence, kv head) pairs (< 256, small batches): partitions that
// give about 512 CTAs (1024 above 4096 tokens), at least 128 tokens each, so
// that a small batch still spreads over the whole GPU.  Otherwise: up to 4096
// tokens, 1536-token partitions; longer contexts, 2048-token partitions, or
// 3072 when there are many pairs (>= 1024) so that fewer partials need merging.
// FP8 pages (per-sequence calls) past 4096 tokens: 4096-token partitions (a
// unit then carries as many bytes as a 2048-token bf16 one; speculative verify
// measured 4 % faster than with 2048, the 70B-shape batch the same as with 3072).
int default_partition_tokens(int max_context_len, int num_seqs, int num_kv_heads,
                             bool fp8_pages = false) {
  if (max_context_len <= 1024) return ceil_div(max_context_len, kBlockSize) * kBlockSize;
  const long long pairs = static_cast<long long>(num_seqs) * num_kv_heads;
  if (pairs > 0 && pairs < 256) {
    const long long target = max_context_len > 4096 ? 1024 : 512;
    const long long parts = (target + pairs - 1) / pairs;
    const int ps = ceil_div(ceil_div(max_context_len, parts), kBlockSize) * kBlockSize;
    return std::max(ps, 128);
  }
  if (max_context_len <= 4096) return 1536;
  if (fp8_pages) return 4096;
  if (pairs >= 1024) return 3072;
  return 2048;
}

// Scratch layout: [O partials][(m, l) pairs][work-unit counter], each region
// 256-byte aligned.
Plan make_plan(int num_seqs, int hq, int T, int max_ctx, int head_dim, int partition_size,
               int max_prefix_blocks) {
  Plan pl;
  const int max_blocks = ceil_div(max_ctx, kBlockSize);
  pl.ppb = partition_size / kBlockSize;
  if (pl.ppb < 1) pl.ppb = 1;
  pl.max_parts = ceil_div(max_prefix_blocks, pl.ppb) + ceil_div(max_blocks, pl.ppb);
  if (pl.max_parts < 1) pl.max_parts = 1;
  if (pl.max_parts == 1 && max_prefix_blocks == 0) return pl;   // no scratch
  const size_t rows = static_cast<size_t>(num_seqs) * T * hq;
  const size_t po = round256(rows * pl.max_parts * head_dim * sizeof(float));
  const size_t pm = round256(rows * pl.max_parts * 2 * sizeof(float));
  pl.off_ml = po;
  pl.off_counter = po + pm;
  pl.ws_bytes = po + pm + 256;
  return pl;
}

struct AttnArgs {
  void* out;
  const void* q;
  const void* new_k;       // query tokens' K/V to append (nullptr: already in the pool)
  const void* new_v;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  int max_context_len;
  int num_seqs, T, num_blocks, hq, hkv, head_dim, block_size;
  float scale;
  int partition_size;
  const int32_t* seq_group;
  const int32_t* group_prefix_blocks;
  int num_groups, max_group_size, max_prefix_blocks;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  bool kv8 = false;                 // FP8 (E4M3) pages with per-kv-head scales
  const float* k_scale = nullptr;
  const float* v_scale = nullptr;
  int window = 0;                   // sliding window (positions per query), 0 = none
};

pa_status run_attention(const AttnArgs& a) {
  if (a.num_seqs < 0 || a.T < 1 || a.hq < 1 || a.hkv < 1 || a.num_blocks < 1 ||
      a.max_blocks_per_seq < 1 || a.partition_size < 0)
    return PA_ERR_INVALID_ARG;
  if (a.num_seqs == 0) return PA_OK;
  if (!a.out || !a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.context_lens)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(a.out) || !aligned16(a.q) || !aligned16(a.k_cache) || !aligned16(a.v_cache))
    return PA_ERR_INVALID_ARG;
  if (a.hq % a.hkv != 0) return PA_ERR_INVALID_ARG;
  if (a.head_dim != 64 && a.head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (a.block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  const int G = a.hq / a.hkv;
  if (static_cast<long long>(G) * a.T > kMaxRows) return PA_ERR_UNSUPPORTED;
  if (a.max_context_len < a.T ||
      static_cast<long long>(a.max_context_len) >
          static_cast<long long>(a.max_blocks_per_seq) * kBlockSize)
    return PA_ERR_INVALID_ARG;
  if (a.partition_size % kBlockSize != 0) return PA_ERR_INVALID_ARG;
  if (a.num_seqs > 65535) return PA_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(a.num_blocks) * a.hkv * kBlockSize;
  if (rows >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
  const bool grouped = a.num_groups > 0;
  if (a.kv8 && (!a.k_scale || !a.v_scale)) return PA_ERR_INVALID_ARG;
  if (a.window < 0) return PA_ERR_INVALID_ARG;
  if (a.window > 0 && grouped) return PA_ERR_UNSUPPORTED;
  if (grouped) {
    if (!a.seq_group || !a.group_prefix_blocks || a.max_group_size < 1 ||
        a.max_prefix_blocks < 0 ||
        static_cast<long long>(a.max_prefix_blocks) * kBlockSize > a.max_context_len)
      return PA_ERR_INVALID_ARG;
    if (static_cast<long long>(G) * a.T > kMaxRows) return PA_ERR_UNSUPPORTED;
  }
  const int max_prefix = grouped ? a.max_prefix_blocks : 0;

  int psize = a.partition_size;
  if (psize == 0) {
    psize = default_partition_tokens(a.max_context_len, a.num_seqs, a.hkv, a.kv8 && !grouped);
    Plan probe = make_plan(a.num_seqs, a.hq, a.T, a.max_context_len, a.head_dim, psize,
                           max_prefix);
    if (!grouped && probe.ws_bytes > 0 && a.workspace == nullptr)
      psize = ceil_div(a.max_context_len, kBlockSize) * kBlockSize;   // whole sequences
  }
  const Plan plan = make_plan(a.num_seqs, a.hq, a.T, a.max_context_len, a.head_dim, psize,
                              max_prefix);
  if (plan.max_parts > kMaxPartitions) return PA_ERR_UNSUPPORTED;   // use larger partitions
  if (plan.ws_bytes > 0) {
    if (!a.workspace || a.workspace_bytes < plan.ws_bytes) return PA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(a.workspace) & 255u) return PA_ERR_INVALID_ARG;
  }

  CUtensorMap tk, tv;
  if (a.kv8) {
    if (!encode_fp8_maps(&tk, &tv, a.k_cache, a.v_cache,
                         static_cast<long long>(a.num_blocks) * a.hkv, a.head_dim))
      return PA_ERR_CUDA;
  } else if (!encode_pool_map(&tk, a.k_cache, rows, a.head_dim) ||
             !encode_pool_map(&tv, a.v_cache, rows, a.head_dim)) {
    return PA_ERR_CUDA;
  }

  AttnParams p{};
  p.q = a.q;
  p.out = a.out;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  if (plan.ws_bytes > 0) {
    char* ws = static_cast<char*>(a.workspace);
    p.part_o = reinterpret_cast<float*>(ws);
    p.part_ml = reinterpret_cast<float2*>(ws + plan.off_ml);
  }
  if (a.new_k != nullptr) {
    if (!a.new_v || !aligned16(a.new_k) || !aligned16(a.new_v)) return PA_ERR_INVALID_ARG;
    p.new_k = a.new_k;
    p.new_v = a.new_v;
    p.k_pool = const_cast<void*>(a.k_cache);
    p.v_pool = const_cast<void*>(a.v_cache);
  }
  p.seq_group = grouped ? a.seq_group : nullptr;
  p.k_scale = a.kv8 ? a.k_scale : nullptr;
  p.v_scale = a.kv8 ? a.v_scale : nullptr;
  p.group_prefix_blocks = grouped ? a.group_prefix_blocks : nullptr;
  p.mbs = a.max_blocks_per_seq;
  p.max_ctx = a.max_context_len;
  p.num_seqs = a.num_seqs;
  p.T = a.T;
  p.Hq = a.hq;
  p.Hkv = a.hkv;
  p.G = G;
  p.num_blocks = a.num_blocks;
  p.ppb = plan.ppb;
  p.max_parts = plan.max_parts;
  p.max_prefix_blocks = max_prefix;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.window = a.window;
  p.wcap = a.window > 0 ? static_cast<unsigned>(a.window) : 0x80000000u;
  p.wspan = a.window > 0 ? a.window : (1 << 30);
  p.timeout_ns = kDefaultTimeoutNs;

  const int max_blocks = ceil_div(a.max_context_len, kBlockSize);
  cudaError_t e = cudaSuccess;
  const bool group_launch = grouped && a.max_prefix_blocks > 0;
  if (group_launch) {
    const int mc = std::min(a.max_group_size, kMaxRows / (G * a.T));
    p.members_per_chunk = mc;
    p.num_chunks = ceil_div(a.max_group_size, mc);
    const long long gz = static_cast<long long>(a.num_groups) * p.num_chunks;
    if (gz > 65535) return PA_ERR_UNSUPPORTED;
    const int rows = mc * G * a.T;
    dim3 grid(ceil_div(a.max_prefix_blocks, plan.ppb), a.hkv, static_cast<unsigned>(gz));
    if (a.kv8)
      e = a.head_dim == 64 ? launch_attn_group8_d64(tk, tv, p, rows, grid, a.stream)
                           : launch_attn_group8_d128(tk, tv, p, rows, grid, a.stream);
    else
      e = a.head_dim == 64 ? launch_attn_group_d64(tk, tv, p, rows, grid, a.stream)
                           : launch_attn_group_d128(tk, tv, p, rows, grid, a.stream);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  {
    const int rows = G * a.T;
    // blocks one sequence may read: all of them, or those under its queries' windows
    int span = max_blocks;
    if (a.window > 0)
      span = static_cast<int>(std::min<long long>(
          max_blocks, (static_cast<long long>(a.window) + a.T - 1 + kBlockSize - 1) / kBlockSize + 1));
    // 1-D, partition-major: unit u = (partition * num_seqs + seq) * hkv + head
    const long long units = static_cast<long long>(ceil_div(span, plan.ppb)) * a.hkv *
                            a.num_seqs;
    if (units >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    dim3 grid(static_cast<unsigned>(units), 1, 1);
    const StreamMode mode = stream_kernel_mode();
    // the tcgen05 kernel, when asked for, takes precedence for its tiles
    const bool tc = !a.kv8 && a.head_dim == 128 && rows > 16 && rows <= 32 &&
                    tensor_core_kernel_enabled();
    bool launched = false;
    if (!grouped && !tc && (rows <= 8 || (rows >= 17 && rows <= 24)) &&
        a.num_seqs <= kStreamMaxSeqs && plan.ppb <= kStreamMaxPpb && mode != kStreamNever) {
      // Claim state 16 bytes into the counter area (the tcgen05 kernel's
      // counter is the first 4 bytes).
      if (plan.ws_bytes > 0)
        p.stream_ctl = static_cast<char*>(a.workspace) + plan.off_counter + 16;
      const bool always = mode == kStreamAlways;
      e = a.head_dim == 64
              ? launch_stream_d64(tk, tv, p, rows, units, a.kv8, always, a.stream, &launched)
              : launch_stream_d128(tk, tv, p, rows, units, a.kv8, always, a.stream, &launched);
      if (e != cudaSuccess) return PA_ERR_CUDA;
      if (!launched) p.stream_ctl = nullptr;
      else g_last_kernel = PA_KERNEL_PERSISTENT;
    }
    if (!launched) {
      if (a.kv8) {
        e = a.head_dim == 64 ? launch_attn8_d64(tk, tv, p, rows, grid, a.stream, group_launch)
                             : launch_attn8_d128(tk, tv, p, rows, grid, a.stream, group_launch);
      } else if (tc) {
        // With scratch, the persistent CTAs claim units from a counter zeroed here.
        if (plan.ws_bytes > 0) {
          p.unit_counter =
              reinterpret_cast<int*>(static_cast<char*>(a.workspace) + plan.off_counter);
          e = cudaMemsetAsync(p.unit_counter, 0, sizeof(int), a.stream);
          if (e != cudaSuccess) return PA_ERR_CUDA;
        }
        e = launch_attn_tc_d128(tk, tv, p, rows, grid, a.stream, group_launch);
        g_last_kernel = PA_KERNEL_TCGEN05;
      } else {
        e = a.head_dim == 64 ? launch_attn_d64(tk, tv, p, rows, grid, a.stream, group_launch)
                             : launch_attn_d128(tk, tv, p, rows, grid, a.stream, group_launch);
      }
      if (e != cudaSuccess) return PA_ERR_CUDA;
      if (!tc) g_last_kernel = PA_KERNEL_PER_UNIT;
    }
  }
  if (plan.ws_bytes > 0) {
    e = launch_reduce(p, a.head_dim, a.stream);
    if (e != cudaSuccess) {
      // The merge resets the persistent kernel's claim counter; without it the
      // tag must go, so that the next launch on this scratch does not claim
      // from a stale counter.
      if (p.stream_ctl != nullptr) cudaMemsetAsync(p.stream_ctl, 0, sizeof(StreamCtl), a.stream);
      return PA_ERR_CUDA;
    }
  }
  return PA_OK;
}

}  // namespace

namespace pa {

int default_partition_for(int max_context_len, int num_seqs, int num_kv_heads, bool fp8_pages) {
  if (max_context_len < 1) return kBlockSize;
  return default_partition_tokens(max_context_len, num_seqs, num_kv_heads, fp8_pages);
}

size_t workspace_for(int num_seqs, int num_q_heads, int num_kv_heads, int num_query_tokens,
                     int max_context_len, int head_dim, int partition_size,
                     int max_prefix_blocks) {
  const int psize = partition_size > 0
                        ? partition_size
                        : default_partition_tokens(max_context_len, num_seqs, num_kv_heads);
  return make_plan(num_seqs, num_q_heads, num_query_tokens, max_context_len, head_dim, psize,
                   max_prefix_blocks)
      .ws_bytes;
}

}  // namespace pa

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_BOUNDS: return "PA_ERR_BOUNDS";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
    case PA_ERR_OUT_OF_BLOCKS: return "PA_ERR_OUT_OF_BLOCKS";
    default: return "PA_ERR_UNKNOWN";
  }
}

int pa_version(void) { return 102; }

int pa_last_attention_kernel(void) { return g_last_kernel; }

pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache,
                               void* v_cache, const int64_t* slot_mapping, int num_tokens,
                               int num_blocks, int num_kv_heads, int head_dim, int block_size,
                               pa_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 8 ||
      head_dim % 8 != 0)
    return PA_ERR_INVALID_ARG;
  if (block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const cudaError_t e =
      launch_reshape(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_blocks,
                     num_kv_heads, head_dim, block_size, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, void* k_cache,
                                   void* v_cache, const int64_t* slot_mapping,
                                   const float* k_scale, const float* v_scale, int num_tokens,
                                   int num_blocks, int num_kv_heads, int head_dim, int block_size,
                                   pa_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 8 ||
      head_dim % 8 != 0)
    return PA_ERR_INVALID_ARG;
  if (block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping || !k_scale || !v_scale)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const cudaError_t e = launch_reshape_fp8(key, value, k_cache, v_cache, slot_mapping, k_scale,
                                           v_scale, num_tokens, num_blocks, num_kv_heads,
                                           head_dim, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs,
                         int num_pairs, int num_blocks, int num_kv_heads, int head_dim,
                         int block_size, pa_stream_t stream) {
  if (num_pairs < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 8 || head_dim % 8 != 0)
    return PA_ERR_INVALID_ARG;
  if (block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  if (num_pairs > 65535) return PA_ERR_UNSUPPORTED;
  if (!k_cache || !v_cache || !block_pairs || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  return launch_copy_blocks(k_cache, v_cache, block_pairs, num_pairs, num_blocks, num_kv_heads,
                            head_dim, block_size, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

int pa_default_partition_size(int num_seqs, int num_kv_heads, int max_context_len,
                              int block_size) {
  (void)block_size;
  if (max_context_len < 1) return kBlockSize;
  return default_partition_tokens(max_context_len, num_seqs, num_kv_heads);
}

size_t pa_workspace_size(int num_seqs, int num_q_heads, int num_query_tokens,
                         int max_context_len, int head_dim, int block_size, int partition_size,
                         int max_prefix_blocks) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_query_tokens <= 0 || max_context_len <= 0 ||
      head_dim <= 0 || block_size != kBlockSize || partition_size < 0 || max_prefix_blocks < 0)
    return 0;
  if (partition_size > 0)
    return pa::workspace_for(num_seqs, num_q_heads, 1, num_query_tokens, max_context_len,
                             head_dim, partition_size, max_prefix_blocks);
  // num_kv_heads is not known here: the largest need over every kv-head count
  size_t most = 0;
  for (int h = 1; h <= num_q_heads; ++h)
    if (num_q_heads % h == 0)
      most = std::max(most, pa::workspace_for(num_seqs, num_q_heads, h, num_query_tokens,
                                              max_context_len, head_dim, 0, max_prefix_blocks));
  return most;
}

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int max_context_len, int num_seqs,
                    int num_blocks, int num_q_heads, int num_kv_heads, int head_dim,
                    int block_size, float scale, int partition_size, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream) {
  AttnArgs a{out, q, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq,
             context_lens, max_context_len, num_seqs, 1, num_blocks, num_q_heads, num_kv_heads,
             head_dim, block_size, scale, partition_size, nullptr, nullptr, 0, 0, 0, workspace,
             workspace_bytes, reinterpret_cast<cudaStream_t>(stream)};
  return run_attention(a);
}

pa_status pa_verify(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int max_context_len, int num_seqs,
                    int num_query_tokens, int num_blocks, int num_q_heads, int num_kv_heads,
                    int head_dim, int block_size, float scale, int partition_size,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  AttnArgs a{out, q, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq,
             context_lens, max_context_len, num_seqs, num_query_tokens, num_blocks,
             num_q_heads, num_kv_heads, head_dim, block_size, scale, partition_size, nullptr,
             nullptr, 0, 0, 0, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream)};
  return run_attention(a);
}

pa_status pa_verify_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens,
                        int max_context_len, int num_seqs, int num_query_tokens, int num_blocks,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        float scale, int partition_size, void* workspace,
                        size_t workspace_bytes, pa_stream_t stream) {
  AttnArgs a{out, q, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq,
             context_lens, max_context_len, num_seqs, num_query_tokens, num_blocks,
             num_q_heads, num_kv_heads, head_dim, block_size, scale, partition_size, nullptr,
             nullptr, 0, 0, 0, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), true, k_scale, v_scale};
  return run_attention(a);
}

pa_status pa_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens,
                        int max_context_len, int num_seqs, int num_blocks, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, float scale,
                        int partition_size, void* workspace, size_t workspace_bytes,
                        pa_stream_t stream) {
  return pa_verify_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                       max_blocks_per_seq, context_lens, max_context_len, num_seqs, 1,
                       num_blocks, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                       partition_size, workspace, workspace_bytes, stream);
}

pa_status pa_attention(void* out, const void* q, const void* new_key, const void* new_value,
                       void* k_cache, void* v_cache, const float* k_scale, const float* v_scale,
                       int kv_dtype, int window_size, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                       int num_seqs, int num_query_tokens, int num_blocks, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, float scale,
                       int partition_size, void* workspace, size_t workspace_bytes,
                       pa_stream_t stream) {
  if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
  if ((new_key == nullptr) != (new_value == nullptr)) return PA_ERR_INVALID_ARG;
  AttnArgs a{out, q, new_key, new_value, k_cache, v_cache, block_tables, max_blocks_per_seq,
             context_lens, max_context_len, num_seqs, num_query_tokens, num_blocks,
             num_q_heads, num_kv_heads, head_dim, block_size, scale, partition_size, nullptr,
             nullptr, 0, 0, 0, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), kv_dtype == PA_KV_FP8_E4M3, k_scale,
             v_scale, window_size};
  return run_attention(a);
}

pa_status pa_decode_append_fp8(void* out, const void* q, const void* new_key,
                               const void* new_value, void* k_cache, void* v_cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int max_context_len, int num_seqs,
                               int num_query_tokens, int num_blocks, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, float scale,
                               int partition_size, void* workspace, size_t workspace_bytes,
                               pa_stream_t stream) {
  if (num_seqs > 0 && (!new_key || !new_value)) return PA_ERR_INVALID_ARG;
  AttnArgs a{out, q, new_key, new_value, k_cache, v_cache, block_tables, max_blocks_per_seq,
             context_lens, max_context_len, num_seqs, num_query_tokens, num_blocks,
             num_q_heads, num_kv_heads, head_dim, block_size, scale, partition_size, nullptr,
             nullptr, 0, 0, 0, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), true, k_scale, v_scale};
  return run_attention(a);
}

pa_status pa_decode_append(void* out, const void* q, const void* new_key, const void* new_value,
                           void* k_cache, void* v_cache, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* context_lens,
                           int max_context_len, int num_seqs, int num_query_tokens,
                           int num_blocks, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, float scale, int partition_size, void* workspace,
                           size_t workspace_bytes, pa_stream_t stream) {
  if (num_seqs > 0 && (!new_key || !new_value)) return PA_ERR_INVALID_ARG;
  AttnArgs a{out, q, new_key, new_value, k_cache, v_cache, block_tables, max_blocks_per_seq,
             context_lens, max_context_len, num_seqs, num_query_tokens, num_blocks,
             num_q_heads, num_kv_heads, head_dim, block_size, scale, partition_size, nullptr,
             nullptr, 0, 0, 0, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream)};
  return run_attention(a);
}

pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_tables,
                                  int max_blocks_per_seq, const int32_t* context_lens,
                                  int max_context_len, int num_seqs, int num_blocks,
                                  int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, float scale, int partition_size,
                                  const int32_t* seq_group, const int32_t* group_prefix_blocks,
                                  int num_groups, int max_group_size, int max_prefix_blocks,
                                  void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  if (num_groups < 0) return PA_ERR_INVALID_ARG;
  AttnArgs a{out, q, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq,
             context_lens, max_context_len, num_seqs, 1, num_blocks, num_q_heads, num_kv_heads,
             head_dim, block_size, scale, partition_size, seq_group, group_prefix_blocks,
             num_groups, max_group_size, max_prefix_blocks, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream)};
  return run_attention(a);
}

pa_status pa_spec_accept(const float* target_probs, const float* draft_probs,
                         const int32_t* draft_tokens, const uint32_t* accept_uniforms,
                         const uint32_t* sample_uniforms, int num_seqs, int num_drafts,
                         int vocab_size, int greedy, int32_t* out_tokens, int32_t* num_accepted,
                         pa_stream_t stream) {
  if (num_seqs < 0 || num_drafts < 0 || vocab_size < 1) return PA_ERR_INVALID_ARG;
  if (vocab_size > kMaxSpecVocab || num_drafts > 64 || num_seqs > (1 << 30))
    return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!target_probs || !out_tokens || !num_accepted || (num_drafts > 0 && !draft_tokens))
    return PA_ERR_INVALID_ARG;
  if (!greedy && (!sample_uniforms || (num_drafts > 0 && (!draft_probs || !accept_uniforms))))
    return PA_ERR_INVALID_ARG;
  return launch_spec_accept(target_probs, draft_probs, draft_tokens, accept_uniforms,
                            sample_uniforms, num_seqs, num_drafts, vocab_size, greedy != 0,
                            out_tokens, num_accepted,
                            reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_decode_shared_prefix_fp8(
    void* out, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
    const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len, int num_seqs, int num_blocks,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
    int partition_size, const int32_t* seq_group, const int32_t* group_prefix_blocks,
    int num_groups, int max_group_size, int max_prefix_blocks, void* workspace,
    size_t workspace_bytes, pa_stream_t stream) {
  if (num_groups < 0) return PA_ERR_INVALID_ARG;
  AttnArgs a{out, q, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq,
             context_lens, max_context_len, num_seqs, 1, num_blocks, num_q_heads, num_kv_heads,
             head_dim, block_size, scale, partition_size, seq_group, group_prefix_blocks,
             num_groups, max_group_size, max_prefix_blocks, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), true, k_scale, v_scale};
  return run_attention(a);
}

pa_status pa_get_device_error(pa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  unsigned bits = 0;
  if (take_error_attn_d64(&bits) != cudaSuccess || take_error_attn_d128(&bits) != cudaSuccess ||
      take_error_group_d64(&bits) != cudaSuccess ||
      take_error_group_d128(&bits) != cudaSuccess || take_error_attn8_d64(&bits) != cudaSuccess ||
      take_error_attn8_d128(&bits) != cudaSuccess || take_error_group8_d64(&bits) != cudaSuccess ||
      take_error_group8_d128(&bits) != cudaSuccess || take_error_spec(&bits) != cudaSuccess ||
      take_error_attn_tc_d128(&bits) != cudaSuccess || take_error_stream_d64(&bits) != cudaSuccess ||
      take_error_stream_d128(&bits) != cudaSuccess || take_error_misc(&bits) != cudaSuccess)
    return PA_ERR_CUDA;
  if (bits & kErrTimeout) return PA_ERR_TIMEOUT;
  if (bits & kErrBounds) return PA_ERR_BOUNDS;
  return PA_OK;
}

pa_status pa_selftest_wait_timeout(unsigned long long timeout_ns, pa_stream_t stream) {
  if (timeout_ns < 1000ull || timeout_ns > 1000000000ull) return PA_ERR_INVALID_ARG;
  return launch_selftest_wait(timeout_ns, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

}  // extern "C"
