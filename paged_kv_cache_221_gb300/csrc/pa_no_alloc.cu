// pa_decode_static_scratch: pa_decode for callers that cannot allocate
// device memory.
//
// Some callers of a decode kernel are not allowed to allocate: a plugin that a
// host runtime hands only its input and output buffers, or a serving process
// that reserves all device memory at start-up and forbids cudaMalloc and
// cudaFree afterwards (both can synchronise the device and fragment the
// memory that was planned for the KV cache).  Such a caller cannot provide the
// split-KV scratch that pa_decode needs for long contexts.  This entry point
// takes that scratch from a fixed array in this library's device image
// instead.  The array belongs to this file's module: under CUDA's lazy module
// loading (the default) the module, and with it the array's 32 MiB, is loaded
// onto a device by the first call made on that device, which looks up the
// array's address; with CUDA_MODULE_LOADING=EAGER it is loaded with the
// library.  Either way it stays until the process exits.
#include <mutex>

#include "paged_attn.h"
#include "pa_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 32ull << 20;   // 32 MiB

// Split-KV partials of pa_decode_static_scratch (never read before written).
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex[kMaxDevices];
void* g_scratch_addr[kMaxDevices];            // set once the lookup has succeeded

// Device address of the array on the current device.  A successful lookup is
// kept; a failed one (for instance no memory left to load the module) is not,
// so the next call tries again.  (On the host, `g_decode_scratch` names a
// host-side stand-in, not device memory.)
cudaError_t scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex[dev]);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();                       // do not leave the error for the next launch
      return e;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_static_scratch(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_blocks, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, float scale, int partition_size, pa_stream_t stream) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_context_len <= 0 ||
      head_dim <= 0 || block_size != pa::kBlockSize || partition_size < 0)
    return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     max_context_len, num_seqs, num_blocks, num_q_heads, num_kv_heads,
                     head_dim, block_size, scale, partition_size, nullptr, 0, stream);
  // Set-up on the first call on this device, whether or not this call needs scratch.
  void* ws = nullptr;
  const cudaError_t se = scratch_address(&ws);
  const size_t need = pa::workspace_for(num_seqs, num_q_heads, num_kv_heads, 1,
                                        max_context_len, head_dim, partition_size, 0);
  if (need == 0)
    return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     max_context_len, num_seqs, num_blocks, num_q_heads, num_kv_heads,
                     head_dim, block_size, scale, partition_size, nullptr, 0, stream);
  if (need > kStaticScratchBytes) {
    // Without scratch pa_decode runs its own checks first.  With the default
    // partition size (0) it then attends over whole sequences, which needs no
    // scratch; with an explicit partition size it returns PA_ERR_WORKSPACE
    // before launching anything.
    return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     max_context_len, num_seqs, num_blocks, num_q_heads, num_kv_heads,
                     head_dim, block_size, scale, partition_size, nullptr, 0, stream);
  }
  if (se != cudaSuccess) return PA_ERR_CUDA;
  return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                   max_context_len, num_seqs, num_blocks, num_q_heads, num_kv_heads, head_dim,
                   block_size, scale, partition_size, ws, kStaticScratchBytes, stream);
}
