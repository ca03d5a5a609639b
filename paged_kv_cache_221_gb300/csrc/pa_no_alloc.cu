// pa_decode_static_scratch: pa_decode for callers that cannot allocate
// device memory.
//
// Some callers of a decode kernel are not allowed to allocate: a plugin that a
// host runtime hands only its input and output buffers, or a serving process
// that reserves all device memory at start-up and forbids cudaMalloc and
// cudaFree afterwards (both can synchronise the device and fragment the
// memory that was planned for the KV cache).  Such a caller cannot provide the
// split-KV scratch that pa_decode needs for long contexts.  This entry point
// takes that scratch from a fixed array that lives in this library's device
// image instead: the array is created when the library's module is loaded on a
// device and stays there until the process exits, on every GPU the library
// is loaded on.
#include <mutex>

#include "paged_attn.h"
#include "pa_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 32ull << 20;   // 32 MiB

// Split-KV partials of pa_decode_static_scratch (never read before written).
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
cudaError_t g_scratch_status[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

// Device address of the array on the current device, looked up once per device.
// (On the host, `g_decode_scratch` names a host-side stand-in, not device memory.)
cudaError_t scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_scratch_once[dev], [dev] {
    void* p = nullptr;
    g_scratch_status[dev] = cudaGetSymbolAddress(&p, g_decode_scratch);
    g_scratch_addr[dev] = p;
  });
  if (g_scratch_status[dev] != cudaSuccess) return g_scratch_status[dev];
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
  const size_t need = pa::workspace_for(num_seqs, num_q_heads, num_kv_heads, 1,
                                        max_context_len, head_dim, partition_size, 0);
  if (need > kStaticScratchBytes) return PA_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0 && scratch_address(&ws) != cudaSuccess) return PA_ERR_CUDA;
  return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                   max_context_len, num_seqs, num_blocks, num_q_heads, num_kv_heads, head_dim,
                   block_size, scale, partition_size, ws, need > 0 ? kStaticScratchBytes : 0,
                   stream);
}
