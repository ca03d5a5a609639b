// CUDA-graph runner with batch-size classes for the decode / verify step.
//
// A captured graph replays a whole step with one launch call, but it fixes
// every pointer and every size.  So the runner captures one graph of the
// attention step per batch class (for example 1, 2, 4, 8, 16 sequences) over
// caller-owned static buffers sized for the largest class.  A step with B
// sequences pads the rows B .. c-1 of the smallest class c >= B with a dummy
// sequence (num_query_tokens tokens in a block nobody else uses), then replays
// graph c ("CUDA Graphs, modèles de raisonnement et service désagrégé", §1:
// capture once during warm-up, replay with one launch; pad incoming batches to
// fixed class sizes and update the inputs in place before the replay).
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <new>
#include <vector>

#include "paged_attn.h"
#include "pa_internal.h"

struct pa_graph_runner {
  pa_runner_config cfg{};
  pa_runner_buffers buf{};
  bool kernel_copy = false;                  // staging copies by the SMs (see stage_copy)
  std::vector<int> classes;
  std::vector<cudaGraphExec_t> execs;
  cudaStream_t capture_stream = nullptr;

  ~pa_graph_runner() {
    for (cudaGraphExec_t e : execs)
      if (e) cudaGraphExecDestroy(e);
    if (capture_stream) cudaStreamDestroy(capture_stream);
  }
};

namespace {

// The partition size a class is captured with: the configured one, or the library
// default for that batch size and page format.
int partition_for(const pa_runner_config& c, int num_seqs) {
  return c.partition_size > 0
             ? c.partition_size
             : pa::default_partition_for(c.max_context_len, num_seqs, c.num_kv_heads,
                                         c.kv_dtype == PA_KV_FP8_E4M3);
}

bool staged(const pa_runner_buffers& b) {
  return b.h_q && b.h_block_tables && b.h_context_lens && b.h_out &&
         (b.new_key == nullptr || (b.h_new_key && b.h_new_value));
}

// Page-locked host memory that the device addresses with the same pointer
// (unified addressing): the staging copies can then run as a kernel.
bool device_addressable_host(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();                      // clear the error of an unknown pointer
    return false;
  }
  return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One staging copy: by the SMs when both sides are device-addressable and 16-byte
// aligned (one kernel, no copy-engine transfer setup), else by cudaMemcpyAsync.
cudaError_t stage_copy(const pa_graph_runner& r, void* dst, const void* src, size_t bytes,
                       cudaMemcpyKind kind, cudaStream_t s) {
  if (r.kernel_copy && bytes % 16 == 0 && aligned16(dst) && aligned16(src))
    return pa::launch_stage_copy(dst, src, bytes, s);
  return cudaMemcpyAsync(dst, src, bytes, kind, s);
}

// When the host inputs and the device inputs each form one range, in the same
// order and at the same offsets (q, new_key, new_value, block_tables,
// context_lens), the bytes of that range for the largest class; else 0.
size_t one_range_bytes(const pa_graph_runner& r) {
  const pa_runner_buffers& b = r.buf;
  if (!b.new_key) return 0;
  const char* d0 = static_cast<const char*>(b.q);
  const char* h0 = static_cast<const char*>(b.h_q);
  const void* dev[4] = {b.new_key, b.new_value, b.block_tables, b.context_lens};
  const void* host[4] = {b.h_new_key, b.h_new_value, b.h_block_tables, b.h_context_lens};
  const char* prev = d0;
  for (int i = 0; i < 4; ++i) {
    const char* d = static_cast<const char*>(dev[i]);
    if (d <= prev || d - d0 != static_cast<const char*>(host[i]) - h0) return 0;
    prev = d;
  }
  const size_t bmax = static_cast<size_t>(r.classes.back());
  return static_cast<size_t>(reinterpret_cast<const char*>(b.context_lens + bmax) - d0);
}

// One step of num_seqs sequences as it is captured: [staging copies in],
// pa_attention, [staging copy out].
pa_status step_for(const pa_graph_runner& r, int num_seqs, cudaStream_t s) {
  const pa_runner_config& c = r.cfg;
  const pa_runner_buffers& b = r.buf;
  const size_t rows = static_cast<size_t>(num_seqs) * c.num_query_tokens;
  const size_t q_bytes = rows * c.num_q_heads * c.head_dim * 2;
  const size_t kv_bytes = rows * c.num_kv_heads * c.head_dim * 2;
  const bool stage = staged(b);
  const size_t one = stage ? one_range_bytes(r) : 0;
  constexpr cudaMemcpyKind H2D = cudaMemcpyHostToDevice;
  if (one > 0) {
    // every input in one copy (the whole range, sized for the largest class); a
    // kernel reads it only if its last byte is device-addressable host memory too
    const bool end_ok = device_addressable_host(static_cast<const char*>(b.h_q) + one - 1);
    if ((end_ok ? stage_copy(r, b.q, b.h_q, one, H2D, s)
                : cudaMemcpyAsync(b.q, b.h_q, one, H2D, s)) != cudaSuccess)
      return PA_ERR_CUDA;
  } else if (stage) {
    if (stage_copy(r, b.q, b.h_q, q_bytes, H2D, s) != cudaSuccess ||
        (b.new_key && (stage_copy(r, b.new_key, b.h_new_key, kv_bytes, H2D, s) != cudaSuccess ||
                       stage_copy(r, b.new_value, b.h_new_value, kv_bytes, H2D, s) !=
                           cudaSuccess)) ||
        stage_copy(r, b.block_tables, b.h_block_tables,
                   static_cast<size_t>(num_seqs) * c.max_blocks_per_seq * 4, H2D, s) !=
            cudaSuccess ||
        stage_copy(r, b.context_lens, b.h_context_lens, static_cast<size_t>(num_seqs) * 4, H2D,
                   s) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  const pa_status st =
      pa_attention(b.out, b.q, b.new_key, b.new_value, b.k_cache, b.v_cache, b.k_scale,
                   b.v_scale, c.kv_dtype, c.window_size, b.block_tables, c.max_blocks_per_seq,
                   b.context_lens, c.max_context_len, num_seqs, c.num_query_tokens,
                   c.num_blocks, c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size,
                   c.scale, partition_for(c, num_seqs), b.workspace, b.workspace_bytes,
                   reinterpret_cast<pa_stream_t>(s));
  if (st != PA_OK) return st;
  if (stage && stage_copy(r, b.h_out, b.out, q_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_runner_create(const pa_runner_config* cfg, const pa_runner_buffers* buffers,
                           pa_graph_runner** out) {
  if (!cfg || !buffers || !out || cfg->num_classes < 1 || !cfg->classes)
    return PA_ERR_INVALID_ARG;
  if (cfg->partition_size < 0 || cfg->pad_block < 0 || cfg->pad_block >= cfg->num_blocks ||
      cfg->num_query_tokens < 1 || cfg->max_context_len < cfg->num_query_tokens)
    return PA_ERR_INVALID_ARG;
  for (int i = 0; i < cfg->num_classes; ++i)
    if (cfg->classes[i] < 1 || (i > 0 && cfg->classes[i] <= cfg->classes[i - 1]))
      return PA_ERR_INVALID_ARG;
  pa_graph_runner* r = new (std::nothrow) pa_graph_runner();
  if (!r) return PA_ERR_INVALID_ARG;
  r->cfg = *cfg;
  r->buf = *buffers;
  r->classes.assign(cfg->classes, cfg->classes + cfg->num_classes);
  r->cfg.classes = nullptr;                   // the runner keeps its own copy
  if (staged(r->buf)) {
    const pa_runner_buffers& b = r->buf;
    r->kernel_copy = device_addressable_host(b.h_q) && device_addressable_host(b.h_block_tables) &&
                     device_addressable_host(b.h_context_lens) &&
                     device_addressable_host(b.h_out) &&
                     (b.new_key == nullptr || (device_addressable_host(b.h_new_key) &&
                                               device_addressable_host(b.h_new_value)));
  }
  if (cudaStreamCreateWithFlags(&r->capture_stream, cudaStreamNonBlocking) != cudaSuccess) {
    delete r;
    return PA_ERR_CUDA;
  }
  for (int c : r->classes) {
    cudaGraph_t graph = nullptr;
    if (cudaStreamBeginCapture(r->capture_stream, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
      delete r;
      return PA_ERR_CUDA;
    }
    const pa_status st = step_for(*r, c, r->capture_stream);
    const cudaError_t ce = cudaStreamEndCapture(r->capture_stream, &graph);
    if (st != PA_OK || ce != cudaSuccess || graph == nullptr) {
      if (graph) cudaGraphDestroy(graph);
      delete r;
      return st != PA_OK ? st : PA_ERR_CUDA;
    }
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) {
      delete r;
      return PA_ERR_CUDA;
    }
    r->execs.push_back(exec);
  }
  *out = r;
  return PA_OK;
}

int pa_runner_class_of(const pa_graph_runner* r, int num_seqs) {
  if (!r || num_seqs < 1) return -1;
  for (int c : r->classes)
    if (c >= num_seqs) return c;
  return -1;
}

pa_status pa_runner_step(pa_graph_runner* r, int num_seqs, pa_stream_t stream) {
  if (!r || num_seqs < 1) return PA_ERR_INVALID_ARG;
  const auto it = std::lower_bound(r->classes.begin(), r->classes.end(), num_seqs);
  if (it == r->classes.end()) return PA_ERR_UNSUPPORTED;
  const int c = *it;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (c > num_seqs && staged(r->buf)) {
    // pad the host rows; the class graph copies them in with the real ones
    for (int row = num_seqs; row < c; ++row) {
      int32_t* t = r->buf.h_block_tables + static_cast<size_t>(row) * r->cfg.max_blocks_per_seq;
      std::fill(t, t + r->cfg.max_blocks_per_seq, r->cfg.pad_block);
      r->buf.h_context_lens[row] = r->cfg.num_query_tokens;
    }
  } else if (c > num_seqs &&
             pa::launch_pad_rows(r->buf.block_tables, r->buf.context_lens, num_seqs, c,
                                 r->cfg.max_blocks_per_seq, r->cfg.pad_block,
                                 r->cfg.num_query_tokens, s) != cudaSuccess) {
    return PA_ERR_CUDA;
  }
  return cudaGraphLaunch(r->execs[static_cast<size_t>(it - r->classes.begin())], s) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

void pa_runner_destroy(pa_graph_runner* r) { delete r; }

}  // extern "C"
