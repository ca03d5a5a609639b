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
// default for that batch size.
int partition_for(const pa_runner_config& c, int num_seqs) {
  return c.partition_size > 0 ? c.partition_size
                              : pa_default_partition_size(num_seqs, c.num_kv_heads,
                                                          c.max_context_len, c.block_size);
}

pa_status attention_for(const pa_graph_runner& r, int num_seqs, cudaStream_t s) {
  const pa_runner_config& c = r.cfg;
  const pa_runner_buffers& b = r.buf;
  return pa_attention(b.out, b.q, b.new_key, b.new_value, b.k_cache, b.v_cache, b.k_scale,
                      b.v_scale, c.kv_dtype, c.window_size, b.block_tables,
                      c.max_blocks_per_seq, b.context_lens, c.max_context_len, num_seqs,
                      c.num_query_tokens, c.num_blocks, c.num_q_heads, c.num_kv_heads,
                      c.head_dim, c.block_size, c.scale, partition_for(c, num_seqs),
                      b.workspace, b.workspace_bytes, reinterpret_cast<pa_stream_t>(s));
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
    const pa_status st = attention_for(*r, c, r->capture_stream);
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
  if (c > num_seqs &&
      pa::launch_pad_rows(r->buf.block_tables, r->buf.context_lens, num_seqs, c,
                          r->cfg.max_blocks_per_seq, r->cfg.pad_block,
                          r->cfg.num_query_tokens, s) != cudaSuccess)
    return PA_ERR_CUDA;
  return cudaGraphLaunch(r->execs[static_cast<size_t>(it - r->classes.begin())], s) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

void pa_runner_destroy(pa_graph_runner* r) { delete r; }

}  // extern "C"
