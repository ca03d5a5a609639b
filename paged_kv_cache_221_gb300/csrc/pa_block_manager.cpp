// Host-side block manager of the paged KV cache (native C++, no CUDA calls).
//
// The KV cache is a pool of fixed-size physical blocks; each sequence owns an
// ordered list of block ids (its block table) and a token count.  Sequences
// that fork from one another (a shared prompt, beams, parallel completions)
// point at the same physical blocks, counted by a reference count per block;
// a block shared by several sequences is copied on the first write into it
// (copy-on-write).  ("PagedAttention, décodage spéculatif, MoE et Blackwell",
// §1: pagination de type système d'exploitation, partage de mémoire / copie
// sur écriture; "LLM inference optimization: KV cache", §4.1 and §4.2.)
//
// Deterministic policy: a new block is always the lowest-numbered free block.
// Not thread-safe: one manager per thread, or external locking.
#include <stdint.h>

#include <map>
#include <new>
#include <set>
#include <vector>

#include "paged_attn.h"

struct pa_block_manager {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int> refcount;        // per physical block; 0 = free
  std::set<int> free_blocks;        // ordered: allocation takes the smallest id
  struct Seq {
    std::vector<int> blocks;
    int num_tokens = 0;
  };
  std::map<int, Seq> seqs;

  int take() {
    const int b = *free_blocks.begin();
    free_blocks.erase(free_blocks.begin());
    refcount[b] = 1;
    return b;
  }
  void release(int b) {
    if (--refcount[b] == 0) free_blocks.insert(b);
  }
};

extern "C" {

pa_status pa_bm_create(int num_blocks, int block_size, pa_block_manager** out) {
  if (!out || num_blocks < 0 || block_size < 1) return PA_ERR_INVALID_ARG;
  pa_block_manager* bm = new (std::nothrow) pa_block_manager();
  if (!bm) return PA_ERR_INVALID_ARG;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->refcount.assign(static_cast<size_t>(num_blocks), 0);
  for (int b = 0; b < num_blocks; ++b) bm->free_blocks.insert(bm->free_blocks.end(), b);
  *out = bm;
  return PA_OK;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

pa_status pa_bm_add_sequence(pa_block_manager* bm, int seq_id, int num_tokens) {
  if (!bm || num_tokens < 0 || bm->seqs.count(seq_id)) return PA_ERR_INVALID_ARG;
  const long long need = (static_cast<long long>(num_tokens) + bm->block_size - 1) /
                         bm->block_size;
  if (need > static_cast<long long>(bm->free_blocks.size())) return PA_ERR_OUT_OF_BLOCKS;
  pa_block_manager::Seq s;
  s.num_tokens = num_tokens;
  for (long long i = 0; i < need; ++i) s.blocks.push_back(bm->take());
  bm->seqs.emplace(seq_id, std::move(s));
  return PA_OK;
}

pa_status pa_bm_fork(pa_block_manager* bm, int parent_id, int child_id) {
  if (!bm || parent_id == child_id) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(parent_id);
  if (it == bm->seqs.end() || bm->seqs.count(child_id)) return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq child = it->second;
  for (int b : child.blocks) ++bm->refcount[b];
  bm->seqs.emplace(child_id, std::move(child));
  return PA_OK;
}

pa_status pa_bm_append_slot(pa_block_manager* bm, int seq_id, int64_t* slot, int32_t* copy_src,
                            int32_t* copy_dst) {
  if (!bm || !slot || !copy_src || !copy_dst) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq& s = it->second;
  const int pos = s.num_tokens;
  const int off = pos % bm->block_size;
  *copy_src = -1;
  *copy_dst = -1;
  if (off == 0) {                                   // the last block is full: a new block
    if (bm->free_blocks.empty()) return PA_ERR_OUT_OF_BLOCKS;
    s.blocks.push_back(bm->take());
  } else if (bm->refcount[s.blocks.back()] > 1) {   // shared partial block: copy on write
    if (bm->free_blocks.empty()) return PA_ERR_OUT_OF_BLOCKS;
    const int old = s.blocks.back();
    const int fresh = bm->take();
    bm->release(old);
    s.blocks.back() = fresh;
    *copy_src = old;
    *copy_dst = fresh;
  }
  *slot = static_cast<int64_t>(s.blocks.back()) * bm->block_size + off;
  s.num_tokens = pos + 1;
  return PA_OK;
}

pa_status pa_bm_free_sequence(pa_block_manager* bm, int seq_id) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
  for (int b : it->second.blocks) bm->release(b);
  bm->seqs.erase(it);
  return PA_OK;
}

pa_status pa_bm_block_table(const pa_block_manager* bm, const int32_t* seq_ids, int num_seqs,
                            int max_blocks_per_seq, int32_t* block_tables,
                            int32_t* context_lens) {
  if (!bm || num_seqs < 0 || max_blocks_per_seq < 0) return PA_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!seq_ids || !block_tables || !context_lens)) return PA_ERR_INVALID_ARG;
  for (int i = 0; i < num_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
    if (static_cast<int>(it->second.blocks.size()) > max_blocks_per_seq)
      return PA_ERR_INVALID_ARG;
  }
  for (int i = 0; i < num_seqs; ++i) {
    const auto& s = bm->seqs.find(seq_ids[i])->second;
    int32_t* row = block_tables + static_cast<size_t>(i) * max_blocks_per_seq;
    for (int j = 0; j < max_blocks_per_seq; ++j)
      row[j] = j < static_cast<int>(s.blocks.size()) ? s.blocks[j] : -1;
    context_lens[i] = s.num_tokens;
  }
  return PA_OK;
}

int pa_bm_num_free_blocks(const pa_block_manager* bm) {
  return bm ? static_cast<int>(bm->free_blocks.size()) : -1;
}

int pa_bm_ref_count(const pa_block_manager* bm, int block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->refcount[block];
}

int pa_bm_num_tokens(const pa_block_manager* bm, int seq_id) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? -1 : it->second.num_tokens;
}

}  // extern "C"
