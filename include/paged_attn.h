/*
 * paged_attn.h — C ABI of the GB300 (sm_103a) paged decode-attention library.
 *
 * The KV cache of every sequence is cut into fixed-size physical blocks of
 * `block_size` tokens (16) placed anywhere in one shared pool; a per-sequence
 * block table maps logical token blocks to physical ones and is resolved on the
 * fly inside the attention kernel ("PagedAttention, décodage spéculatif, MoE et
 * Blackwell", §1, pagination de type système d'exploitation; "LLM inference
 * optimization: KV cache", §4.1).
 *
 * Data layouts (all device pointers, row-major, contiguous, bf16 = IEEE
 * bfloat16 stored as 2 bytes):
 *   q, out        [num_seqs, num_query_tokens, num_q_heads, head_dim]   bf16
 *   k_cache,
 *   v_cache       [num_blocks, num_kv_heads, block_size, head_dim]      bf16
 *                 (one (block, kv head) "page" of block_size*head_dim values
 *                  is contiguous: 4 KB at head_dim 128)
 *   block_tables  [num_seqs, max_blocks_per_seq]                        int32
 *   context_lens  [num_seqs]                                            int32
 *   key, value    [num_tokens, num_kv_heads, head_dim]                  bf16
 *   slot_mapping  [num_tokens]   slot = physical_block*block_size+offset int64
 *
 * Conventions:
 *   - context_lens[b] counts every cached token of sequence b INCLUDING its
 *     num_query_tokens newest ones (the new decode token, or the drafts), whose
 *     K/V must already have been written with pa_reshape_and_cache.
 *   - Query head h reads kv head h / (num_q_heads / num_kv_heads).
 *   - Query token t of sequence b sees positions j <= context_lens[b] - T + t
 *     (T = num_query_tokens; a causal mask among the drafts).
 *   - Softmax statistics and accumulation are fp32; the output is rounded to
 *     bf16 (round to nearest even) once.
 *
 * Ownership: the caller owns every buffer.  The library never allocates or
 * frees device memory and keeps no per-call state on the host; `workspace` is
 * scratch the caller provides (its size comes from pa_workspace_size).
 *
 * Execution: every call only validates its arguments on the host, then
 * enqueues kernels on `stream` and returns; it never synchronises (except
 * pa_get_device_error, which says so).
 *
 * Kernels: per-sequence attention runs in a one-CTA-per-work-unit kernel or,
 * for at most 8 or 17-24 query rows per kv head, in a persistent kernel whose
 * CTAs stream units back to back (chosen for FP8 pages and for launches with
 * at least 4 units per resident CTA).  Both give bit-identical results.  The
 * environment variable PA_DECODE_KERNEL ("per_unit" or "persistent", read on
 * every call) forces one of them; PA_VERIFY_KERNEL = "tcgen05" selects a
 * tensor-memory kernel for 17-32 rows at head_dim 128 with bf16 pages (within
 * the same tolerance of the exact result, not bit-identical, and slower on
 * GB300 than the default).  Neither variable changes argument checks or
 * scratch sizes.
 *
 * Errors: argument errors are returned synchronously and nothing is launched.
 * A launch failure returns PA_ERR_CUDA.  Conditions only the device can see
 * (a block id outside the pool, a slot outside the pool, a context length
 * above max_context_len or below num_query_tokens, a pipeline wait that
 * exceeded its time limit) set a sticky device error word; the affected work
 * is skipped, never read or written out of bounds, and pa_get_device_error
 * reports the condition.  Nothing throws across this ABI.
 */
#ifndef PAGED_ATTN_H
#define PAGED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t / CUstream; NULL = legacy default stream. */
typedef struct CUstream_st* pa_stream_t;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size, misaligned pointer, ...      */
  PA_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim not 64/128, ...       */
  PA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than pa_workspace_size */
  PA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed                */
  PA_ERR_BOUNDS = 5,        /* device saw a block id / slot / length out of range  */
  PA_ERR_TIMEOUT = 6,       /* device pipeline wait exceeded its limit             */
  PA_ERR_OUT_OF_BLOCKS = 7  /* block manager: no free physical block left          */
} pa_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* pa_status_string(int status);

/* ABI version of this library (major*100 + minor). */
int pa_version(void);

/* Which kernel the last per-sequence attention launch made by this host thread
 * used (a diagnostic; the choice is described under "Kernels" above):
 * PA_KERNEL_NONE (no launch yet on this thread), PA_KERNEL_PER_UNIT (one CTA per
 * work unit), PA_KERNEL_PERSISTENT, PA_KERNEL_TCGEN05.  Group (shared-prefix)
 * launches do not change it.  No device work, no error. */
enum { PA_KERNEL_NONE = 0, PA_KERNEL_PER_UNIT = 1, PA_KERNEL_PERSISTENT = 2,
       PA_KERNEL_TCGEN05 = 3 };
int pa_last_attention_kernel(void);

/*
 * pa_reshape_and_cache — store the K and V vectors of `num_tokens` new tokens
 * into their cache slots: for token i with s = slot_mapping[i] >= 0,
 *   k_cache[s / block_size, h, s % block_size, :] = key[i, h, :]   for all h
 * and the same for V.  A negative slot marks a padding token and is skipped.
 * Bits are copied unchanged (bit-exact).  Two tokens naming the same slot leave
 * that slot holding one of them (which one is unspecified).
 * Cited: "LLM inference optimization: KV cache", §3.1 (the new token's K and V
 * are saved into the KV cache); the slot arithmetic follows from the block
 * layout above.
 * Requirements: all pointers non-NULL and 16-byte aligned, head_dim a multiple
 * of 8, block_size 16.  A slot >= num_blocks*block_size sets PA_ERR_BOUNDS on
 * the device and that token is skipped.
 */
pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache,
                               void* v_cache, const int64_t* slot_mapping, int num_tokens,
                               int num_blocks, int num_kv_heads, int head_dim, int block_size,
                               pa_stream_t stream);

/*
 * pa_workspace_size — bytes of scratch the attention calls need for split-KV
 * partials with these sizes (0 if no sequence can need more than one
 * partition).  With partition_size = 0 it returns the largest need of the
 * library default over every kv-head count that divides num_q_heads (the
 * default depends on num_kv_heads, which this call does not take), so the
 * result always suffices.  max_prefix_blocks is 0 for pa_decode / pa_verify.
 */
size_t pa_workspace_size(int num_seqs, int num_q_heads, int num_query_tokens,
                         int max_context_len, int head_dim, int block_size, int partition_size,
                         int max_prefix_blocks);

/* Partition size (tokens) that partition_size = 0 selects for this shape, bf16
 * pages.  Per-sequence calls over FP8 pages select 4096 tokens instead where
 * this returns 2048 or 3072 (contexts past 4096 tokens, 256 or more (sequence,
 * kv head) pairs); their scratch need is then at most the bf16 one. */
int pa_default_partition_size(int num_seqs, int num_kv_heads, int max_context_len,
                              int block_size);

/*
 * pa_decode — single-token paged decode attention (num_query_tokens = 1):
 *   out[b, 0, h, :] = sum_j softmax_j(scale * q[b,0,h,:] . K_j) V_j
 * over the context_lens[b] cached positions j of sequence b, K_j / V_j read
 * from page block_tables[b, j / block_size], slot j % block_size, kv head
 * h / (Hq/Hkv).  Cited: "LLM inference optimization: KV cache", §3.1 (attention
 * from the new token's Q over the cached K, V) and §4.1 (block table);
 * "PagedAttention, ..." §1.
 *
 * Long contexts are split into partitions of partition_size tokens (0 = the
 * library default) that are processed in parallel and merged with the
 * log-sum-exp rule by a second kernel; this needs `workspace` of at least
 * pa_workspace_size(...) bytes.  The workspace needs no initialisation (every
 * partial is written before it is read) and may be reused by later calls on
 * the same stream.  Its last 256 bytes also carry, from one call to the next,
 * the work-claim counter of the persistent decode kernel (at most 8 query rows
 * per kv head): a tagged counter that the merge kernel zeroes at the end of
 * each call; a workspace that is new or was overwritten in between lacks the
 * tag, and the next call then takes work units in a fixed order and sets the
 * tag.  Two calls in flight at once must not share a workspace (their
 * partials would collide anyway).  With partition_size = 0 and workspace == NULL every
 * sequence is processed whole (no scratch, fewer parallel units).  With an
 * explicit partition_size that needs scratch, a missing or short workspace
 * returns PA_ERR_WORKSPACE.
 *
 * max_context_len must bound every context_lens[b] and be at most
 * max_blocks_per_seq*block_size; it sizes the launch without a device read.
 * At most 4096 partitions per sequence (PA_ERR_UNSUPPORTED beyond: choose a
 * larger partition_size).
 * Requirements: head_dim 64 or 128, block_size 16, num_q_heads a multiple of
 * num_kv_heads with at most 64 query heads per kv head, q/out/k_cache/v_cache
 * 16-byte aligned, num_blocks*num_kv_heads*block_size < 2^31.
 */
pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int max_context_len, int num_seqs,
                    int num_blocks, int num_q_heads, int num_kv_heads, int head_dim,
                    int block_size, float scale, int partition_size, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_verify — speculative-decoding verification: the num_query_tokens (T)
 * draft tokens of every sequence attend over the paged cache in one pass,
 * draft t seeing positions j <= context_lens[b] - T + t (causal mask among the
 * drafts, whose K/V occupy the last T positions).  Cited: "PagedAttention, ..."
 * §1 (vérification parallèle of K drafts in one forward pass); "LLM inference
 * optimization: KV cache", §5.2.  Other arguments as pa_decode; requires
 * 1 <= T and (num_q_heads/num_kv_heads) * T <= 64.
 */
pa_status pa_verify(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int max_context_len, int num_seqs,
                    int num_query_tokens, int num_blocks, int num_q_heads, int num_kv_heads,
                    int head_dim, int block_size, float scale, int partition_size,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * FP8 (E4M3) pages — the same cache with every K and V value stored as one
 * byte, which halves the bytes decode streams ("ranksignal" post, Quantifier :
 * des nombres plus petits: halving the precision halves what decode loads, FP8
 * being the usual compromise, the softmax kept at full precision;
 * "PagedAttention, ..." §3 on FP8).  Format: E4M3 without infinities (sign,
 * 4-bit exponent with bias 7, 3-bit mantissa; exponent 0 = subnormals m*2^-9;
 * 0x7F / 0xFF = NaN; largest magnitude 448).  Scales: k_scale[h], v_scale[h]
 * (device float32 [num_kv_heads]) are chosen by the caller; a value x of kv
 * head h is stored as the code nearest to x / scale[h] and read as
 * value(code) * scale[h].  Layouts (uint8, each (block, kv head) page
 * contiguous, block_size*head_dim bytes):
 *   k_cache  [num_blocks, num_kv_heads, block_size, head_dim]   (token-major)
 *   v_cache  [num_blocks, num_kv_heads, head_dim, block_size]   (transposed)
 */

/*
 * pa_reshape_and_cache_fp8 — pa_reshape_and_cache into FP8 pages: for token i
 * with s = slot_mapping[i] >= 0, block = s / block_size, t = s % block_size,
 *   k_cache[block, h, t, d] = e4m3(key[i, h, d] / k_scale[h])
 *   v_cache[block, h, d, t] = e4m3(value[i, h, d] / v_scale[h])
 * where the division is IEEE float32 and e4m3() rounds to nearest even and
 * saturates to +-448 (NaN stays NaN).  key/value are bf16 [num_tokens,
 * num_kv_heads, head_dim].  Requirements and errors as pa_reshape_and_cache;
 * k_scale and v_scale non-NULL.
 */
pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, void* k_cache,
                                   void* v_cache, const int64_t* slot_mapping,
                                   const float* k_scale, const float* v_scale, int num_tokens,
                                   int num_blocks, int num_kv_heads, int head_dim, int block_size,
                                   pa_stream_t stream);

/*
 * pa_decode_fp8 / pa_verify_fp8 — pa_decode / pa_verify over FP8 pages: the
 * same result with K_j = value(k code) * k_scale[h] and V_j = value(v code) *
 * v_scale[h].  The products run on f16 operands with fp32 accumulation: q is
 * converted to f16 (exact for |q| in [2^-14, 65504]; larger magnitudes are
 * not supported, smaller ones lose the bits below 2^-24) and the softmax
 * weights are rounded to f16 before they multiply V.  Workspace, partitions,
 * requirements and errors as pa_decode / pa_verify, plus k_scale, v_scale
 * non-NULL; partition_size 0 selects the FP8 rule of pa_default_partition_size
 * (4096-token partitions past 4096-token contexts), whose scratch need is at
 * most pa_workspace_size's.
 */
pa_status pa_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens,
                        int max_context_len, int num_seqs, int num_blocks, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, float scale,
                        int partition_size, void* workspace, size_t workspace_bytes,
                        pa_stream_t stream);

pa_status pa_verify_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens,
                        int max_context_len, int num_seqs, int num_query_tokens, int num_blocks,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        float scale, int partition_size, void* workspace,
                        size_t workspace_bytes, pa_stream_t stream);

/* KV page formats for pa_attention. */
enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1 };

/*
 * pa_attention — the general per-sequence call; pa_decode, pa_verify,
 * pa_decode_append and their _fp8 forms are special cases of it.
 *   kv_dtype     PA_KV_BF16 (pools as in pa_decode) or PA_KV_FP8_E4M3 (pools and
 *                scales as in pa_decode_fp8; k_scale / v_scale ignored for bf16)
 *   new_key,
 *   new_value    NULL, or the query tokens' K/V (bf16 [num_seqs *
 *                num_query_tokens, num_kv_heads, head_dim]) to store at positions
 *                context_lens[b] - T .. context_lens[b] - 1 inside the launch, as
 *                pa_decode_append / pa_decode_append_fp8 do (both or neither)
 *   window_size  0: every query token sees its whole causal context.  W > 0: a
 *                sliding window; query token t, at position pos = context_lens[b]
 *                - T + t, sees only positions j with pos - W < j <= pos, and
 *                blocks wholly before the first query's window are not read.
 * Cited for the window: "ranksignal" post, the attention-kernels section
 * (sliding-window attention looks only at the latest tokens; the window size
 * is a parameter).  Other arguments, requirements and errors as pa_verify;
 * window_size < 0 is PA_ERR_INVALID_ARG.
 */
pa_status pa_attention(void* out, const void* q, const void* new_key, const void* new_value,
                       void* k_cache, void* v_cache, const float* k_scale, const float* v_scale,
                       int kv_dtype, int window_size, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                       int num_seqs, int num_query_tokens, int num_blocks, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, float scale,
                       int partition_size, void* workspace, size_t workspace_bytes,
                       pa_stream_t stream);

/*
 * pa_decode_append_fp8 — pa_reshape_and_cache_fp8 fused into pa_verify_fp8
 * (the FP8 counterpart of pa_decode_append below): the num_query_tokens new
 * tokens of every sequence, new_key / new_value bf16 [num_seqs *
 * num_query_tokens, num_kv_heads, head_dim] in sequence-major order, are
 * quantised exactly as pa_reshape_and_cache_fp8 does and stored at positions
 * context_lens[b] - T .. context_lens[b] - 1 of each sequence's pages inside the
 * attention launch, before those pages are read.  The pools are written, so
 * they are not const.  Other arguments, requirements and errors as
 * pa_verify_fp8; new_key and new_value must be 16-byte aligned.
 */
pa_status pa_decode_append_fp8(void* out, const void* q, const void* new_key,
                               const void* new_value, void* k_cache, void* v_cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int max_context_len, int num_seqs,
                               int num_query_tokens, int num_blocks, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, float scale,
                               int partition_size, void* workspace, size_t workspace_bytes,
                               pa_stream_t stream);

/*
 * pa_decode_append — reshape_and_cache fused into the attention call: the K
 * and V vectors of every sequence's num_query_tokens (T) query tokens,
 *   new_key, new_value  [num_seqs, T, num_kv_heads, head_dim]  bf16,
 * are stored at positions context_lens[b] - T + t of their sequence (block
 * block_tables[b, pos / block_size], slot pos % block_size, bit-exact) by the
 * attention CTA that reads that page, immediately before it reads it; then the
 * call computes pa_verify (pa_decode for T = 1).  Same result as
 * pa_reshape_and_cache with those slots followed by pa_verify, in one launch.
 * Cited: "LLM inference optimization: KV cache", §3.1 and its diagram (the
 * new token's K and V are saved into the cache, then attention reads the cache).
 * k_cache / v_cache are written; other arguments and errors as pa_verify.
 */
pa_status pa_decode_append(void* out, const void* q, const void* new_key, const void* new_value,
                           void* k_cache, void* v_cache, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* context_lens,
                           int max_context_len, int num_seqs, int num_query_tokens,
                           int num_blocks, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, float scale, int partition_size, void* workspace,
                           size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_shared_prefix — pa_decode for batches where groups of sequences
 * share their first blocks copy-on-write (one prompt, several beams or
 * parallel completions point at the same physical blocks: "PagedAttention,
 * ..." §1, partage de mémoire; "LLM inference optimization: KV cache", §4.2).
 * The shared pages of a group are read from memory once per kv head for all
 * members of the group together; the members' private pages are read per
 * sequence; all partial results are merged per sequence.  The result equals
 * pa_decode on the same tables.
 *
 *   seq_group[b]            group of sequence b, or -1 if it shares nothing
 *   group_prefix_blocks[g]  number of leading block-table entries that are
 *                           identical in the tables of every member of g
 *   max_group_size          upper bound on members per group (host-side sizing)
 *   max_prefix_blocks       upper bound on group_prefix_blocks[g]
 * Every member must have context_lens[b] >= group_prefix_blocks[g]*block_size.
 * Requires a workspace of pa_workspace_size(..., max_prefix_blocks) bytes.
 */
pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_tables,
                                  int max_blocks_per_seq, const int32_t* context_lens,
                                  int max_context_len, int num_seqs, int num_blocks,
                                  int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, float scale, int partition_size,
                                  const int32_t* seq_group, const int32_t* group_prefix_blocks,
                                  int num_groups, int max_group_size, int max_prefix_blocks,
                                  void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_shared_prefix_fp8 — pa_decode_shared_prefix over FP8 (E4M3) pages
 * and per-kv-head scales, laid out as for pa_decode_fp8: the group's prefix
 * pages are read once per group, the private pages once per sequence.
 * Arguments, requirements and errors as pa_decode_shared_prefix, plus k_scale
 * and v_scale non-NULL.
 */
pa_status pa_decode_shared_prefix_fp8(
    void* out, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
    const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len, int num_seqs, int num_blocks,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
    int partition_size, const int32_t* seq_group, const int32_t* group_prefix_blocks,
    int num_groups, int max_group_size, int max_prefix_blocks, void* workspace,
    size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_static_scratch — pa_decode without caller-provided scratch, for
 * callers that may not allocate device memory: a plugin that its host runtime
 * gives only input and output buffers, or a server that reserves all device
 * memory at start-up and must not call cudaMalloc/cudaFree afterwards.  The
 * paper has no counterpart; this is a library convenience.
 *
 * The split-KV scratch comes from one fixed array of 32 MiB (33554432 bytes)
 * inside this library's device image, held until the process exits on every
 * GPU where it has been loaded.  If the call needs more than 32 MiB (the
 * scratch pa_decode needs with these sizes, num_kv_heads included): with
 * partition_size 0 it attends over whole sequences, which needs no scratch
 * (the result pa_decode gives without a workspace); with an explicit
 * partition_size it returns PA_ERR_WORKSPACE and launches nothing.  Argument
 * errors take precedence over PA_ERR_WORKSPACE, as in pa_decode.
 *
 * Set-up: the first call on each device, with that device current, looks up
 * the array's device address (cudaGetSymbolAddress).  Under CUDA's lazy module
 * loading, the default, that lookup is also what loads the array onto the
 * device, so that first call reserves the 32 MiB (with
 * CUDA_MODULE_LOADING=EAGER the array is loaded with the library instead).
 * Make the first call on each device during start-up, before the rest of
 * device memory is reserved and before any stream capture.  A failed lookup
 * returns PA_ERR_CUDA (when the call needs scratch) and is retried by the next
 * call.  After set-up, no call allocates device memory.
 *
 * All calls in the process share the one array and it keeps what the last
 * call wrote; nothing in it needs to start at zero (every partial is written
 * before it is read).  Calls whose executions overlap on the GPU (e.g. on two
 * streams) race on the array: serialise them.  Arguments, results and errors
 * are otherwise those of pa_decode.
 */
pa_status pa_decode_static_scratch(void* out, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables,
                                   int max_blocks_per_seq, const int32_t* context_lens,
                                   int max_context_len, int num_seqs, int num_blocks,
                                   int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, float scale, int partition_size,
                                   pa_stream_t stream);

/*
 * pa_copy_blocks — copy whole physical blocks (every kv head, K and V pools)
 * for copy-on-write: for each i, block block_pairs[2i] is copied onto block
 * block_pairs[2i+1] (device int32 pairs), bits unchanged.  Used after
 * pa_bm_append_slot reports a copy, before the new token is written.  A pair
 * naming a block outside the pool sets PA_ERR_BOUNDS on the device and is
 * skipped; a destination must not also be a source in the same call.
 * Cited: "PagedAttention, ..." §1 (partage de mémoire, copie sur écriture);
 * "LLM inference optimization: KV cache", §4.2.
 */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs,
                         int num_pairs, int num_blocks, int num_kv_heads, int head_dim,
                         int block_size, pa_stream_t stream);

/*
 * pa_spec_accept — speculative decoding, after pa_verify: which of the K draft
 * tokens of each sequence the target keeps, and the one token the target then
 * emits ("ranksignal" post, Spéculer : plusieurs tokens par passe: drafts are
 * kept while they agree with the target, the first disagreement drops every
 * later draft, and the target adds one token of its own; "LLM inference
 * optimization: KV cache", §5.2 and §5.3: with rejection sampling the output
 * follows the target's distribution exactly).
 *
 *   target_probs     [num_seqs, K + 1, vocab]  float32  target probabilities at
 *                    the K draft positions and the bonus position K
 *   draft_probs      [num_seqs, K, vocab]      float32  (sampling only)
 *   draft_tokens     [num_seqs, K]             int32
 *   accept_uniforms  [num_seqs, K]             uint32   low 24 bits used (sampling)
 *   sample_uniforms  [num_seqs]                uint32   (sampling)
 *   out_tokens       [num_seqs, K + 1]         int32    kept drafts, then the emitted
 *                    token, then -1
 *   num_accepted     [num_seqs]                int32    number of kept drafts
 *
 * greedy != 0: draft i is kept while it equals the most probable token of row
 * i (lowest index on ties); the emitted token is the most probable token of the
 * first row whose draft differs (row K if every draft is kept).
 * greedy == 0 (rejection sampling): draft x_i is kept iff
 * draft_probs[i][x_i] * a_i < target_probs[i][x_i] * 2^24 (a_i = low 24 bits of
 * accept_uniforms, compared exactly); the emitted token is drawn from
 * max(0, p_i - q_i) (float32) at the first rejected position i, or from p_K,
 * by an exact integer inverse-CDF draw: weights w(x) = floor(r(x) * 2^40), W =
 * sum w, token = the smallest x whose prefix sum of w exceeds
 * floor(sample_uniform * W / 2^32); if W = 0, the most probable token of that
 * row.  The result does not depend on summation order.
 * Requirements: 1 <= vocab <= 2^19, 0 <= K <= 64, probabilities finite and in
 * [0, 1].  A draft token outside [0, vocab) sets PA_ERR_BOUNDS on the device
 * and is treated as not kept.  One CTA per sequence; all device pointers.
 */
pa_status pa_spec_accept(const float* target_probs, const float* draft_probs,
                         const int32_t* draft_tokens, const uint32_t* accept_uniforms,
                         const uint32_t* sample_uniforms, int num_seqs, int num_drafts,
                         int vocab_size, int greedy, int32_t* out_tokens, int32_t* num_accepted,
                         pa_stream_t stream);

/*
 * Graph runner — CUDA graphs of the attention step for fixed batch-size
 * classes ("CUDA Graphs, modèles de raisonnement et service désagrégé", §1:
 * a captured graph replays a whole step with one launch call but needs static
 * addresses and shapes, so incoming batches are padded to fixed class sizes
 * such as 1, 2, 4, 8, 16 and the inputs are updated in place before replay).
 *
 * pa_runner_create captures, for every class c, one pa_attention call with
 * num_seqs = c over the caller's static buffers (sized for the largest class;
 * the runner keeps their addresses, the caller keeps them alive and writes the
 * step's inputs into them: q, new_key / new_value, block_tables, context_lens
 * rows 0 .. B-1).  pa_runner_step(B) pads rows B .. c-1 of the smallest class
 * c >= B with a one-block dummy sequence (context num_query_tokens, every table
 * entry pad_block, a physical block no sequence uses and that the padded rows'
 * appends may overwrite), then replays graph c on `stream`.  Output rows 0 .. B-1
 * are those of pa_attention with num_seqs = B and the class's partition size:
 * partition_size if > 0, else the library default for num_seqs = c
 * (pa_default_partition_size, with its FP8 rule for FP8 pages).  max_context_len is the bound every captured
 * launch is sized for.  The workspace must hold the largest need over the
 * classes (pa_workspace_size for each class).  The runner owns
 * one CUDA stream (for capture) and the instantiated graphs, nothing else.
 * pa_runner_step returns PA_ERR_UNSUPPORTED when B exceeds the largest class.
 */
typedef struct pa_runner_config {
  int num_q_heads, num_kv_heads, head_dim, block_size;
  int num_query_tokens;
  int max_blocks_per_seq, max_context_len, num_blocks;
  int kv_dtype, window_size, partition_size;
  float scale;
  int pad_block;
  int num_classes;
  const int* classes;          /* host array, strictly increasing, each >= 1 */
} pa_runner_config;

typedef struct pa_runner_buffers {   /* device pointers, as for pa_attention */
  void* out;
  void* q;
  void* new_key;                     /* NULL: no fused append */
  void* new_value;
  int32_t* block_tables;
  int32_t* context_lens;
  void* k_cache;
  void* v_cache;
  const float* k_scale;              /* FP8 pages only */
  const float* v_scale;
  void* workspace;
  size_t workspace_bytes;
  /* Optional host staging (page-locked host memory, same shapes as the device
   * buffers above; all NULL = none).  With staging every class graph also holds
   * the copies of its c rows of q, new_key, new_value, block_tables and
   * context_lens from these buffers to the device buffers before the attention
   * call, and the copy of c rows of out back to h_out after it; pa_runner_step
   * then pads host rows B .. c-1 of h_block_tables / h_context_lens on the CPU
   * instead of launching the padding kernel.  When the five host inputs and the
   * five device inputs each lie in one range, in the order q, new_key,
   * new_value, block_tables, context_lens and at the same offsets, the graph
   * copies that whole range (sized for the largest class) in one piece.  When
   * every host buffer is page-locked memory that the device addresses with the
   * same pointer (checked once, at creation), the copies are made by a kernel
   * of the class graph (16-byte vectors; sizes and addresses multiples of 16),
   * otherwise by cudaMemcpyAsync.  Read h_out, and rewrite the host inputs for
   * the next step, only after the stream has finished the step. */
  void* h_q;
  void* h_new_key;
  void* h_new_value;
  int32_t* h_block_tables;
  int32_t* h_context_lens;
  void* h_out;
} pa_runner_buffers;

typedef struct pa_graph_runner pa_graph_runner;

pa_status pa_runner_create(const pa_runner_config* config, const pa_runner_buffers* buffers,
                           pa_graph_runner** out);
pa_status pa_runner_step(pa_graph_runner* runner, int num_seqs, pa_stream_t stream);
/* The class a batch of num_seqs would use, or -1 if none is large enough. */
int pa_runner_class_of(const pa_graph_runner* runner, int num_seqs);
void pa_runner_destroy(pa_graph_runner* runner);

/*
 * Block manager — host-side bookkeeping of the physical block pool (no device
 * memory, no CUDA calls): sequences own ordered lists of physical blocks (their
 * block tables); forked sequences share blocks through reference counts; the
 * first write into a shared, partly filled block copies it (copy-on-write).
 * Cited: "PagedAttention, ..." §1 (blocks placed anywhere, block table,
 * partage de mémoire / copie sur écriture); "LLM inference optimization: KV
 * cache", §4.1 (only the blocks needed are allocated), §4.2.
 * Policy: a new block is always the lowest-numbered free block.  Not
 * thread-safe.  Sequence ids are arbitrary ints.
 */
typedef struct pa_block_manager pa_block_manager;

/* A manager for num_blocks blocks of block_size tokens; *out receives it. */
pa_status pa_bm_create(int num_blocks, int block_size, pa_block_manager** out);
void pa_bm_destroy(pa_block_manager* bm);

/* New sequence holding num_tokens tokens (ceil(num_tokens/block_size) fresh
 * blocks).  PA_ERR_OUT_OF_BLOCKS (nothing changed) if too few are free;
 * PA_ERR_INVALID_ARG if seq_id exists. */
pa_status pa_bm_add_sequence(pa_block_manager* bm, int seq_id, int num_tokens);

/* child_id shares every block of parent_id (reference counts + 1). */
pa_status pa_bm_fork(pa_block_manager* bm, int parent_id, int child_id);

/* Reserve the slot of the sequence's next token and count the token.  If the
 * last block is full a fresh block is appended; if it is partly filled and
 * shared, it is replaced by a fresh block and *copy_src -> *copy_dst names
 * the copy to run (pa_copy_blocks) before writing; otherwise both are -1.
 * *slot = physical_block*block_size + offset.  PA_ERR_OUT_OF_BLOCKS leaves the
 * manager unchanged. */
pa_status pa_bm_append_slot(pa_block_manager* bm, int seq_id, int64_t* slot, int32_t* copy_src,
                            int32_t* copy_dst);

/* Drop a sequence; blocks whose reference count reaches 0 become free. */
pa_status pa_bm_free_sequence(pa_block_manager* bm, int seq_id);

/* Host arrays: block_tables [num_seqs, max_blocks_per_seq] (-1 past the end)
 * and context_lens [num_seqs] for the given sequences.  PA_ERR_INVALID_ARG if
 * a sequence is unknown or holds more than max_blocks_per_seq blocks. */
pa_status pa_bm_block_table(const pa_block_manager* bm, const int32_t* seq_ids, int num_seqs,
                            int max_blocks_per_seq, int32_t* block_tables,
                            int32_t* context_lens);

/* Free blocks; reference count of a block; tokens of a sequence (-1: unknown). */
int pa_bm_num_free_blocks(const pa_block_manager* bm);
int pa_bm_ref_count(const pa_block_manager* bm, int block);
int pa_bm_num_tokens(const pa_block_manager* bm, int seq_id);

/*
 * pa_get_device_error — synchronise `stream`, then return and clear the sticky
 * device error word: PA_ERR_TIMEOUT if any pipeline wait gave up, else
 * PA_ERR_BOUNDS if any out-of-range id, slot or length was seen, else PA_OK
 * (PA_ERR_CUDA if the synchronisation itself failed).
 */
pa_status pa_get_device_error(pa_stream_t stream);

/*
 * pa_selftest_wait_timeout — failure-detection self test.  Launches one CTA
 * that waits on a shared-memory barrier nothing ever signals, with a limit of
 * timeout_ns nanoseconds (1000 .. 10^9); the wait gives up, records
 * PA_ERR_TIMEOUT in the device error word and the kernel returns normally.
 * Read the result with pa_get_device_error.  Nothing faults or hangs.
 */
pa_status pa_selftest_wait_timeout(unsigned long long timeout_ns, pa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PAGED_ATTN_H */
