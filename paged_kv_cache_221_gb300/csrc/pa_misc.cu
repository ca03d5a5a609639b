// reshape_and_cache, the split-KV merge and the wait-timeout self test.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>

#include "pa_ptx.cuh"

namespace pa {

// ---------------------------------------------------------------- reshape_and_cache
// One thread per 16-byte vector of one (token, kv head) row of K and of V:
// slot s -> block s / block_size, offset s % block_size; bits copied unchanged.
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                             uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                             const int64_t* __restrict__ slots, int num_tokens, int hkv, int vecs,
                             int block_size, long long num_slots) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(num_tokens) * hkv * vecs;
  if (idx >= total) return;
  const int v = static_cast<int>(idx % vecs);
  const long long th = idx / vecs;
  const int h = static_cast<int>(th % hkv);
  const long long i = th / hkv;
  const long long s = slots[i];
  if (s < 0) return;                        // padding token
  if (s >= num_slots) {
    atomicOr(&g_pa_err, kErrBounds);
    return;
  }
  const long long blk = s / block_size, off = s % block_size;
  const size_t dst = ((static_cast<size_t>(blk) * hkv + h) * block_size + off) * vecs + v;
  const size_t src = (static_cast<size_t>(i) * hkv + h) * vecs + v;
  k_cache[dst] = key[src];
  v_cache[dst] = value[src];
}

cudaError_t launch_reshape(const void* key, const void* value, void* k_cache, void* v_cache,
                           const int64_t* slots, int num_tokens, int num_blocks, int hkv,
                           int head_dim, int block_size, cudaStream_t s) {
  const int vecs = head_dim / 8;
  const long long total = static_cast<long long>(num_tokens) * hkv * vecs;
  if (total == 0) return cudaSuccess;
  const long long blocks = (total + 255) / 256;
  reshape_and_cache_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slots, num_tokens, hkv, vecs,
      block_size, static_cast<long long>(num_blocks) * block_size);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- reshape_and_cache (FP8)
// One thread per 8 head dims of one (token, kv head): each bf16 value x is
// stored as the E4M3 code nearest to x / scale[head] (IEEE float32 division,
// round to nearest even, saturating to +-448).  K pages are token-major
// [NB, Hkv, 16, D]; V pages are transposed [NB, Hkv, D, 16], so one token's V
// lands as one byte in each of D rows of 16 bytes.  Consecutive threads take
// consecutive tokens of the same (kv head, 8 dims): the tokens of a prefill
// chunk fill consecutive slots, so a warp's V byte stores land in one or two
// 16-byte rows instead of 32 rows apart.

__global__ void __launch_bounds__(256)
    reshape_and_cache_fp8_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                 uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                                 const int64_t* __restrict__ slots,
                                 const float* __restrict__ k_scale,
                                 const float* __restrict__ v_scale, int num_tokens, int hkv,
                                 int head_dim, long long num_slots) {
  const int vecs = head_dim / 8;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(num_tokens) * hkv * vecs;
  if (idx >= total) return;
  const long long i = idx % num_tokens;
  const long long hv = idx / num_tokens;
  const int v = static_cast<int>(hv % vecs);
  const int h = static_cast<int>(hv / vecs);
  const long long s = slots[i];
  if (s < 0) return;                        // padding token
  if (s >= num_slots) {
    atomicOr(&g_pa_err, kErrBounds);
    return;
  }
  const long long blk = s / kBlockSize, off = s % kBlockSize;
  const size_t src = (static_cast<size_t>(i) * hkv + h) * vecs + v;
  const uint4 kx = key[src], vx = value[src];
  const float ks = k_scale[h], vs = v_scale[h];
  const uint32_t kw[4] = {kx.x, kx.y, kx.z, kx.w};
  const uint32_t vw[4] = {vx.x, vx.y, vx.z, vx.w};
  uint32_t kc[2] = {0u, 0u};
  const size_t page = static_cast<size_t>(blk) * hkv + h;
  uint8_t* vdst = v_cache + (page * head_dim + 8 * v) * kBlockSize + off;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t kp = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(kw[e]), ks),
                                        __fdiv_rn(bf16_hi(kw[e]), ks));
    const uint32_t vp = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(vw[e]), vs),
                                        __fdiv_rn(bf16_hi(vw[e]), vs));
    kc[e >> 1] |= kp << (16 * (e & 1));
    vdst[(2 * e) * kBlockSize] = static_cast<uint8_t>(vp & 0xFFu);
    vdst[(2 * e + 1) * kBlockSize] = static_cast<uint8_t>(vp >> 8);
  }
  *reinterpret_cast<uint2*>(k_cache + (page * kBlockSize + off) * head_dim + 8 * v) =
      make_uint2(kc[0], kc[1]);
}

cudaError_t launch_reshape_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slots, const float* k_scale, const float* v_scale,
                               int num_tokens, int num_blocks, int hkv, int head_dim,
                               cudaStream_t s) {
  const long long total = static_cast<long long>(num_tokens) * hkv * (head_dim / 8);
  if (total == 0) return cudaSuccess;
  const long long blocks = (total + 255) / 256;
  reshape_and_cache_fp8_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value),
      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), slots, k_scale, v_scale,
      num_tokens, hkv, head_dim, static_cast<long long>(num_blocks) * kBlockSize);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- copy_blocks
// Copy-on-write support: whole physical blocks (every kv head, K and V) are
// copied from pairs[i][0] to pairs[i][1], bits unchanged.  Grid: (chunks of
// one block, pair).  A pair naming a block outside the pool sets the BOUNDS
// bit and is skipped.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       const int32_t* __restrict__ pairs, int num_blocks, long long vecs) {
  const int src = pairs[2 * blockIdx.y], dst = pairs[2 * blockIdx.y + 1];
  if (static_cast<unsigned>(src) >= static_cast<unsigned>(num_blocks) ||
      static_cast<unsigned>(dst) >= static_cast<unsigned>(num_blocks)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&g_pa_err, kErrBounds);
    return;
  }
  if (src == dst) return;
  for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < vecs;
       v += static_cast<long long>(gridDim.x) * blockDim.x) {
    k_cache[dst * vecs + v] = k_cache[src * vecs + v];
    v_cache[dst * vecs + v] = v_cache[src * vecs + v];
  }
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                               int num_blocks, int hkv, int head_dim, int block_size,
                               cudaStream_t s) {
  if (num_pairs == 0) return cudaSuccess;
  const long long vecs = static_cast<long long>(hkv) * block_size * head_dim / 8;
  const long long chunks = (vecs + 255) / 256;
  dim3 grid(static_cast<unsigned>(chunks < 64 ? chunks : 64), static_cast<unsigned>(num_pairs), 1);
  copy_blocks_kernel<<<grid, 256, 0, s>>>(static_cast<uint4*>(k_cache),
                                          static_cast<uint4*>(v_cache), pairs, num_blocks, vecs);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- split-KV merge
// W warps per query row (W = 1, 2 or 4; 4/W rows per 128-thread CTA).  The
// rows of (sequence b, kv head g) are its G*T query rows (the q heads that read
// kv head g, times the query tokens).  Partition i of a row holds O_i
// (normalised) and (m_i, l_i): reference max in the log2 domain and sum of
// 2^(s - m_i).  The merged row is sum_i w_i O_i / sum_i w_i with
// w_i = l_i 2^(m_i - M), M = max_i m_i.  Warp k of a row merges partitions
// k, k + W, ... against its own max (lane j weighting partition j of each
// block of 32, every lane summing its head dims with eight 16-byte loads in
// flight); the W partial merges are then combined by the same rule.  A warp
// with at most kMergeFast partitions issues all their (m, l) and O loads at
// once, before it knows M, so the merge costs one memory round trip.
// Sequences that fit in one partition were written by the attention kernel
// directly and are skipped (same predicate).
// The kernel is launched as a programmatic dependent of the attention kernel
// (whose CTAs trigger at their start): it may become resident during the
// attention kernel's last wave and waits for that grid's completion before it
// reads any partial.
constexpr int kMergeWarps = 4;
constexpr int kMergeFast = 12;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    splitkv_reduce_kernel(const AttnParams p, int warps_per_row) {
  constexpr int DL = D / 32;                  // head dims per lane (4 or 2)
  __shared__ float s_acc[kMergeWarps][D];
  __shared__ float s_ms[kMergeWarps][2];
  const int W = warps_per_row;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (p.stream_ctl != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
    // The persistent decode kernel has made its last claim: reset its counter
    // for the next launch on this scratch.
    grid_dependency_wait();
    StreamCtl* ctl = static_cast<StreamCtl*>(p.stream_ctl);
    ctl->next = 0;
    __threadfence();
    ctl->tag = kStreamTag;
  }
  const int rows_per_cta = kMergeWarps / W;
  const int rows = p.G * p.T;
  const int chunks = (rows + rows_per_cta - 1) / rows_per_cta;
  const int bg = blockIdx.x / chunks;
  const int r = (blockIdx.x % chunks) * rows_per_cta + warp / W;
  const int sub = warp % W;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int L = p.context_lens[b];
  if (L < p.T || L > p.max_ctx) return;
  const int pre = (p.seq_group != nullptr && p.seq_group[b] >= 0)
                      ? p.group_prefix_blocks[p.seq_group[b]] : 0;
  if (pre < 0 || pre > p.max_prefix_blocks || pre * kBlockSize > L) return;
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  const int first =
      p.window > 0 ? max(pre, max(0, L - p.T - p.window + 1) / kBlockSize) : pre;
  const int npre = (pre + p.ppb - 1) / p.ppb;
  const int nparts = npre + (nblk - first + p.ppb - 1) / p.ppb;
  if (pre == 0 && nparts == 1) return;       // uniform over the CTA
  const bool live = r < rows;
  // row r = t * G + hl  ->  orow = (b*T + t)*Hq + g*G + hl
  const size_t orow =
      (static_cast<size_t>(b) * p.T + (live ? r : 0) / p.G) * p.Hq + g * p.G + (live ? r : 0) % p.G;
  const float2* ml = p.part_ml + orow * p.max_parts;
  const float* po = p.part_o + orow * p.max_parts * D + lane * DL;

  // this warp's partitions: sub, sub + W, sub + 2W, ...
  const int mine = live ? (nparts - sub + W - 1) / W : 0;
  float M = -CUDART_INF_F;
  float S = 0.f, acc[DL];
#pragma unroll
  for (int k = 0; k < DL; ++k) acc[k] = 0.f;
  grid_dependency_wait();                    // the attention grid's partials are complete
  if (mine <= kMergeFast) {
    // every lane loads every (m, l) (one broadcast each) and its head dims of every O
    float2 mv[kMergeFast];
    float xv[kMergeFast][DL];
#pragma unroll
    for (int k = 0; k < kMergeFast; ++k) {
      mv[k] = make_float2(-CUDART_INF_F, 0.f);
#pragma unroll
      for (int d = 0; d < DL; ++d) xv[k][d] = 0.f;
      if (k < mine) {
        mv[k] = ml[sub + k * W];
        const float* src = po + static_cast<size_t>(sub + k * W) * D;
        if constexpr (DL == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src);
          xv[k][0] = x.x;
          xv[k][1] = x.y;
          xv[k][2] = x.z;
          xv[k][3] = x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(src);
          xv[k][0] = x.x;
          xv[k][1] = x.y;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kMergeFast; ++k) M = fmaxf(M, mv[k].x);
#pragma unroll
    for (int k = 0; k < kMergeFast; ++k) {
      const float w = (mv[k].x == -CUDART_INF_F || M == -CUDART_INF_F)
                          ? 0.f : mv[k].y * exp2f(mv[k].x - M);
      S += w;
#pragma unroll
      for (int d = 0; d < DL; ++d) acc[d] += w * xv[k][d];
    }
  } else {
    for (int k = lane; k < mine; k += 32) M = fmaxf(M, ml[sub + k * W].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    for (int base = 0; base < mine; base += 32) {
      // (m, l) of this lane's partition of the block (an L1 hit, loaded just above)
      const float2 mlv = base + lane < mine ? ml[sub + (base + lane) * W]
                                            : make_float2(-CUDART_INF_F, 0.f);
      const float w = (mlv.x == -CUDART_INF_F || M == -CUDART_INF_F) ? 0.f
                                                                    : mlv.y * exp2f(mlv.x - M);
      S += w;
      const int n = min(32, mine - base);
#pragma unroll 8
      for (int k = 0; k < n; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        const float* src = po + static_cast<size_t>(sub + (base + k) * W) * D;
        if constexpr (DL == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src);
          acc[0] += wk * x.x;
          acc[1] += wk * x.y;
          acc[2] += wk * x.z;
          acc[3] += wk * x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(src);
          acc[0] += wk * x.x;
          acc[1] += wk * x.y;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  }

  if (W > 1) {
    // combine the W partial merges of the row: weights 2^(M_k - M_row)
#pragma unroll
    for (int k = 0; k < DL; ++k) s_acc[warp][lane * DL + k] = acc[k];
    if (lane == 0) {
      s_ms[warp][0] = M;
      s_ms[warp][1] = S;
    }
    __syncthreads();
    if (sub != 0 || !live) return;
    float Mr = -CUDART_INF_F;
    for (int k = 0; k < W; ++k) Mr = fmaxf(Mr, s_ms[warp + k][0]);
    S = 0.f;
#pragma unroll
    for (int d = 0; d < DL; ++d) acc[d] = 0.f;
    for (int k = 0; k < W; ++k) {
      const float Mk = s_ms[warp + k][0];
      const float f = (Mk == -CUDART_INF_F) ? 0.f : exp2f(Mk - Mr);
      S += f * s_ms[warp + k][1];
#pragma unroll
      for (int d = 0; d < DL; ++d) acc[d] += f * s_acc[warp + k][lane * DL + d];
    }
  }
  if (!live) return;
  const float inv = S > 0.f ? 1.f / S : 0.f;
  __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(p.out) + (orow * D + lane * DL) / 2;
#pragma unroll
  for (int k = 0; k < DL; k += 2) dst[k / 2] = __floats2bfloat162_rn(acc[k] * inv, acc[k + 1] * inv);
}

cudaError_t launch_reduce(const AttnParams& p, int head_dim, cudaStream_t s) {
  // more warps per row when rows have many partitions (more loads in flight)
  const int W = p.max_parts >= 32 ? 4 : (p.max_parts >= 12 ? 2 : 1);
  const int rows_per_cta = kMergeWarps / W;
  const long long chunks = (static_cast<long long>(p.G) * p.T + rows_per_cta - 1) / rows_per_cta;
  const long long ctas = static_cast<long long>(p.num_seqs) * p.Hkv * chunks;
  if (ctas == 0) return cudaSuccess;
  // programmatic stream serialisation: may start during the attention kernel's last wave
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (head_dim == 64) return cudaLaunchKernelEx(&cfg, splitkv_reduce_kernel<64>, p, W);
  return cudaLaunchKernelEx(&cfg, splitkv_reduce_kernel<128>, p, W);
}

// ---------------------------------------------------------------- graph runner staging
// Copy of 16-byte vectors by the SMs.  Used by the graph runner to move a step's
// inputs from page-locked host memory and its output back: host memory that the
// device addresses directly (unified addressing over the CPU-GPU link), so a
// small copy costs one kernel instead of a copy-engine transfer.
__global__ void stage_copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                  long long n) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    dst[i] = src[i];
}

cudaError_t launch_stage_copy(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  const long long n = static_cast<long long>(bytes / 16);
  const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 2 * 152));
  stage_copy_kernel<<<blocks, 256, 0, s>>>(static_cast<uint4*>(dst),
                                           static_cast<const uint4*>(src), n);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- graph runner padding
__global__ void pad_rows_kernel(int32_t* __restrict__ tables, int32_t* __restrict__ lens,
                                int from, int to, int mbs, int pad_block, int len) {
  const long long n = static_cast<long long>(to - from) * mbs;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int row = from + static_cast<int>(i / mbs);
    tables[static_cast<size_t>(row) * mbs + i % mbs] = pad_block;
    if (i % mbs == 0) lens[row] = len;
  }
}

cudaError_t launch_pad_rows(int32_t* block_tables, int32_t* context_lens, int from, int to,
                            int max_blocks_per_seq, int pad_block, int len, cudaStream_t s) {
  const long long n = static_cast<long long>(to - from) * max_blocks_per_seq;
  if (n <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 1024));
  pad_rows_kernel<<<blocks, 256, 0, s>>>(block_tables, context_lens, from, to,
                                         max_blocks_per_seq, pad_block, len);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- self test
// Waits on a barrier that nothing signals; the bounded wait must give up, set
// the TIMEOUT bit and let the kernel finish normally.
__global__ void selftest_wait_kernel(unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0u, timeout_ns);
}

cudaError_t launch_selftest_wait(unsigned long long timeout_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(timeout_ns);
  return cudaGetLastError();
}

cudaError_t take_error_misc(unsigned* bits) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_pa_err, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_pa_err, &zero, sizeof(zero));
  *bits |= v;
  return e;
}

}  // namespace pa
