// reshape_and_cache, the split-KV merge and the wait-timeout self test.
#include <cuda_bf16.h>
#include <math_constants.h>

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

// ---------------------------------------------------------------- split-KV merge
// One CTA per (sequence b, kv head g, chunk of RB query rows); the rows of
// (b, g) are its G*T query rows (the q heads that read kv head g, times the
// query tokens).  Partition i of a row holds O_i (normalised), m_i (reference
// max, log2 domain) and l_i (sum of 2^(s - m_i)); the merged row is
// sum_i w_i O_i / sum_i w_i with w_i = l_i 2^(m_i - M), M = max_i m_i.
// Phase 1 loads every (row, partition) statistic of the CTA at once and turns
// it into a weight; phase 2 gives each thread 4 head dims of one row and sums
// the partial rows with independent 16-byte loads.  Sequences that fit in one
// partition were written by the attention kernel directly and are skipped
// (same predicate).
constexpr int kMergeThreads = 128;
constexpr int kMergeMaxWeights = kMaxPartitions;   // rows x partitions per pass

template <int D>
__global__ void __launch_bounds__(kMergeThreads) splitkv_reduce_kernel(const AttnParams p) {
  constexpr int C4 = D / 4;                   // float4 chunks per row
  constexpr int RB = kMergeThreads / C4;      // rows per CTA: 4 (D 128) or 8 (D 64)
  __shared__ float s_w[kMergeMaxWeights];
  __shared__ float s_inv[RB];
  const int rows = p.G * p.T;
  const int chunks = (rows + RB - 1) / RB;
  const int bg = blockIdx.x / chunks;
  const int r0 = (blockIdx.x % chunks) * RB;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int L = p.context_lens[b];
  if (L < p.T || L > p.max_ctx) return;
  const int pre = (p.seq_group != nullptr && p.seq_group[b] >= 0)
                      ? p.group_prefix_blocks[p.seq_group[b]] : 0;
  if (pre < 0 || pre > p.max_prefix_blocks || pre * kBlockSize > L) return;
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  const int npre = (pre + p.ppb - 1) / p.ppb;
  const int nparts = npre + (nblk - pre + p.ppb - 1) / p.ppb;
  if (pre == 0 && nparts == 1) return;
  const int nr = min(RB, rows - r0);
  // row r = t * G + hl  ->  orow = (b*T + t)*Hq + g*G + hl
  auto orow_of = [&](int r) {
    return (static_cast<size_t>(b) * p.T + r / p.G) * p.Hq + g * p.G + r % p.G;
  };
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kMergeThreads / 32;
  const int per_pass = max(1, min(nr, kMergeMaxWeights / nparts));
  for (int q0 = 0; q0 < nr; q0 += per_pass) {
    const int nq = min(per_pass, nr - q0);
    __syncthreads();
    // phase 1: m_i for every (row, partition) -> row max -> weights
    for (int k = tid; k < nq * nparts; k += kMergeThreads)
      s_w[k] = p.part_m[orow_of(r0 + q0 + k / nparts) * p.max_parts + k % nparts];
    __syncthreads();
    for (int r = warp; r < nq; r += kWarps) {
      float M = -CUDART_INF_F;
      for (int i = lane; i < nparts; i += 32) M = fmaxf(M, s_w[r * nparts + i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float S = 0.f;
      for (int i = lane; i < nparts; i += 32) {
        const float mi = s_w[r * nparts + i];
        const float w = (mi == -CUDART_INF_F || M == -CUDART_INF_F)
                            ? 0.f
                            : p.part_l[orow_of(r0 + q0 + r) * p.max_parts + i] * exp2f(mi - M);
        s_w[r * nparts + i] = w;
        S += w;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
      if (lane == 0) s_inv[r] = S > 0.f ? 1.f / S : 0.f;
    }
    __syncthreads();
    // phase 2: O = sum_i w_i O_i / S, 4 head dims per thread
    const int r = tid / C4, c = tid % C4;
    if (r < nq) {
      const size_t orow = orow_of(r0 + q0 + r);
      const float4* po = reinterpret_cast<const float4*>(p.part_o + orow * p.max_parts * D) + c;
      const float* w = s_w + r * nparts;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
      for (int i = 0; i < nparts; ++i) {
        const float4 x = po[static_cast<size_t>(i) * C4];
        acc.x += w[i] * x.x;
        acc.y += w[i] * x.y;
        acc.z += w[i] * x.z;
        acc.w += w[i] * x.w;
      }
      const float inv = s_inv[r];
      __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(p.out) + (orow * D + 4 * c) / 2;
      dst[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      dst[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    }
  }
}

cudaError_t launch_reduce(const AttnParams& p, int head_dim, cudaStream_t s) {
  const int rb = kMergeThreads / (head_dim / 4);
  const long long chunks = (static_cast<long long>(p.G) * p.T + rb - 1) / rb;
  const long long ctas = static_cast<long long>(p.num_seqs) * p.Hkv * chunks;
  if (ctas == 0) return cudaSuccess;
  if (head_dim == 64)
    splitkv_reduce_kernel<64><<<static_cast<unsigned>(ctas), kMergeThreads, 0, s>>>(p);
  else
    splitkv_reduce_kernel<128><<<static_cast<unsigned>(ctas), kMergeThreads, 0, s>>>(p);
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
