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
// One CTA per query row (b, t, h), one thread per head dim.  Partition i of the
// row holds O_i (normalised), m_i (running max, log2 domain) and l_i (sum of
// 2^(s - m_i)); the merged row is sum_i w_i O_i / sum_i w_i, w_i = l_i 2^(m_i - M),
// M = max_i m_i.  Rows whose sequence fit in one partition were written by the
// attention kernel directly and are skipped here (same predicate).  The
// statistics of up to kChunk partitions are loaded in parallel (one per
// thread) and the partial rows are summed with independent loads in flight.
template <int D>
__global__ void __launch_bounds__(D) splitkv_reduce_kernel(const AttnParams p) {
  constexpr int kChunk = D;
  constexpr int kWarps = D / 32;
  __shared__ float s_w[kChunk];
  __shared__ float s_red[kWarps];
  // Launched as a programmatic dependent of the attention kernel: wait for its
  // completion (and the visibility of its partials) before reading anything.
  grid_dependency_wait();
  const int orow = blockIdx.x;
  const int b = orow / (p.T * p.Hq);
  const int L = p.context_lens[b];
  if (L < p.T || L > p.max_ctx) return;
  const int pre = (p.seq_group != nullptr && p.seq_group[b] >= 0)
                      ? p.group_prefix_blocks[p.seq_group[b]] : 0;
  if (pre < 0 || pre > p.max_prefix_blocks || pre * kBlockSize > L) return;
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  const int npre = (pre + p.ppb - 1) / p.ppb;
  const int nparts = npre + (nblk - pre + p.ppb - 1) / p.ppb;
  if (pre == 0 && nparts == 1) return;
  const float* pm = p.part_m + static_cast<size_t>(orow) * p.max_parts;
  const float* pl = p.part_l + static_cast<size_t>(orow) * p.max_parts;
  const float* po = p.part_o + static_cast<size_t>(orow) * p.max_parts * D;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // M = max_i m_i
  float M = -CUDART_INF_F;
  for (int i = tid; i < nparts; i += D) M = fmaxf(M, pm[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_red[warp] = M;
  __syncthreads();
  M = s_red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_red[w]);

  float S = 0.f, o = 0.f;
  for (int c0 = 0; c0 < nparts; c0 += kChunk) {
    const int n = min(kChunk, nparts - c0);
    __syncthreads();                          // s_w / s_red reuse
    if (tid < n) {
      const float mi = pm[c0 + tid];
      s_w[tid] = (mi == -CUDART_INF_F || M == -CUDART_INF_F) ? 0.f
                                                           : pl[c0 + tid] * exp2f(mi - M);
    }
    __syncthreads();
    const float* pc = po + static_cast<size_t>(c0) * D + tid;
    int i = 0;
    for (; i + 4 <= n; i += 4) {
      const float x0 = pc[(i + 0) * D], x1 = pc[(i + 1) * D];
      const float x2 = pc[(i + 2) * D], x3 = pc[(i + 3) * D];
      o += s_w[i] * x0 + s_w[i + 1] * x1 + s_w[i + 2] * x2 + s_w[i + 3] * x3;
      S += s_w[i] + s_w[i + 1] + s_w[i + 2] + s_w[i + 3];
    }
    for (; i < n; ++i) {
      o += s_w[i] * pc[i * D];
      S += s_w[i];
    }
  }
  reinterpret_cast<__nv_bfloat16*>(p.out)[static_cast<size_t>(orow) * D + tid] =
      __float2bfloat16_rn(S > 0.f ? o / S : 0.f);
}

cudaError_t launch_reduce(const AttnParams& p, int head_dim, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.num_seqs) * p.T * p.Hq;
  if (rows == 0) return cudaSuccess;
  // Programmatic stream serialisation: the launch may overlap the tail of the
  // attention kernel; the kernel's first instruction waits for it to finish.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows), 1, 1);
  cfg.blockDim = dim3(head_dim == 64 ? 64 : 128, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const AttnParams args = p;
  return head_dim == 64 ? cudaLaunchKernelEx(&cfg, splitkv_reduce_kernel<64>, args)
                        : cudaLaunchKernelEx(&cfg, splitkv_reduce_kernel<128>, args);
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
