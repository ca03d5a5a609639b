// Speculative-decoding acceptance: which draft tokens the target keeps, and the
// one token the target emits after them ("ranksignal" post, Spéculer : plusieurs
// tokens par passe; "LLM inference optimization: KV cache", §5.2 and §5.3).
//
// Greedy: the first position whose draft differs from the target's most probable
// token (lowest index on ties) stops the run and emits that token; after K kept
// drafts the bonus position K emits its most probable token.  Sampling: draft
// x_i is kept iff q_i(x_i) * a_i < p_i(x_i) * 2^24 (a_i a 24-bit uniform; exact in
// fp64), and the emitted token is an inverse-CDF draw with one 32-bit uniform s
// over the weights w(x) = floor(r(x) * 2^40), r = max(0, p_i - q_i) in float32 at
// the rejected position i (r = p_K after K kept drafts): the smallest x whose
// prefix sum of w exceeds floor(s * W / 2^32), W the sum of all w.  The weights
// are integers, so the draw does not depend on the order of summation.  If W is
// 0 the most probable token is emitted.
//
// A cluster of kCluster CTAs serves one sequence; CTA r owns a contiguous slice
// of the vocabulary (whole 128-element tiles).  Each CTA decides the kept prefix
// itself (a few scalar loads), sums the weights of its tiles (warps take tiles
// in turn; tile sums stay in shared memory) and publishes its slice total.
// Every CTA then reads the kCluster totals through distributed shared memory
// and finds the slice that holds the target prefix; only that CTA locates the
// tile (block scan over its tile sums) and the element (warp scan over the
// tile, re-read from L2) and writes the sequence's outputs.  The greedy rule
// reduces (value, index) maxima the same way, one position at a time.
#include <cooperative_groups.h>
#include <math_constants.h>
#include <stdint.h>

#include "pa_ptx.cuh"

namespace cg = cooperative_groups;

namespace pa {

constexpr int kCluster = 8;                                 // CTAs per sequence
constexpr int kSpecThreads = 256;
constexpr int kSpecWarps = kSpecThreads / 32;
constexpr int kTileW = 128;                                 // elements per warp tile (32 x 4)
constexpr int kMaxSliceTiles = kMaxSpecVocab / kTileW / kCluster;
constexpr int kTilesPerThread = kMaxSliceTiles / kSpecThreads;
static_assert(kMaxSliceTiles % kSpecThreads == 0, "tile sums split evenly over the threads");

__device__ __forceinline__ unsigned long long weight_of(float r) {
  // r in [0, 1]; r * 2^40 is exact; truncation is the floor for r >= 0
  return __float2ull_rz(r * 1099511627776.0f);
}

struct ArgMax {
  float v;
  int i;
};

__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}

struct SpecShared {
  unsigned long long tile_sum[kMaxSliceTiles];
  unsigned long long wsum[kSpecWarps + 1];
  unsigned long long slice_total;       // read by the other CTAs of the cluster
  ArgMax slice_max;                     // read by the other CTAs of the cluster
  ArgMax red[kSpecWarps];
  int pick[2];
  int stop;
};

// Most probable index over this CTA's slice [x0, x1) of row, published in
// sh.slice_max (block-wide; ends with a barrier).
__device__ void slice_argmax(const float* __restrict__ row, int x0, int x1, SpecShared& sh) {
  ArgMax m{-CUDART_INF_F, 0x7fffffff};
#pragma unroll 4
  for (int x = x0 + threadIdx.x; x < x1; x += kSpecThreads)
    m = better(m, ArgMax{__ldg(row + x), x});
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgMax other{__shfl_xor_sync(0xffffffffu, m.v, o), __shfl_xor_sync(0xffffffffu, m.i, o)};
    m = better(m, other);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) sh.red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    ArgMax best = sh.red[0];
    for (int k = 1; k < kSpecWarps; ++k) best = better(best, sh.red[k]);
    sh.slice_max = best;
  }
  __syncthreads();
}

// The cluster-wide most probable index of row (lowest index on ties).
__device__ int cluster_argmax(const float* __restrict__ row, int x0, int x1, SpecShared& sh,
                              cg::cluster_group& cluster) {
  slice_argmax(row, x0, x1, sh);
  cluster.sync();                                  // every slice maximum is published
  ArgMax best{-CUDART_INF_F, 0x7fffffff};
  for (int r = 0; r < kCluster; ++r) best = better(best, cluster.map_shared_rank(&sh, r)->slice_max);
  cluster.sync();                                  // nobody reuses slice_max before all read it
  return best.i == 0x7fffffff ? 0 : best.i;
}

// Weights of this lane's 4 consecutive elements of tile t: max(0, p - q) or p alone.
__device__ __forceinline__ void tile_weights(const float* __restrict__ p,
                                             const float* __restrict__ q, int V, int t,
                                             unsigned long long (&w)[4]) {
  const int x0 = t * kTileW + (threadIdx.x & 31) * 4;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int x = x0 + e;
    float r = 0.f;
    if (x < V) {
      r = __ldg(p + x);
      if (q != nullptr) r = fmaxf(r - __ldg(q + x), 0.f);
    }
    w[e] = weight_of(r);
  }
}

__device__ __forceinline__ unsigned long long warp_inclusive_sum(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Inverse-CDF draw over the weights of p (q == nullptr) or of max(0, p - q).
// Returns the token on the owning CTA, -1 on the others, and -2 on every CTA
// when all weights are 0.  Tiles [t0, t1) belong to this CTA.
__device__ int cluster_draw(const float* __restrict__ p, const float* __restrict__ q, int V,
                            int t0, int t1, uint32_t s, SpecShared& sh,
                            cg::cluster_group& cluster) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = t1 - t0;
  // pass 1: warp w sums the weights of local tiles w, w + kSpecWarps, ...
#pragma unroll 4
  for (int lt = warp; lt < nt; lt += kSpecWarps) {
    unsigned long long w[4];
    tile_weights(p, q, V, t0 + lt, w);
    unsigned long long v = w[0] + w[1] + w[2] + w[3];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sh.tile_sum[lt] = v;
  }
  __syncthreads();
  // block scan over the local tile sums: thread j holds tiles [j * kTilesPerThread, ...)
  unsigned long long mine = 0;
#pragma unroll
  for (int k = 0; k < kTilesPerThread; ++k) {
    const int lt = threadIdx.x * kTilesPerThread + k;
    if (lt < nt) mine += sh.tile_sum[lt];
  }
  const unsigned long long incl = warp_inclusive_sum(mine);
  if (lane == 31) sh.wsum[warp] = incl;
  __syncthreads();
  unsigned long long before = incl - mine, local_total = 0;
  for (int k = 0; k < kSpecWarps; ++k) {
    if (k < warp) before += sh.wsum[k];
    local_total += sh.wsum[k];
  }
  if (threadIdx.x == 0) sh.slice_total = local_total;
  cluster.sync();                                  // every slice total is published
  unsigned long long total = 0, slice_before = 0;
  const int me = static_cast<int>(cluster.block_rank());
  for (int r = 0; r < kCluster; ++r) {
    const unsigned long long st = cluster.map_shared_rank(&sh, r)->slice_total;
    if (r < me) slice_before += st;
    total += st;
  }
  cluster.sync();                                  // all remote reads done
  if (total == 0) return -2;
  // floor(s * total / 2^32) without overflow: total < 2^60, s < 2^32
  const unsigned long long lo = static_cast<unsigned long long>(s) * (total & 0xFFFFFFFFull);
  const unsigned long long hi = static_cast<unsigned long long>(s) * (total >> 32);
  const unsigned long long target = hi + (lo >> 32);
  if (target < slice_before || target >= slice_before + local_total) return -1;
  const unsigned long long rank_in_slice = target - slice_before;
  if (threadIdx.x == 0) sh.pick[0] = -1;
  __syncthreads();
  if (before <= rank_in_slice && rank_in_slice < before + mine) {
    unsigned long long run = before;
    for (int k = 0; k < kTilesPerThread; ++k) {
      const int lt = threadIdx.x * kTilesPerThread + k;
      const unsigned long long ts = lt < nt ? sh.tile_sum[lt] : 0ull;
      if (rank_in_slice < run + ts) {
        sh.pick[0] = lt;
        sh.wsum[kSpecWarps] = rank_in_slice - run;   // rank inside the picked tile
        break;
      }
      run += ts;
    }
  }
  __syncthreads();
  const int pick = sh.pick[0];
  // pass 2: warp 0 finds the element of the picked tile whose prefix exceeds the rank
  if (warp == 0) {
    const unsigned long long rank = sh.wsum[kSpecWarps];
    unsigned long long w[4];
    tile_weights(p, q, V, t0 + pick, w);
    const unsigned long long own = w[0] + w[1] + w[2] + w[3];
    const unsigned long long in = warp_inclusive_sum(own);
    const unsigned long long ex = in - own;
    if (ex <= rank && rank < in) {
      unsigned long long run = ex;
      int hit = 3;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        run += w[e];
        if (run > rank) {
          hit = e;
          break;
        }
      }
      sh.pick[1] = (t0 + pick) * kTileW + lane * 4 + hit;
    }
  }
  __syncthreads();
  return sh.pick[1];
}

template <bool GREEDY>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kSpecThreads)
    spec_accept_kernel(const float* __restrict__ p, const float* __restrict__ q,
                       const int32_t* __restrict__ drafts, const uint32_t* __restrict__ a24,
                       const uint32_t* __restrict__ s32, int K, int V,
                       int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_kept) {
  __shared__ SpecShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int b = blockIdx.x / kCluster;
  const int me = static_cast<int>(cluster.block_rank());
  // this CTA's slice: whole tiles [t0, t1), elements [x0, x1)
  const int tiles = (V + kTileW - 1) / kTileW;
  const int per = (tiles + kCluster - 1) / kCluster;
  const int t0 = min(tiles, me * per), t1 = min(tiles, t0 + per);
  const int x0 = t0 * kTileW, x1 = min(V, t1 * kTileW);
  const float* pb = p + static_cast<size_t>(b) * (K + 1) * V;
  const float* qb = GREEDY ? nullptr : q + static_cast<size_t>(b) * K * V;
  const int32_t* db = drafts + static_cast<size_t>(b) * K;

  int stop = K;
  int final_tok = -1;
  bool writer = me == 0;
  if constexpr (GREEDY) {
    for (int i = 0; i < K; ++i) {
      const int best = cluster_argmax(pb + static_cast<size_t>(i) * V, x0, x1, sh, cluster);
      const int x = db[i];
      if (static_cast<unsigned>(x) >= static_cast<unsigned>(V) && writer && threadIdx.x == 0)
        atomicOr(&g_pa_err, kErrBounds);
      if (x != best) {
        stop = i;
        final_tok = best;
        break;
      }
    }
    if (stop == K)
      final_tok = cluster_argmax(pb + static_cast<size_t>(K) * V, x0, x1, sh, cluster);
  } else {
    if (threadIdx.x == 0) {
      int i = 0;
      for (; i < K; ++i) {
        const int x = db[i];
        if (static_cast<unsigned>(x) >= static_cast<unsigned>(V)) {
          if (writer) atomicOr(&g_pa_err, kErrBounds);
          break;                              // an impossible draft is not kept
        }
        const double px = static_cast<double>(__ldg(pb + static_cast<size_t>(i) * V + x));
        const double qx = static_cast<double>(__ldg(qb + static_cast<size_t>(i) * V + x));
        if (!(qx * static_cast<double>(a24[static_cast<size_t>(b) * K + i] & 0xFFFFFFu) <
              px * 16777216.0))
          break;
      }
      sh.stop = i;
    }
    __syncthreads();
    stop = sh.stop;
    const float* prow = pb + static_cast<size_t>(stop) * V;
    const float* qrow = stop < K ? qb + static_cast<size_t>(stop) * V : nullptr;
    final_tok = cluster_draw(prow, qrow, V, t0, t1, s32[b], sh, cluster);
    if (final_tok == -2) {
      final_tok = cluster_argmax(prow, x0, x1, sh, cluster);
    } else {
      writer = final_tok >= 0;                // the owning CTA writes the outputs
    }
  }
  if (!writer) return;
  int32_t* ob = out_tokens + static_cast<size_t>(b) * (K + 1);
  for (int i = threadIdx.x; i <= K; i += kSpecThreads)
    ob[i] = i < stop ? db[i] : (i == stop ? final_tok : -1);
  if (threadIdx.x == 0) out_kept[b] = stop;
}

cudaError_t launch_spec_accept(const float* p, const float* q, const int32_t* drafts,
                               const uint32_t* a24, const uint32_t* s32, int num_seqs, int K,
                               int V, bool greedy, int32_t* out_tokens, int32_t* out_kept,
                               cudaStream_t s) {
  if (num_seqs == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(num_seqs) * kCluster;
  if (greedy)
    spec_accept_kernel<true><<<grid, kSpecThreads, 0, s>>>(p, q, drafts, a24, s32, K, V,
                                                           out_tokens, out_kept);
  else
    spec_accept_kernel<false><<<grid, kSpecThreads, 0, s>>>(p, q, drafts, a24, s32, K, V,
                                                            out_tokens, out_kept);
  return cudaGetLastError();
}

cudaError_t take_error_spec(unsigned* bits) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_pa_err, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_pa_err, &zero, sizeof(zero));
  *bits |= v;
  return e;
}

}  // namespace pa
