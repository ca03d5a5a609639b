// Speculative-decoding acceptance: which draft tokens the target keeps, and the
// one token the target emits after them ("ranksignal" post, Spéculer : plusieurs
// tokens par passe; "LLM inference optimization: KV cache", §5.2 and §5.3).
//
// One CTA per sequence.  Greedy: the first position whose draft differs from the
// target's most probable token (lowest index on ties) stops the run and emits
// that token; after K kept drafts the bonus position K emits its most probable
// token.  Sampling: draft x_i is kept iff q_i(x_i) * a_i < p_i(x_i) * 2^24 (a_i a
// 24-bit uniform; exact in fp64), and the emitted token is an inverse-CDF draw
// with one 32-bit uniform s over the weights w(x) = floor(r(x) * 2^40), r =
// max(0, p_i - q_i) in float32 at the rejected position i (r = p_K after K kept
// drafts): the smallest x whose prefix sum of w exceeds floor(s * W / 2^32), W
// the sum of all w.  The weights are integers, so the draw does not depend on
// the order of summation.  If W is 0 the most probable token is emitted.
//
// The draw reads the row once, each warp summing the weights of its tiles of
// 128 elements (tile sums kept in shared memory), finds the tile that holds the
// target prefix with a block scan over the tile sums, then re-reads that one
// tile (from L2) and finds the element with a warp scan.
#include <math_constants.h>
#include <stdint.h>

#include "pa_ptx.cuh"

namespace pa {

constexpr int kSpecThreads = 512;
constexpr int kSpecWarps = kSpecThreads / 32;
constexpr int kTileW = 128;                                 // elements per warp tile (32 x 4)
constexpr int kMaxTiles = kMaxSpecVocab / kTileW;
constexpr int kTilesPerThread = kMaxTiles / kSpecThreads;   // tile sums one thread scans
static_assert(kMaxTiles % kSpecThreads == 0, "tile sums split evenly over the threads");

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

// Most probable index of row[0, V) (lowest index among equal maxima); all threads
// of the block get the result.
__device__ int block_argmax(const float* __restrict__ row, int V, ArgMax* red) {
  ArgMax m{-CUDART_INF_F, 0x7fffffff};
#pragma unroll 4
  for (int x = threadIdx.x; x < V; x += kSpecThreads) m = better(m, ArgMax{__ldg(row + x), x});
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgMax other{__shfl_xor_sync(0xffffffffu, m.v, o), __shfl_xor_sync(0xffffffffu, m.i, o)};
    m = better(m, other);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < kSpecWarps ? red[lane] : ArgMax{-CUDART_INF_F, 0x7fffffff};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ArgMax other{__shfl_xor_sync(0xffffffffu, m.v, o), __shfl_xor_sync(0xffffffffu, m.i, o)};
      m = better(m, other);
    }
    if (lane == 0) red[0] = m;
  }
  __syncthreads();
  const int r = red[0].i;
  __syncthreads();
  return r == 0x7fffffff ? 0 : r;
}

// Weights of this lane's 4 consecutive elements of warp tile t: residual max(0, p - q)
// or p alone.
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
// Returns -1 when every weight is 0.
__device__ int integer_draw(const float* __restrict__ p, const float* __restrict__ q, int V,
                            uint32_t s, unsigned long long* tile_sum,
                            unsigned long long* wsum, int* s_pick) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = (V + kTileW - 1) / kTileW;
  // pass 1: warp w sums the weights of tiles w, w + 16, ...
#pragma unroll 4
  for (int t = warp; t < tiles; t += kSpecWarps) {
    unsigned long long w[4];
    tile_weights(p, q, V, t, w);
    unsigned long long v = w[0] + w[1] + w[2] + w[3];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) tile_sum[t] = v;
  }
  __syncthreads();
  // block scan over the tile sums: thread j holds tiles [j * kTilesPerThread, ...)
  unsigned long long mine = 0;
#pragma unroll
  for (int k = 0; k < kTilesPerThread; ++k) {
    const int t = threadIdx.x * kTilesPerThread + k;
    if (t < tiles) mine += tile_sum[t];
  }
  const unsigned long long incl = warp_inclusive_sum(mine);
  if (lane == 31) wsum[warp] = incl;
  if (threadIdx.x == 0) s_pick[0] = -1;
  __syncthreads();
  unsigned long long before = incl - mine, total = 0;
  for (int k = 0; k < kSpecWarps; ++k) {
    if (k < warp) before += wsum[k];
    total += wsum[k];
  }
  if (total > 0) {
    // floor(s * total / 2^32) without overflow: total < 2^60, s < 2^32
    const unsigned long long lo = static_cast<unsigned long long>(s) * (total & 0xFFFFFFFFull);
    const unsigned long long hi = static_cast<unsigned long long>(s) * (total >> 32);
    const unsigned long long target = hi + (lo >> 32);
    if (before <= target && target < before + mine) {
      unsigned long long run = before;
      for (int k = 0; k < kTilesPerThread; ++k) {
        const int t = threadIdx.x * kTilesPerThread + k;
        const unsigned long long ts = t < tiles ? tile_sum[t] : 0ull;
        if (target < run + ts) {
          s_pick[0] = t;
          s_pick[1] = -1;
          wsum[kSpecWarps] = target - run;      // rank inside the picked tile
          break;
        }
        run += ts;
      }
    }
  }
  __syncthreads();
  const int pick_tile = s_pick[0];
  if (pick_tile < 0) return -1;
  // pass 2: warp 0 finds the element of the picked tile whose prefix exceeds the rank
  if (warp == 0) {
    const unsigned long long rank = wsum[kSpecWarps];
    unsigned long long w[4];
    tile_weights(p, q, V, pick_tile, w);
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
      s_pick[1] = pick_tile * kTileW + lane * 4 + hit;
    }
  }
  __syncthreads();
  return s_pick[1];
}

template <bool GREEDY>
__global__ void __launch_bounds__(kSpecThreads)
    spec_accept_kernel(const float* __restrict__ p, const float* __restrict__ q,
                       const int32_t* __restrict__ drafts, const uint32_t* __restrict__ a24,
                       const uint32_t* __restrict__ s32, int K, int V,
                       int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_kept) {
  __shared__ unsigned long long tile_sum[kMaxTiles];
  __shared__ unsigned long long wsum[kSpecWarps + 1];
  __shared__ ArgMax red[kSpecWarps];
  __shared__ int s_pick[2];
  __shared__ int s_stop;
  const int b = blockIdx.x;
  const float* pb = p + static_cast<size_t>(b) * (K + 1) * V;
  const float* qb = GREEDY ? nullptr : q + static_cast<size_t>(b) * K * V;
  const int32_t* db = drafts + static_cast<size_t>(b) * K;

  int stop = K;
  int final_tok = -1;
  if constexpr (GREEDY) {
    for (int i = 0; i < K; ++i) {
      const int best = block_argmax(pb + static_cast<size_t>(i) * V, V, red);
      const int x = db[i];
      if (static_cast<unsigned>(x) >= static_cast<unsigned>(V) && threadIdx.x == 0)
        atomicOr(&g_pa_err, kErrBounds);
      if (x != best) {
        stop = i;
        final_tok = best;
        break;
      }
    }
    if (stop == K) final_tok = block_argmax(pb + static_cast<size_t>(K) * V, V, red);
  } else {
    if (threadIdx.x == 0) {
      int i = 0;
      for (; i < K; ++i) {
        const int x = db[i];
        if (static_cast<unsigned>(x) >= static_cast<unsigned>(V)) {
          atomicOr(&g_pa_err, kErrBounds);
          break;                              // an impossible draft is not kept
        }
        const double px = static_cast<double>(__ldg(pb + static_cast<size_t>(i) * V + x));
        const double qx = static_cast<double>(__ldg(qb + static_cast<size_t>(i) * V + x));
        if (!(qx * static_cast<double>(a24[static_cast<size_t>(b) * K + i] & 0xFFFFFFu) <
              px * 16777216.0))
          break;
      }
      s_stop = i;
    }
    __syncthreads();
    stop = s_stop;
    const float* prow = pb + static_cast<size_t>(stop) * V;
    const float* qrow = stop < K ? qb + static_cast<size_t>(stop) * V : nullptr;
    final_tok = integer_draw(prow, qrow, V, s32[b], tile_sum, wsum, s_pick);
    if (final_tok < 0) final_tok = block_argmax(prow, V, red);
  }
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
  if (greedy)
    spec_accept_kernel<true><<<num_seqs, kSpecThreads, 0, s>>>(p, q, drafts, a24, s32, K, V,
                                                               out_tokens, out_kept);
  else
    spec_accept_kernel<false><<<num_seqs, kSpecThreads, 0, s>>>(p, q, drafts, a24, s32, K, V,
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
