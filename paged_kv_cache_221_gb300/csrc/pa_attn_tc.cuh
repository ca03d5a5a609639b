// Paged multi-query attention on the fifth-generation tensor cores (tcgen05),
// for the speculative-verify tile: up to 32 query rows per kv head (the GQA
// group x the draft tokens) attending over one sequence's pages.
//
// One CTA owns one work unit (partition of one sequence's pages, kv head), as
// in the mma.sync kernel, and streams its pages through the block table with
// TMA.  Eight 16-token pages form one group of 128 tokens, the M dimension of
// the score MMA:
//
//   S^T[128 tokens x 32 rows] = K[128 tokens x D] . Q^T[D x 32 rows]     (TMEM)
//   O^T[D x 32 rows]         += V^T[D x 16 tokens] . P^T[16 tokens x 32 rows]
//                               per page, P as a bf16 high part and a bf16
//                               residual (two MMAs), so P keeps ~16 bits
//
// Both accumulators live in tensor memory.  Roles (192 threads):
//   warps 0-3  softmax: thread i owns TMEM lane i, i.e. token i of the group
//              (scores) and head dim i (output).  Per group: load the scores,
//              mask, keep a per-row reference max that only moves when a score
//              exceeds it by 8 (log2 units; then O is rescaled in TMEM), write
//              P^T to shared memory, accumulate per-thread row sums.
//   warp 4     producer: block-table lookup and TMA loads of K and V pages
//              into a ring of kGroups groups (128-byte swizzle).
//   warp 5     TMEM allocation; lane 0 issues every MMA and commits them to
//              mbarriers.
// The K ring is laid out [head-dim half][ring page][16 tokens][128 B] so that
// the 128 tokens of a group are one K-major operand with a uniform stride; V
// is [ring page][half][16 tokens][128 B], one MN-major operand per page.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include <atomic>

#include "pa_ptx.cuh"
#include "pa_tc.cuh"

namespace pa {

struct TcGeo {
  static constexpr int D = 128;
  static constexpr int kGroupPages = 8;                  // pages per score MMA (M = 128)
  static constexpr int kGroups = 2;                      // ring groups
  static constexpr int kSlots = kGroups * kGroupPages;   // ring pages
  static constexpr int kRows = 32;                       // N of both MMAs
  static constexpr int kHalfBytes = kBlockSize * 128;    // 16 tokens x 64 dims bf16
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int kKOff = 0;                                        // [2][kSlots][2048]
  static constexpr int kVOff = kKOff + 2 * kSlots * kHalfBytes;          // [kSlots][2][2048]
  static constexpr int kQOff = kVOff + 2 * kSlots * kHalfBytes;          // [2][32][128]
  static constexpr int kPOff = kQOff + 2 * kRows * 128;                  // [2 buf][2 hi/lo][2][32][128]
  static constexpr int kPBytes = 2 * kRows * 128;                        // one (buf, hi/lo) operand
  static constexpr int kMiscOff = kPOff + 4 * kPBytes;
  static constexpr int kAlloc = kMiscOff + 2048 + 1024;
  static constexpr uint32_t kTmemCols = 128;   // S buffers at 0 and 32, O at 64
};

// Small shared state (barriers, flags, reduction buffers).
struct TcMisc {
  uint64_t kv_full[TcGeo::kGroups];
  uint64_t kv_empty[TcGeo::kGroups];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t p_empty[2];                       // completes after the P.V of group h (buffer h & 1)
  uint64_t fin;
  uint32_t tmem_base;
  int stage_ok[TcGeo::kSlots];
  int lim[TcGeo::kRows];
  int flag[2][4];
  float red[4][TcGeo::kRows];
};
static_assert(sizeof(TcMisc) <= 2048, "misc area");

__device__ __forceinline__ uint32_t tc_sw128(int row, int byte_in_row) {
  // byte offset inside a 128-byte-swizzled block of rows of 128 bytes
  return static_cast<uint32_t>(row * 128 + ((((byte_in_row >> 4) ^ (row & 7)) << 4) |
                                            (byte_in_row & 15)));
}

__global__ void __launch_bounds__(192, 1)
    paged_attn_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
  using Gm = TcGeo;
  constexpr int D = Gm::D;
  constexpr int NR = Gm::kRows;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  TcMisc& ms = *reinterpret_cast<TcMisc*>(smem + Gm::kMiscOff);

  grid_launch_dependents();
  if (blockIdx.x == gridDim.x - 1) grid_dependency_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ------------------------------------------------------------------ unit
  const int unit_p = static_cast<int>(blockIdx.x / (p.Hkv * p.num_seqs));
  const int g = static_cast<int>(blockIdx.x % p.Hkv);
  const int b = static_cast<int>((blockIdx.x / p.Hkv) % p.num_seqs);
  const int G = p.G, T = p.T;
  const int L = p.context_lens[b];
  const int pre = (p.seq_group != nullptr && p.seq_group[b] >= 0)
                      ? p.group_prefix_blocks[p.seq_group[b]] : 0;
  if (L < T || L > p.max_ctx || pre < 0 || pre > p.max_prefix_blocks || pre * kBlockSize > L) {
    if (threadIdx.x == 0 && unit_p == 0) atomicOr(&g_pa_err, kErrBounds);
    return;
  }
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  const int first = p.window > 0 ? max(pre, max(0, L - T - p.window + 1) / kBlockSize) : pre;
  const int pg0 = first + unit_p * p.ppb;
  if (pg0 >= nblk) return;                   // partition past this sequence's end
  const int pg1 = min(pg0 + p.ppb, nblk);
  const int npre = (pre + p.ppb - 1) / p.ppb;
  const int nparts = npre + (nblk - first + p.ppb - 1) / p.ppb;
  const int slot = npre + unit_p;
  const bool direct = (pre == 0 && nparts == 1);
  const int nrows = G * T;
  const int npages = pg1 - pg0;
  const int ngroups = (npages + Gm::kGroupPages - 1) / Gm::kGroupPages;
  const int32_t* trow = p.block_tables + static_cast<size_t>(b) * p.mbs;

  const uint32_t kring = smem_u32(smem + Gm::kKOff);
  const uint32_t vring = smem_u32(smem + Gm::kVOff);
  const uint32_t qsm = smem_u32(smem + Gm::kQOff);
  const uint32_t psm = smem_u32(smem + Gm::kPOff);

  // ------------------------------------------------------------------ setup
  if (threadIdx.x == 0) {
    for (int i = 0; i < Gm::kGroups; ++i) {
      mbar_init(&ms.kv_full[i], 1);
      mbar_init(&ms.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms.s_full[i], 1);
      mbar_init(&ms.s_free[i], 4);
      mbar_init(&ms.p_full[i], 4);
      mbar_init(&ms.p_empty[i], 1);
    }
    mbar_init(&ms.fin, 1);
    fence_barrier_init();
  }
  if (warp == 5) tc::tmem_alloc(&ms.tmem_base, Gm::kTmemCols);
  if (warp < 4) {
    // Q rows (zero rows pad to 32), K-major with the 128-byte swizzle:
    // [dim half][row][128 B]
    constexpr int CH = D / 8;
    for (int idx = threadIdx.x; idx < NR * CH; idx += 128) {
      const int n = idx / CH, ch = idx % CH;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (n < nrows) {
        const int t = n / G, hl = n % G;
        const size_t row = (static_cast<size_t>(b) * T + t) * p.Hq + g * G + hl;
        v = reinterpret_cast<const uint4*>(p.q)[row * CH + ch];
      }
      *reinterpret_cast<uint4*>(smem + Gm::kQOff + (ch >> 3) * (NR * 128) +
                                tc_sw128(n, (ch & 7) * 16)) = v;
    }
    // P operands start at zero (rows >= nrows stay zero)
    for (int idx = threadIdx.x; idx < 4 * Gm::kPBytes / 16; idx += 128)
      reinterpret_cast<uint4*>(smem + Gm::kPOff)[idx] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x < NR)
      ms.lim[threadIdx.x] = threadIdx.x < nrows ? L - T + static_cast<int>(threadIdx.x) / G : -1;
    tc::fence_proxy_async_smem();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ms.tmem_base;
  const uint32_t tmem_o = tmem + 64;

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    // Query tokens' K/V that land in this unit's pages are stored first
    // (reshape_and_cache fused), then made visible to the TMA reads.
    if (p.new_k != nullptr) {
      const int jlo = max(0, (L - T) / kBlockSize - pg0);
      const int jhi = min(npages - 1, (L - 1) / kBlockSize - pg0);
      for (int j = jlo; j <= jhi; ++j) {
        const int phys = __ldg(trow + pg0 + j);
        if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) continue;
        const int pos0 = (pg0 + j) * kBlockSize;
        const int lo = max(L - T, pos0), hi = min(L - 1, pos0 + kBlockSize - 1);
        for (int pos = lo; pos <= hi; ++pos) {
          const size_t src = (static_cast<size_t>(b) * T + (pos - (L - T))) * p.Hkv + g;
          const size_t dst = (static_cast<size_t>(phys) * p.Hkv + g) * kBlockSize +
                             (pos & (kBlockSize - 1));
          constexpr int CH = D / 8;
          for (int c = lane; c < 2 * CH; c += 32) {
            const bool isv = c >= CH;
            const int cc = isv ? c - CH : c;
            const uint4 v =
                reinterpret_cast<const uint4*>(isv ? p.new_v : p.new_k)[src * CH + cc];
            reinterpret_cast<uint4*>(isv ? p.v_pool : p.k_pool)[dst * CH + cc] = v;
          }
        }
      }
      fence_proxy_async_global();
      __syncwarp();
    }
    if (lane == 0) {
      tma_prefetch_map(&tmk);
      tma_prefetch_map(&tmv);
    }
    bool aborted = false;
    for (int grp = 0; grp < ngroups; ++grp) {
      const int rb = grp % Gm::kGroups;
      const uint32_t use = static_cast<uint32_t>(grp / Gm::kGroups);
      if (!aborted && !mbar_wait(&ms.kv_empty[rb], (use & 1u) ^ 1u, p.timeout_ns)) aborted = true;
      aborted = __any_sync(0xffffffffu, aborted);
      const int pi = grp * Gm::kGroupPages + lane;
      const bool in = lane < Gm::kGroupPages && pi < npages;
      const int phys = in ? __ldg(trow + pg0 + pi) : 0;
      const bool ok = in && !aborted &&
                      static_cast<unsigned>(phys) < static_cast<unsigned>(p.num_blocks);
      if (in && static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks))
        atomicOr(&g_pa_err, kErrBounds);
      const int sl = rb * Gm::kGroupPages + lane;
      if (lane < Gm::kGroupPages) ms.stage_ok[sl] = ok ? 1 : 0;
      const unsigned okm = __ballot_sync(0xffffffffu, ok);
      __syncwarp();
      if (lane == 0)
        mbar_arrive_expect_tx(&ms.kv_full[rb],
                              static_cast<uint32_t>(__popc(okm)) * 4u * Gm::kHalfBytes);
      __syncwarp();
      if (ok) {
        const int row = (phys * p.Hkv + g) * kBlockSize;
        uint8_t* kd = smem + Gm::kKOff + sl * Gm::kHalfBytes;
        uint8_t* vd = smem + Gm::kVOff + sl * 2 * Gm::kHalfBytes;
        tma_load_2d(kd, &tmk, &ms.kv_full[rb], 0, row);
        tma_load_2d(kd + Gm::kSlots * Gm::kHalfBytes, &tmk, &ms.kv_full[rb], 64, row);
        tma_load_2d(vd, &tmv, &ms.kv_full[rb], 0, row);
        tma_load_2d(vd + Gm::kHalfBytes, &tmv, &ms.kv_full[rb], 64, row);
      }
    }
    // Do not leave while copies issued by this warp may still be landing.
    if (lane == 0) {
      for (int grp = max(0, ngroups - Gm::kGroups); grp < ngroups; ++grp)
        mbar_wait(&ms.kv_full[grp % Gm::kGroups],
                  static_cast<uint32_t>(grp / Gm::kGroups) & 1u, p.timeout_ns);
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdQK = tc::idesc_f16<128, NR, false, false, true>();
      constexpr uint32_t kIdPV = tc::idesc_f16<128, NR, true, false, true>();
      bool aborted = false;
      uint32_t any_pv = 0;
      auto issue_pv = [&](int h) {
        const int pb = h & 1;
        const int rb = h % Gm::kGroups;
        if (!aborted && !mbar_wait(&ms.p_full[pb], static_cast<uint32_t>(h >> 1) & 1u,
                                   p.timeout_ns))
          aborted = true;
        tc::fence_after_sync();
        if (!aborted) {
          for (int j = 0; j < Gm::kGroupPages; ++j) {
            const int sl = rb * Gm::kGroupPages + j;
            if (h * Gm::kGroupPages + j >= npages || !ms.stage_ok[sl]) continue;
            // A = V^T (MN-major): dims 64..127 one 2048-byte half further, tokens
            // 8..15 one 1024-byte atom further
            const uint64_t ad = tc::smem_desc(vring + sl * 2 * Gm::kHalfBytes, Gm::kHalfBytes,
                                              1024);
            // B = P^T stored as P[row][token] (K-major): this page's 16 tokens
            const uint32_t pbase = psm + (pb * 2) * Gm::kPBytes + (j >> 2) * (NR * 128) +
                                   (j & 3) * 32;
            tc::mma_f16_ss(tmem_o, ad, tc::smem_desc(pbase, 16, 1024), kIdPV, any_pv);
            tc::mma_f16_ss(tmem_o, ad, tc::smem_desc(pbase + Gm::kPBytes, 16, 1024), kIdPV, 1u);
            any_pv = 1u;
          }
          tc::commit(&ms.kv_empty[rb]);
          tc::commit(&ms.p_empty[pb]);
        } else {
          mbar_arrive(&ms.kv_empty[rb]);
          mbar_arrive(&ms.p_empty[pb]);
        }
      };
      for (int grp = 0; grp < ngroups; ++grp) {
        const int rb = grp % Gm::kGroups;
        const int sb = grp & 1;
        if (!aborted && !mbar_wait(&ms.kv_full[rb], static_cast<uint32_t>(grp / Gm::kGroups) & 1u,
                                   p.timeout_ns))
          aborted = true;
        if (!aborted && !mbar_wait(&ms.s_free[sb], (static_cast<uint32_t>(grp >> 1) & 1u) ^ 1u,
                                   p.timeout_ns))
          aborted = true;
        tc::fence_after_sync();
        if (!aborted) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = kring + (kk >> 2) * (Gm::kSlots * Gm::kHalfBytes) +
                                rb * Gm::kGroupPages * Gm::kHalfBytes + (kk & 3) * 32;
            const uint32_t qa = qsm + (kk >> 2) * (NR * 128) + (kk & 3) * 32;
            tc::mma_f16_ss(tmem + sb * NR, tc::smem_desc(ka, 16, 1024),
                           tc::smem_desc(qa, 16, 1024), kIdQK, kk > 0 ? 1u : 0u);
          }
          tc::commit(&ms.s_full[sb]);
        } else {
          mbar_arrive(&ms.s_full[sb]);
        }
        if (grp > 0) issue_pv(grp - 1);
      }
      if (ngroups > 0) issue_pv(ngroups - 1);
      // every MMA of this unit has completed before the CTA may release TMEM
      tc::commit(&ms.fin);
      mbar_wait(&ms.fin, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax
    const int t = threadIdx.x;                 // TMEM lane: token of the group, head dim
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    float m[NR], lp[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      m[r] = -CUDART_INF_F;
      lp[r] = 0.f;
    }
    int lim[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) lim[r] = ms.lim[r];
    bool aborted = false;
    bool pv_before = false;                    // a valid page was in an earlier group
    const int tail_tok = L - (pg0 + npages - 1) * kBlockSize;   // valid tokens of the last page
    for (int grp = 0; grp < ngroups; ++grp) {
      const int rb = grp % Gm::kGroups;
      const int sb = grp & 1;
      if (!aborted && !mbar_wait(&ms.kv_full[rb], static_cast<uint32_t>(grp / Gm::kGroups) & 1u,
                                 p.timeout_ns))
        aborted = true;
      if (!aborted && !mbar_wait(&ms.s_full[sb], static_cast<uint32_t>(grp >> 1) & 1u,
                                 p.timeout_ns))
        aborted = true;
      aborted = __any_sync(0xffffffffu, aborted);
      tc::fence_after_sync();
      uint32_t sr[32];
      tc::tmem_ld32(tmem + lane_addr + sb * NR, sr);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms.s_free[sb]);

      const int pidx = grp * Gm::kGroupPages + (t >> 4);
      const int sl = rb * Gm::kGroupPages + (t >> 4);
      const bool valid = !aborted && pidx < npages && ms.stage_ok[sl] != 0;
      const int j = (pg0 + pidx) * kBlockSize + (t & 15);
      float x[NR];
      bool exceed = false;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const bool vis = valid && r < nrows &&
                         static_cast<unsigned>(lim[r] - j) < p.wcap;
        x[r] = vis ? __uint_as_float(sr[r]) * sl2 : -CUDART_INF_F;
        exceed |= x[r] > m[r] + 8.f;
      }
      // group-wide decision on moving the reference maxima
      const bool wexceed = __any_sync(0xffffffffu, exceed);
      if (lane == 0) ms.flag[sb][warp] = wexceed ? 1 : 0;
      named_bar_sync(1, 128);
      const bool any = (ms.flag[sb][0] | ms.flag[sb][1] | ms.flag[sb][2] | ms.flag[sb][3]) != 0;
      if (any) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          float v = x[r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
          if (lane == 0) ms.red[warp][r] = v;
        }
        named_bar_sync(1, 128);
        float alpha[NR];
        bool need_o = false;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float mx = fmaxf(fmaxf(ms.red[0][r], ms.red[1][r]),
                                 fmaxf(ms.red[2][r], ms.red[3][r]));
          alpha[r] = 1.f;
          if (mx > m[r] + 8.f) {
            if (m[r] != -CUDART_INF_F) {
              alpha[r] = hw_exp2(m[r] - mx);
              need_o = true;
            } else {
              alpha[r] = 0.f;
            }
            m[r] = mx;
          }
          lp[r] *= alpha[r];
        }
        named_bar_sync(1, 128);                // red[] may be rewritten next group
        if (need_o && pv_before && !aborted) {
          // O holds the pages of earlier groups: wait for their P.V (group grp - 1,
          // whose buffer's previous P.V, of group grp - 3, this thread already
          // waited for), then rescale in TMEM
          if (!mbar_wait(&ms.p_empty[(grp - 1) & 1], static_cast<uint32_t>((grp - 1) >> 1) & 1u,
                         p.timeout_ns))
            aborted = true;
          aborted = __any_sync(0xffffffffu, aborted);
          tc::fence_after_sync();
          uint32_t orr[32];
          tc::tmem_ld32(tmem_o + lane_addr, orr);
          tc::tmem_wait_ld();
#pragma unroll
          for (int r = 0; r < NR; ++r) orr[r] = __float_as_uint(__uint_as_float(orr[r]) * alpha[r]);
          tc::tmem_st32(tmem_o + lane_addr, orr);
          tc::tmem_wait_st();
        }
      }
      // P^T for this group: bf16 high part and residual, [row][token] swizzled
      const int pb = grp & 1;
      if (!aborted && !mbar_wait(&ms.p_empty[pb], (static_cast<uint32_t>(grp >> 1) & 1u) ^ 1u,
                                 p.timeout_ns))
        aborted = true;
      uint8_t* ph = smem + Gm::kPOff + (pb * 2) * Gm::kPBytes + (t >> 6) * (NR * 128);
      uint8_t* plo = ph + Gm::kPBytes;
      const int tb = (t & 63) * 2;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (r >= nrows) break;
        const float mr = m[r] == -CUDART_INF_F ? 0.f : m[r];
        const float pr = hw_exp2(x[r] - mr);
        lp[r] += pr;
        const __nv_bfloat16 h = __float2bfloat16_rn(pr);
        const __nv_bfloat16 lo = __float2bfloat16_rn(pr - __bfloat162float(h));
        const uint32_t off = tc_sw128(r, tb);
        *reinterpret_cast<__nv_bfloat16*>(ph + off) = h;
        *reinterpret_cast<__nv_bfloat16*>(plo + off) = lo;
      }
      // V rows past the context end in the last page may hold anything (even
      // NaN); their weight is 0, but 0 * NaN is NaN: zero them before the P.V.
      if (pidx == npages - 1 && (t & 15) >= tail_tok && ms.stage_ok[sl] != 0) {
        uint4* vrow = reinterpret_cast<uint4*>(smem + Gm::kVOff + sl * 2 * Gm::kHalfBytes +
                                               (t & 15) * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          vrow[c] = make_uint4(0, 0, 0, 0);
          vrow[c + Gm::kHalfBytes / 16] = make_uint4(0, 0, 0, 0);
        }
      }
      // the MMA thread issues P.V for every page of the group that is in the unit
      // and was loaded: from the next group on, O holds data
#pragma unroll
      for (int jj = 0; jj < Gm::kGroupPages; ++jj)
        pv_before |= grp * Gm::kGroupPages + jj < npages &&
                     ms.stage_ok[rb * Gm::kGroupPages + jj] != 0;
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms.p_full[pb]);
    }

    // ---------------------------------------------------------------- epilogue
    // the last group's P.V (the one before it on the same buffer was waited for)
    if (ngroups > 0 && !aborted &&
        !mbar_wait(&ms.p_empty[(ngroups - 1) & 1], static_cast<uint32_t>((ngroups - 1) >> 1) & 1u,
                   p.timeout_ns))
      aborted = true;
    aborted = __any_sync(0xffffffffu, aborted);
    tc::fence_after_sync();
    uint32_t orr[32];
    tc::tmem_ld32(tmem_o + lane_addr, orr);
    tc::tmem_wait_ld();
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      float v = lp[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) ms.red[warp][r] = v;
    }
    named_bar_sync(1, 128);
    const int d = t;                           // head dim of this thread's O^T lane
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      if (r >= nrows) break;
      const float Ls = ms.red[0][r] + ms.red[1][r] + ms.red[2][r] + ms.red[3][r];
      const int tq = r / G, hl = r % G;
      const size_t orow = (static_cast<size_t>(b) * T + tq) * p.Hq + g * G + hl;
      const float o = Ls > 0.f ? __uint_as_float(orr[r]) / Ls : 0.f;
      if (direct) {
        reinterpret_cast<__nv_bfloat16*>(p.out)[orow * D + d] = __float2bfloat16_rn(o);
      } else {
        const size_t pidx2 = orow * p.max_parts + slot;
        p.part_o[pidx2 * D + d] = o;
        if (d == 0) p.part_ml[pidx2] = make_float2(m[r], Ls);
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Gm::kTmemCols);
    tc::tmem_relinquish();
  }
}

inline cudaError_t launch_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                             dim3 grid, cudaStream_t s, bool overlap_previous) {
  constexpr int smem = TcGeo::kAlloc;
  auto kern = paged_attn_tc_kernel;
  static std::atomic<unsigned long long> configured{0ull};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit == 0 || (configured.load(std::memory_order_acquire) & bit) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace pa
