// Paged multi-query attention on the fifth-generation tensor cores (tcgen05),
// for the speculative-verify tile: up to 32 query rows per kv head (the GQA
// group x the draft tokens) attending over one sequence's pages.
//
// Work units are those of the mma.sync kernel: (partition of one sequence's
// pages, kv head), in partition-major order.  The kernel is persistent: one
// CTA per SM claims units one after another (from a counter in the split-KV
// scratch, so that CTAs that finish early take more, or else every
// gridDim.x-th unit), and its producers stream the next unit's pages while the
// current one finishes, so that no unit pays a pipeline ramp or an epilogue on
// the critical path.
// Pages stream through the block table with TMA.  Eight 16-token pages form
// one group of 128 tokens, the M dimension of the score MMA:
//
//   S^T[128 tokens x 32 row slots] = K[128 tokens x D] . Q^T[D x 32]      (TMEM)
//   O^T[D x 64] += V^T[D x 16 tokens] . [P_hi^T | P_lo^T][16 tokens x 64] per page
//
// P is split into a bf16 high part and a bf16 residual (so it keeps ~16 bits)
// that sit side by side in one B operand: one MMA per page accumulates both
// halves of O^T, which are added at the end.  Both accumulators live in tensor
// memory (O in two buffers, one per unit parity).  Query rows are placed in two
// halves of 16 row slots (rows 0 .. h-1 in slots 0 .. h-1, rows h .. n-1 in
// slots 16 .. 16+n-h-1, h = ceil(n/2)), so that each half of the softmax warps
// carries an equal share.
//
// Roles (352 threads):
//   warps 0-7  softmax: warp w reads TMEM lanes 32 (w % 4) .. +31 (tokens of a
//              group for S, head dims for O) and the 16 row slots of half w / 4.
//              Per group: load the scores, mask (pages wholly visible to every
//              row skip it), keep a per-row reference max that moves only when
//              a score exceeds it by 8 (log2 units; O is then rescaled in TMEM),
//              write P^T (MN-major, 16-byte stores), accumulate row sums.  Per
//              unit: read O, normalise, write the output or the split-KV partial.
//   warp 8     K producer: each unit's query rows into one of two Q buffers,
//              then its K pages, with block-table ids read ahead, by TMA into a
//              ring of kKGroups groups (128-byte swizzle).
//   warp 10    V producer: V pages into a ring of kVGroups groups.  A group's K
//              is free again once its scores are computed, its V once its P.V
//              is, so K runs ahead.
//   warp 9     TMEM allocation; lane 0 issues every MMA, whichever of the next
//              score MMA and the next P.V is ready first, and commits them to
//              mbarriers.
// The K producer claims each unit and passes its index to the other roles
// through a four-entry queue in shared memory; every role then walks the same
// sequence of units and groups and numbers the groups continuously across
// units: ring slots and mbarrier phases follow that running count.  The K ring is laid out [head-dim half][ring page][16 tokens]
// [128 B] so that the 128 tokens of a group are one K-major operand with a
// uniform stride; V is [ring page][half][16 tokens][128 B], one MN-major
// operand per page.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <atomic>

#include "pa_ptx.cuh"
#include "pa_tc.cuh"

namespace pa {

struct TcGeo {
  static constexpr int D = 128;
  static constexpr int kGroupPages = 8;                  // pages per score MMA (M = 128)
  static constexpr int kKGroups = 3;                     // K ring groups
  static constexpr int kVGroups = 3;                     // V ring groups
  static constexpr int kKSlots = kKGroups * kGroupPages; // K ring pages
  static constexpr int kVSlots = kVGroups * kGroupPages; // V ring pages
  static constexpr int kRows = 32;                       // N of the score MMA (row slots)
  static constexpr int kHalfRows = 16;                   // row slots per softmax half
  static constexpr int kSoftmaxWarps = 8;
  static constexpr int kThreads = (kSoftmaxWarps + 3) * 32;
  static constexpr int kHalfBytes = kBlockSize * 128;    // 16 tokens x 64 dims bf16
  // P^T operand, MN-major without swizzle: core matrices of 8 tokens x 8 row
  // slots (8 rows of 16 bytes, one per token); token blocks kPKStride apart,
  // row-slot blocks (hi slots 0-31, then lo slots 0-31) kPNStride apart
  static constexpr int kPKStride = 128;
  static constexpr int kPNStride = (kGroupPages * kBlockSize / 8) * kPKStride;   // 2048
  static constexpr int kPBytes = 2 * kRows / 8 * kPNStride;                     // 16 KB
  static constexpr int kQBytes = 2 * kRows * 128;                               // 8 KB
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int kKOff = 0;                                        // [2][kKSlots][2048]
  static constexpr int kVOff = kKOff + 2 * kKSlots * kHalfBytes;         // [kVSlots][2][2048]
  static constexpr int kQOff = kVOff + 2 * kVSlots * kHalfBytes;         // [2 units][2][32][128]
  static constexpr int kPOff = kQOff + 2 * kQBytes;                      // [16 KB]
  static constexpr int kMiscOff = kPOff + kPBytes;
  static constexpr int kMiscBytes = 1536;
  static constexpr int kAlloc = kMiscOff + kMiscBytes + 1024;
  // TMEM columns: S buffers at 0 and 32, O buffers (per unit parity) at 64 and 128
  static constexpr uint32_t kTmemCols = 256;
};
static_assert(TcGeo::kAlloc <= 232448, "shared memory per block");

// Small shared state (barriers, flags, reduction buffers).
struct TcMisc {
  uint64_t k_full[TcGeo::kKGroups];
  uint64_t k_empty[TcGeo::kKGroups];         // completes after the score MMA of the group
  uint64_t v_full[TcGeo::kVGroups];
  uint64_t v_empty[TcGeo::kVGroups];         // completes after the P.V of the group
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t p_empty;                          // completes after the P.V of each group, in order
  uint64_t q_full[2];                        // per unit parity: query rows staged
  uint64_t q_empty[2];                       // per unit parity: the unit's score MMAs done
  uint64_t o_free[2];                        // per unit parity: the unit's O read out
  uint64_t uq_full[4];                       // queue of claimed units: entry written
  uint64_t uq_empty[4];                      //   entry read by every role
  uint64_t fin;
  uint32_t tmem_base;
  int stage_ok[4][TcGeo::kGroupPages];       // [group % 4][page]: loaded (for the P.V)
  int unit_q[4];                             // claimed unit indices (-1: no more units)
  int flag[2][2][4];                         // [S buffer][half][warp of the half]
  float red[2][4][TcGeo::kHalfRows];
};
static_assert(sizeof(TcMisc) <= TcGeo::kMiscBytes, "misc area");

// One work unit, as every role derives it from the launch parameters.
struct TcUnit {
  int b, g, L, pg0, npages, ngroups, slot;
  bool direct;
};

// Roles that read the queue of claimed units: the V producer, the MMA thread
// (once for its score cursor, once for its P.V cursor) and the softmax warps.
constexpr int kTcQueueReaders = 1 + 2 + TcGeo::kSoftmaxWarps;

// The unit with index u (partition-major: partition, sequence, kv head).  Returns
// false when it has no pages: its partition lies past the sequence's end, or the
// sequence's length or prefix is out of range (*bad is then set).
__device__ __forceinline__ bool tc_unit(const AttnParams& p, int u, TcUnit& un, bool* bad) {
  const int unit_p = u / (p.Hkv * p.num_seqs);
  const int g = u % p.Hkv;
  const int b = (u / p.Hkv) % p.num_seqs;
  const int L = p.context_lens[b];
  const int pre = (p.seq_group != nullptr && p.seq_group[b] >= 0)
                      ? p.group_prefix_blocks[p.seq_group[b]] : 0;
  *bad = false;
  if (L < p.T || L > p.max_ctx || pre < 0 || pre > p.max_prefix_blocks || pre * kBlockSize > L) {
    *bad = unit_p == 0;                      // reported once per (sequence, kv head)
    return false;
  }
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  const int first = p.window > 0 ? max(pre, max(0, L - p.T - p.window + 1) / kBlockSize) : pre;
  const int pg0 = first + unit_p * p.ppb;
  if (pg0 >= nblk) return false;             // partition past this sequence's end
  const int pg1 = min(pg0 + p.ppb, nblk);
  const int npre = (pre + p.ppb - 1) / p.ppb;
  const int nparts = npre + (nblk - first + p.ppb - 1) / p.ppb;
  un.b = b;
  un.g = g;
  un.L = L;
  un.pg0 = pg0;
  un.npages = pg1 - pg0;
  un.ngroups = (un.npages + TcGeo::kGroupPages - 1) / TcGeo::kGroupPages;
  un.slot = npre + unit_p;
  un.direct = pre == 0 && nparts == 1;
  return true;
}

// Next entry c of the queue of claimed units (blocking; one arrival per reader
// on the entry's empty barrier).  False at the end marker.
__device__ __forceinline__ bool tc_queue_next(TcMisc& ms, const AttnParams& p, int& c,
                                              TcUnit& un, bool arrive, bool& aborted) {
  if (!aborted &&
      !mbar_wait(&ms.uq_full[c & 3], static_cast<uint32_t>(c >> 2) & 1u, p.timeout_ns))
    aborted = true;
  const int u = aborted ? -1 : *reinterpret_cast<volatile int*>(&ms.unit_q[c & 3]);
  if (arrive) mbar_arrive(&ms.uq_empty[c & 3]);
  ++c;
  bool bad;
  return u >= 0 && tc_unit(p, u, un, &bad);
}

__device__ __forceinline__ uint32_t tc_sw128(int row, int byte_in_row) {
  // byte offset inside a 128-byte-swizzled block of rows of 128 bytes
  return static_cast<uint32_t>(row * 128 + ((((byte_in_row >> 4) ^ (row & 7)) << 4) |
                                            (byte_in_row & 15)));
}

// Two floats as a bf16x2 word, rounded to nearest even (`lo` in bits 0-15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// NA: row slots per half that can hold a row (even, <= 16): 10 covers up to
// 20 query rows per kv head, 16 up to 32.
template <int NA>
__global__ void __launch_bounds__(TcGeo::kThreads, 1)
    paged_attn_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const AttnParams p,
                         int num_units) {
  using Gm = TcGeo;
  constexpr int D = Gm::D;
  constexpr int NR = Gm::kRows;
  constexpr int NH = Gm::kHalfRows;
  static_assert(NA % 2 == 0 && NA <= NH, "active row slots");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  TcMisc& ms = *reinterpret_cast<TcMisc*>(smem + Gm::kMiscOff);

  grid_launch_dependents();
  if (blockIdx.x == gridDim.x - 1) grid_dependency_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G, T = p.T;
  const int nrows = G * T;
  const int hA = (nrows + 1) / 2;            // rows in the first half of the row slots

  const uint32_t kring = smem_u32(smem + Gm::kKOff);
  const uint32_t vring = smem_u32(smem + Gm::kVOff);
  const uint32_t qsm = smem_u32(smem + Gm::kQOff);
  const uint32_t psm = smem_u32(smem + Gm::kPOff);

  // ------------------------------------------------------------------ setup
  if (threadIdx.x == 0) {
    for (int i = 0; i < Gm::kKGroups; ++i) {
      mbar_init(&ms.k_full[i], 1);
      mbar_init(&ms.k_empty[i], 1);
    }
    for (int i = 0; i < Gm::kVGroups; ++i) {
      mbar_init(&ms.v_full[i], 1);
      mbar_init(&ms.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms.s_full[i], 1);
      mbar_init(&ms.s_free[i], Gm::kSoftmaxWarps);
      mbar_init(&ms.p_full[i], Gm::kSoftmaxWarps);
      mbar_init(&ms.q_full[i], 1);
      mbar_init(&ms.q_empty[i], 1);
      mbar_init(&ms.o_free[i], Gm::kSoftmaxWarps);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&ms.uq_full[i], 1);
      mbar_init(&ms.uq_empty[i], kTcQueueReaders);
    }
    mbar_init(&ms.p_empty, 1);
    mbar_init(&ms.fin, 1);
    fence_barrier_init();
  }
  if (warp == Gm::kSoftmaxWarps + 1) tc::tmem_alloc(&ms.tmem_base, Gm::kTmemCols);
  if (warp < Gm::kSoftmaxWarps) {
    // Q buffers start at zero: row slots that hold no row stay zero
    for (int idx = threadIdx.x; idx < 2 * Gm::kQBytes / 16; idx += Gm::kSoftmaxWarps * 32)
      reinterpret_cast<uint4*>(smem + Gm::kQOff)[idx] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ms.tmem_base;

  if (warp == Gm::kSoftmaxWarps || warp == Gm::kSoftmaxWarps + 2) {
    // ---------------------------------------------------------------- producers
    const bool isv = warp == Gm::kSoftmaxWarps + 2;
    if (lane == 0) tma_prefetch_map(isv ? &tmv : &tmk);
    const int ngr = isv ? Gm::kVGroups : Gm::kKGroups;
    uint64_t* fullb = isv ? ms.v_full : ms.k_full;
    uint64_t* emptyb = isv ? ms.v_empty : ms.k_empty;
    bool aborted = false;
    int gc = 0;                                // running group count
    int uc = 0;                                // running unit count (queue entries)
    int next_static = blockIdx.x;              // fixed order when there is no counter
    TcUnit un;
    while (true) {
      if (!isv) {
        // The K producer claims the units of this CTA, one at a time as it starts
        // them (from the shared counter, or every gridDim.x-th one), and passes
        // them on through the queue; units without pages are skipped.
        int u = -1;
        bool found = false;
        while (!found) {
          if (lane == 0) {
            if (p.unit_counter != nullptr) {
              u = atomicAdd(p.unit_counter, 1);
            } else {
              u = next_static;
              next_static += gridDim.x;
            }
          }
          u = __shfl_sync(0xffffffffu, u, 0);
          if (u >= num_units) {
            u = -1;
            break;
          }
          bool bad;
          found = tc_unit(p, u, un, &bad);
          if (bad && lane == 0) atomicOr(&g_pa_err, kErrBounds);
        }
        if (!aborted && !mbar_wait(&ms.uq_empty[uc & 3], (static_cast<uint32_t>(uc >> 2) & 1u) ^ 1u,
                                   p.timeout_ns))
          aborted = true;
        aborted = __any_sync(0xffffffffu, aborted);
        if (lane == 0) {
          ms.unit_q[uc & 3] = aborted ? -1 : u;
          mbar_arrive(&ms.uq_full[uc & 3]);
        }
        if (u < 0 || aborted) break;
      } else {
        int c = uc;
        if (!tc_queue_next(ms, p, c, un, lane == 0, aborted)) break;
      }
      const int32_t* trow = p.block_tables + static_cast<size_t>(un.b) * p.mbs;
      if (!isv) {
        // the unit's query rows, K-major with the 128-byte swizzle, into Q buffer
        // uc & 1 once the score MMAs of unit uc - 2 are done
        if (!aborted && !mbar_wait(&ms.q_empty[uc & 1], (static_cast<uint32_t>(uc >> 1) & 1u) ^ 1u,
                                   p.timeout_ns))
          aborted = true;
        aborted = __any_sync(0xffffffffu, aborted);
        constexpr int CH = D / 8;
        constexpr int QV = NR * CH / 32;       // 16-byte chunks per lane
        uint8_t* qb = smem + Gm::kQOff + (uc & 1) * Gm::kQBytes;
        uint4 qv[QV];
#pragma unroll
        for (int i = 0; i < QV; ++i) {         // every load in flight at once
          const int idx = lane + 32 * i, r = idx / CH, ch = idx % CH;
          if (r < nrows) {
            const size_t row =
                (static_cast<size_t>(un.b) * T + r / G) * p.Hq + un.g * G + r % G;
            qv[i] = reinterpret_cast<const uint4*>(p.q)[row * CH + ch];
          }
        }
#pragma unroll
        for (int i = 0; i < QV; ++i) {
          const int idx = lane + 32 * i, r = idx / CH, ch = idx % CH;
          if (r < nrows) {
            const int n = r < hA ? r : NH + (r - hA);
            *reinterpret_cast<uint4*>(qb + (ch >> 3) * (NR * 128) + tc_sw128(n, (ch & 7) * 16)) =
                qv[i];
          }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.q_full[uc & 1]);
      }
      // Query tokens' K (V) that land in this unit's pages are stored first
      // (reshape_and_cache fused), then made visible to this warp's TMA reads.
      if (p.new_k != nullptr) {
        const int L = un.L;
        const int jlo = max(0, (L - T) / kBlockSize - un.pg0);
        const int jhi = min(un.npages - 1, (L - 1) / kBlockSize - un.pg0);
        for (int j = jlo; j <= jhi; ++j) {
          const int phys = __ldg(trow + un.pg0 + j);
          if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) continue;
          const int pos0 = (un.pg0 + j) * kBlockSize;
          const int lo = max(L - T, pos0), hi = min(L - 1, pos0 + kBlockSize - 1);
          for (int pos = lo; pos <= hi; ++pos) {
            const size_t src = (static_cast<size_t>(un.b) * T + (pos - (L - T))) * p.Hkv + un.g;
            const size_t dst = (static_cast<size_t>(phys) * p.Hkv + un.g) * kBlockSize +
                               (pos & (kBlockSize - 1));
            constexpr int CH = D / 8;
            if (lane < CH) {
              const uint4 v =
                  reinterpret_cast<const uint4*>(isv ? p.new_v : p.new_k)[src * CH + lane];
              reinterpret_cast<uint4*>(isv ? p.v_pool : p.k_pool)[dst * CH + lane] = v;
            }
          }
        }
        fence_proxy_async_global();
        __syncwarp();
      }
      // block ids of pages [32 i, 32 i + 32) in lane order, one batch read ahead
      int ids_cur = lane < un.npages ? __ldg(trow + un.pg0 + lane) : 0;
      int ids_nxt = 32 + lane < un.npages ? __ldg(trow + un.pg0 + 32 + lane) : 0;
      for (int grp = 0; grp < un.ngroups; ++grp, ++gc) {
        const int base = grp * Gm::kGroupPages;
        if (grp > 0 && (base & 31) == 0) {
          ids_cur = ids_nxt;
          ids_nxt = base + 32 + lane < un.npages ? __ldg(trow + un.pg0 + base + 32 + lane) : 0;
        }
        const int phys = __shfl_sync(0xffffffffu, ids_cur, (base & 31) + (lane & 7));
        const bool in = lane < Gm::kGroupPages && base + lane < un.npages;
        const bool inpool = static_cast<unsigned>(phys) < static_cast<unsigned>(p.num_blocks);
        if (isv && in && !inpool) atomicOr(&g_pa_err, kErrBounds);
        // the buffer is free once the score MMA (K) or the P.V (V) of group
        // gc - ngr has completed
        const int rb = gc % ngr;
        const uint32_t use = static_cast<uint32_t>(gc / ngr);
        if (!aborted && !mbar_wait(&emptyb[rb], (use & 1u) ^ 1u, p.timeout_ns)) aborted = true;
        aborted = __any_sync(0xffffffffu, aborted);
        const bool ok = in && inpool && !aborted;
        const unsigned okm = __ballot_sync(0xffffffffu, ok);
        // which pages the P.V may use (read by the MMA thread after v_full; the P.V
        // of group gc - 4, the previous reader of this entry, has completed)
        if (isv && lane < Gm::kGroupPages) ms.stage_ok[gc & 3][lane] = ok ? 1 : 0;
        __syncwarp();
        if (lane == 0)
          mbar_arrive_expect_tx(&fullb[rb],
                                static_cast<uint32_t>(__popc(okm)) * 2u * Gm::kHalfBytes);
        __syncwarp();
        if (ok) {
          const int row = (phys * p.Hkv + un.g) * kBlockSize;
          const int sl = rb * Gm::kGroupPages + lane;
          if (isv) {
            uint8_t* vd = smem + Gm::kVOff + sl * 2 * Gm::kHalfBytes;
            tma_load_2d(vd, &tmv, &fullb[rb], 0, row);
            tma_load_2d(vd + Gm::kHalfBytes, &tmv, &fullb[rb], 64, row);
          } else {
            uint8_t* kd = smem + Gm::kKOff + sl * Gm::kHalfBytes;
            tma_load_2d(kd, &tmk, &fullb[rb], 0, row);
            tma_load_2d(kd + Gm::kKSlots * Gm::kHalfBytes, &tmk, &fullb[rb], 64, row);
          }
        }
      }
      ++uc;
    }
    // Do not leave while copies issued by this warp may still be landing.
    if (lane == 0) {
      for (int c = max(0, gc - ngr); c < gc; ++c)
        mbar_wait(&fullb[c % ngr], static_cast<uint32_t>(c / ngr) & 1u, p.timeout_ns);
    }
  } else if (warp == Gm::kSoftmaxWarps + 1) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdQK = tc::idesc_f16<128, NR, false, false, true>();
      constexpr uint32_t kIdPV = tc::idesc_f16<128, 2 * NR, true, true, true>();
      // two cursors over the same units and groups: the next score MMA and the
      // next P.V (unit, unit count, group in the unit, running group count).  A
      // cursor takes its next unit from the queue when that entry is ready.
      TcUnit unq, unp;
      bool hq = false, hp = false;             // cursor holds a unit
      bool eq = false, ep = false;             // cursor reached the end of the queue
      int cq = 0, cp = 0, lq = 0, lp = 0, gq = 0, gp = 0;
      auto take = [&](int c, TcUnit& un, bool& have, bool& end) {
        if (have || end || !tc::mbar_test(&ms.uq_full[c & 3], static_cast<uint32_t>(c >> 2) & 1u))
          return;
        const int u = *reinterpret_cast<volatile int*>(&ms.unit_q[c & 3]);
        mbar_arrive(&ms.uq_empty[c & 3]);
        bool bad;
        if (u >= 0 && tc_unit(p, u, un, &bad)) have = true;
        else end = true;
      };
      uint32_t any_pv = 0;                     // a P.V of the current unit was issued
      bool aborted = false;
      unsigned long long t_prog = global_timer_ns();
      while (!ep && !aborted) {
        bool prog = false;
        take(cq, unq, hq, eq);
        take(cp, unp, hp, ep);
        // scores of group gq: query rows staged (first group of a unit), K
        // landed, its S buffer read out (group gq - 2), and at most one group
        // ahead of the P.V (the S and P barrier pairs)
        if (hq && gq <= gp + 1 &&
            (lq > 0 || tc::mbar_test(&ms.q_full[cq & 1], static_cast<uint32_t>(cq >> 1) & 1u)) &&
            tc::mbar_test(&ms.k_full[gq % Gm::kKGroups],
                          static_cast<uint32_t>(gq / Gm::kKGroups) & 1u) &&
            tc::mbar_test(&ms.s_free[gq & 1], (static_cast<uint32_t>(gq >> 1) & 1u) ^ 1u)) {
          tc::fence_after_sync();
          const int kb = gq % Gm::kKGroups;
          const uint32_t qb = qsm + (cq & 1) * Gm::kQBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = kring + (kk >> 2) * (Gm::kKSlots * Gm::kHalfBytes) +
                                kb * Gm::kGroupPages * Gm::kHalfBytes + (kk & 3) * 32;
            const uint32_t qa = qb + (kk >> 2) * (NR * 128) + (kk & 3) * 32;
            tc::mma_f16_ss(tmem + (gq & 1) * NR, tc::smem_desc(ka, 16, 1024),
                           tc::smem_desc(qa, 16, 1024), kIdQK, kk > 0 ? 1u : 0u);
          }
          tc::commit(&ms.k_empty[kb]);
          tc::commit(&ms.s_full[gq & 1]);
          ++gq;
          if (++lq == unq.ngroups) {
            tc::commit(&ms.q_empty[cq & 1]);
            lq = 0;
            ++cq;
            hq = false;
          }
          prog = true;
        }
        // P.V of group gp: O buffer of this unit read out (first group of a unit:
        // the unit two before used it), its P written and its V landed
        if (hp && gp < gq &&
            (lp > 0 ||
             tc::mbar_test(&ms.o_free[cp & 1], (static_cast<uint32_t>(cp >> 1) & 1u) ^ 1u)) &&
            tc::mbar_test(&ms.p_full[gp & 1], static_cast<uint32_t>(gp >> 1) & 1u) &&
            tc::mbar_test(&ms.v_full[gp % Gm::kVGroups],
                          static_cast<uint32_t>(gp / Gm::kVGroups) & 1u)) {
          tc::fence_after_sync();
          const int vb = gp % Gm::kVGroups;
          const uint32_t tmem_o = tmem + 2 * NR + (cp & 1) * 2 * NR;
          for (int j = 0; j < Gm::kGroupPages; ++j) {
            if (lp * Gm::kGroupPages + j >= unp.npages || !ms.stage_ok[gp & 3][j]) continue;
            const int sl = vb * Gm::kGroupPages + j;
            // A = V^T (MN-major, 128-byte swizzle): dims 64..127 one 2048-byte half
            // further (leading offset), tokens 8..15 one 1024-byte atom further
            const uint64_t ad = tc::smem_desc(vring + sl * 2 * Gm::kHalfBytes, Gm::kHalfBytes,
                                              1024);
            // B = [P_hi^T | P_lo^T] (MN-major, no swizzle): this page's two token
            // blocks (leading offset), row-slot blocks kPNStride apart (stride offset)
            const uint64_t bd = tc::smem_desc(psm + j * 2 * Gm::kPKStride, Gm::kPKStride,
                                              Gm::kPNStride, tc::kSwizzleNone);
            tc::mma_f16_ss(tmem_o, ad, bd, kIdPV, any_pv);
            any_pv = 1u;
          }
          tc::commit(&ms.v_empty[vb]);
          tc::commit(&ms.p_empty);
          ++gp;
          if (++lp == unp.ngroups) {
            lp = 0;
            any_pv = 0u;
            ++cp;
            hp = false;
          }
          prog = true;
        }
        if (prog) {
          t_prog = global_timer_ns();
        } else if (global_timer_ns() - t_prog > p.timeout_ns) {
          // the other roles' waits are bounded as well: they run out and finish
          atomicOr(&g_pa_err, kErrTimeout);
          aborted = true;
        }
      }
      // every MMA issued has completed before the CTA may release TMEM
      tc::commit(&ms.fin);
      mbar_wait(&ms.fin, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax
    const int q = warp & 3;                    // TMEM lane quarter
    const int hf = warp >> 2;                  // row-slot half
    const int t = q * 32 + lane;               // token of the group; head dim for O
    const int cnt = hf == 0 ? hA : nrows - hA; // rows of this half
    const int r0 = hf == 0 ? 0 : hA;           // first query row of this half
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const float sl2 = p.scale_log2;
    const int bar = 1 + hf;                    // named barrier of this half's 4 warps
    const bool nowin = p.window <= 0;
    bool aborted = false;
    int gs = 0;                                // running group count
    int cs = 0;                                // running unit count
    int cqe = 0;                               // queue entries read
    TcUnit un;
    while (tc_queue_next(ms, p, cqe, un, lane == 0, aborted)) {
      const int32_t* trow = p.block_tables + static_cast<size_t>(un.b) * p.mbs;
      // per row slot: reference max m, the threshold m + 8 past which it moves,
      // the exponent offset (m, or 0 while the row has seen nothing), row sum,
      // and the last position the row sees
      float m[NA], thr[NA], mref[NA], lp[NA];
      int lim[NA];
#pragma unroll
      for (int k = 0; k < NA; ++k) {
        m[k] = -CUDART_INF_F;
        thr[k] = -CUDART_INF_F;
        mref[k] = 0.f;
        lp[k] = 0.f;
        lim[k] = k < cnt ? un.L - T + (r0 + k) / G : -1;
      }
      const int minlim = un.L - T;             // every row sees positions <= L - T
      bool pv_before = false;                  // O holds data of an earlier group of the unit
      const int tail_tok = un.L - (un.pg0 + un.npages - 1) * kBlockSize;  // valid tokens, last page
      // block id of this thread's page in the next group, read one group ahead
      int id_next = t / 16 < un.npages ? __ldg(trow + un.pg0 + t / 16) : -1;
      for (int grp = 0; grp < un.ngroups; ++grp, ++gs) {
        const int sb = gs & 1;
        const int pidx = grp * Gm::kGroupPages + (t >> 4);
        const int id = id_next;
        id_next = pidx + Gm::kGroupPages < un.npages
                      ? __ldg(trow + un.pg0 + pidx + Gm::kGroupPages) : -1;
        if (!aborted && !mbar_wait(&ms.s_full[sb], static_cast<uint32_t>(gs >> 1) & 1u,
                                   p.timeout_ns))
          aborted = true;
        aborted = __any_sync(0xffffffffu, aborted);
        tc::fence_after_sync();
        uint32_t sr[NH];
        tc::tmem_ld16(tmem + lane_addr + sb * NR + hf * NH, sr);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.s_free[sb]);

        // a page outside the unit or naming a block outside the pool is not
        // loaded: its scores are masked and the MMA thread skips its P.V
        const bool valid = !aborted && pidx < un.npages &&
                           static_cast<unsigned>(id) < static_cast<unsigned>(p.num_blocks);
        const int j = (un.pg0 + pidx) * kBlockSize + (t & 15);
        const bool interior = valid && nowin && j <= minlim;
        float x[NA];
        bool exceed = false;
        if (interior) {                        // every row of the unit sees this token
#pragma unroll
          for (int k = 0; k < NA; ++k) {
            x[k] = k < cnt ? __uint_as_float(sr[k]) * sl2 : -CUDART_INF_F;
            exceed |= x[k] > thr[k];
          }
        } else {
#pragma unroll
          for (int k = 0; k < NA; ++k) {
            const bool vis = k < cnt && valid && static_cast<unsigned>(lim[k] - j) < p.wcap;
            x[k] = vis ? __uint_as_float(sr[k]) * sl2 : -CUDART_INF_F;
            exceed |= x[k] > thr[k];
          }
        }
        // decision of this half on moving its rows' reference maxima
        // (bit 0: some score of the warp exceeds its row's threshold; bit 1: the
        // warp's two pages include a loaded one)
        const bool wexceed = __any_sync(0xffffffffu, exceed);
        const bool wvalid = __any_sync(0xffffffffu, valid);
        if (lane == 0) ms.flag[sb][hf][q] = (wexceed ? 1 : 0) | (wvalid ? 2 : 0);
        named_bar_sync(bar, 128);
        const int fl = ms.flag[sb][hf][0] | ms.flag[sb][hf][1] | ms.flag[sb][hf][2] |
                       ms.flag[sb][hf][3];
        if (fl & 1) {
#pragma unroll
          for (int k = 0; k < NA; ++k) {
            float v = x[k];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) ms.red[hf][q][k] = v;
          }
          named_bar_sync(bar, 128);
          float alpha[NA];
          bool need_o = false;
#pragma unroll
          for (int k = 0; k < NA; ++k) {
            const float mx = fmaxf(fmaxf(ms.red[hf][0][k], ms.red[hf][1][k]),
                                   fmaxf(ms.red[hf][2][k], ms.red[hf][3][k]));
            alpha[k] = 1.f;
            if (mx > thr[k]) {
              if (m[k] != -CUDART_INF_F) {
                alpha[k] = hw_exp2(m[k] - mx);
                need_o = true;
              } else {
                alpha[k] = 0.f;
              }
              m[k] = mx;
              thr[k] = mx + 8.f;
              mref[k] = mx;
            }
            lp[k] *= alpha[k];
          }
          named_bar_sync(bar, 128);            // red[] may be rewritten next group
          if (need_o && pv_before && !aborted) {
            // O holds earlier groups of the unit: wait for their P.V (that of the
            // previous group; this thread waited for the one before it), then
            // rescale this half's columns in TMEM
            if (!mbar_wait(&ms.p_empty, (static_cast<uint32_t>(gs) & 1u) ^ 1u, p.timeout_ns))
              aborted = true;
            aborted = __any_sync(0xffffffffu, aborted);
            tc::fence_after_sync();
            const uint32_t to = tmem + 2 * NR + (cs & 1) * 2 * NR + lane_addr + hf * NH;
            uint32_t oh[NH], ol[NH];
            tc::tmem_ld16(to, oh);
            tc::tmem_ld16(to + NR, ol);
            tc::tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < NA; ++k) {
              oh[k] = __float_as_uint(__uint_as_float(oh[k]) * alpha[k]);
              ol[k] = __float_as_uint(__uint_as_float(ol[k]) * alpha[k]);
            }
            tc::tmem_st16(to, oh);
            tc::tmem_st16(to + NR, ol);
            tc::tmem_wait_st();
          }
        }
        // weights, row sums, and P^T as two bf16 parts (MN-major: one 16-byte row
        // of 8 row slots per token and core matrix)
        uint32_t hi[NH / 2], lo[NH / 2];
#pragma unroll
        for (int k = NA; k < NH; k += 2) hi[k / 2] = lo[k / 2] = 0u;
#pragma unroll
        for (int k = 0; k < NA; k += 2) {
          const float p0 = hw_exp2(x[k] - mref[k]), p1 = hw_exp2(x[k + 1] - mref[k + 1]);
          lp[k] += p0;
          lp[k + 1] += p1;
          const uint32_t h2 = pack_bf16x2(p0, p1);
          hi[k / 2] = h2;
          lo[k / 2] = pack_bf16x2(p0 - __uint_as_float(h2 << 16),
                                  p1 - __uint_as_float(h2 & 0xFFFF0000u));
        }
        // the P operand is free once the P.V of the previous group has completed
        if (!aborted && !mbar_wait(&ms.p_empty, (static_cast<uint32_t>(gs) & 1u) ^ 1u,
                                   p.timeout_ns))
          aborted = true;
        uint8_t* pt = smem + Gm::kPOff + (t >> 3) * Gm::kPKStride + (t & 7) * 16;
#pragma unroll
        for (int c = 0; c < NH / 8; ++c) {
          *reinterpret_cast<uint4*>(pt + (2 * hf + c) * Gm::kPNStride) =
              make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
          *reinterpret_cast<uint4*>(pt + (NR / 8 + 2 * hf + c) * Gm::kPNStride) =
              make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
        }
        // V rows past the context end in the last page may hold anything (even
        // NaN); their weight is 0, but 0 * NaN is NaN: zero them once they have
        // landed, before the P.V.  (The V buffer of this group is refilled only
        // after this group's P.V, so its barrier phase cannot run ahead.)
        if (hf == 0 && pidx == un.npages - 1 && (t & 15) >= tail_tok && valid &&
            mbar_wait(&ms.v_full[gs % Gm::kVGroups],
                      static_cast<uint32_t>(gs / Gm::kVGroups) & 1u, p.timeout_ns)) {
          const int sl = (gs % Gm::kVGroups) * Gm::kGroupPages + (t >> 4);
          uint4* vrow = reinterpret_cast<uint4*>(smem + Gm::kVOff + sl * 2 * Gm::kHalfBytes +
                                                 (t & 15) * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            vrow[c] = make_uint4(0, 0, 0, 0);
            vrow[c + Gm::kHalfBytes / 16] = make_uint4(0, 0, 0, 0);
          }
        }
        // the MMA thread issues P.V for every page of the group that is in the
        // unit and was loaded: from the next group on, O holds data
        pv_before |= (fl & 2) != 0;
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.p_full[sb]);
      }

      // -------------------------------------------------------------- unit output
      // the unit's last P.V (this thread waited for the one before it)
      if (!aborted && !mbar_wait(&ms.p_empty, static_cast<uint32_t>(gs - 1) & 1u, p.timeout_ns))
        aborted = true;
      aborted = __any_sync(0xffffffffu, aborted);
      tc::fence_after_sync();
      const uint32_t to = tmem + 2 * NR + (cs & 1) * 2 * NR + lane_addr + hf * NH;
      uint32_t oh[NH], ol[NH];
      tc::tmem_ld16(to, oh);
      tc::tmem_ld16(to + NR, ol);
      tc::tmem_wait_ld();
      // this unit's O buffer may take the unit after next
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms.o_free[cs & 1]);
#pragma unroll
      for (int k = 0; k < NA; ++k) {
        float v = lp[k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) ms.red[hf][q][k] = v;
      }
      named_bar_sync(bar, 128);
      const int d = t;                         // head dim of this thread's O^T lane
      int tq = r0 / G, hl = r0 % G;            // draft token and head in the group of the row
#pragma unroll
      for (int k = 0; k < NA; ++k) {
        if (k >= cnt) break;
        const float Ls =
            ms.red[hf][0][k] + ms.red[hf][1][k] + ms.red[hf][2][k] + ms.red[hf][3][k];
        const size_t orow = (static_cast<size_t>(un.b) * T + tq) * p.Hq + un.g * G + hl;
        if (++hl == G) {
          hl = 0;
          ++tq;
        }
        const float osum = __uint_as_float(oh[k]) + __uint_as_float(ol[k]);
        const float o = Ls > 0.f ? osum * __frcp_rn(Ls) : 0.f;
        if (un.direct) {
          reinterpret_cast<__nv_bfloat16*>(p.out)[orow * D + d] = __float2bfloat16_rn(o);
        } else {
          const size_t pidx2 = orow * p.max_parts + un.slot;
          p.part_o[pidx2 * D + d] = o;
          if (d == 0) p.part_ml[pidx2] = make_float2(m[k], Ls);
        }
      }
      named_bar_sync(bar, 128);                // red[] is rewritten by the next unit
      ++cs;
    }
  }

  // ------------------------------------------------------------------ teardown
  tc::fence_before_sync();
  __syncthreads();
  if (warp == Gm::kSoftmaxWarps + 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Gm::kTmemCols);
    tc::tmem_relinquish();
  }
}

template <int NA>
cudaError_t launch_tc_na(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                         int num_units, cudaStream_t s, bool overlap_previous) {
  constexpr int smem = TcGeo::kAlloc;
  auto kern = paged_attn_tc_kernel<NA>;
  static std::atomic<unsigned long long> configured{0ull};
  static std::atomic<int> sm_count[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  int sms = bit ? sm_count[dev].load(std::memory_order_relaxed) : 0;
  if (bit == 0 || (configured.load(std::memory_order_acquire) & bit) == 0 || sms == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (bit) {
      sm_count[dev].store(sms, std::memory_order_relaxed);
      configured.fetch_or(bit, std::memory_order_acq_rel);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::min(num_units, sms)), 1, 1);
  cfg.blockDim = dim3(TcGeo::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p, num_units);
}

// rows = query rows per kv head (17 .. 32); num_units = the work units
// (partitions x sequences x kv heads, partition-major); one CTA per SM.
inline cudaError_t launch_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                             int rows, int num_units, cudaStream_t s, bool overlap_previous) {
  if (num_units <= 0) return cudaSuccess;
  if (rows <= 20) return launch_tc_na<10>(tk, tv, p, num_units, s, overlap_previous);
  return launch_tc_na<16>(tk, tv, p, num_units, s, overlap_previous);
}

}  // namespace pa
