// Persistent paged attention, per-sequence mode, bf16 or FP8 pages: decode
// shapes (at most 8 query rows per kv head: one row column, four page lanes,
// 3 CTAs per SM) and verify tiles (17-24 rows: three row columns, two page
// lanes, two ring stages per softmax step, 2 CTAs per SM).
//
// The one-CTA-per-unit kernel (pa_attn.cuh) pays a start-up on every work
// unit: the context length, the block ids and the query rows are fetched before
// the unit's first page is requested, so its ring is empty for one to two
// memory round trips; and units past a sequence's end still cost a CTA.  Here
// as many CTAs as fit at once stream units back to back through one ring each:
//
//  * CTA c opens with partition 0 of sequence c / Hkv, kv head c % Hkv, which
//    needs only that sequence's length.  Meanwhile page lane 0 reads all context
//    lengths and builds the same dense, largest-first list of the remaining
//    units in every CTA: every full partition (ppb pages) of every sequence,
//    in sequence order, then every sequence's last partition, largest first (a
//    stable counting sort into 32 size classes).  List position i and kv head
//    h form unit i * Hkv + h; units past a sequence's end do not exist.
//  * CTAs claim list positions from a counter in the split-KV scratch (StreamCtl,
//    pa_internal.h: the merge that follows each launch resets it), so that an
//    idle CTA takes the next largest unit.  Without scratch, or on scratch whose
//    counter is not (yet) known to be reset, CTA c takes positions c,
//    2S - 1 - c, 2S + c, ... (S CTAs): a snake over the largest-first list.
//  * The producer warp publishes each unit into one of two records, with the
//    unit's query rows copied by cp.async into the record's query buffer, and
//    streams the unit's pages into the ring right behind the previous unit's.
//    The next claim goes out three issue groups before the end of the current
//    unit; the next unit is decoded, and its first 32 block ids requested, two
//    groups before the end; each later batch of 32 block ids is requested one
//    batch ahead.
//  * Units start on a multiple of the page-lane count in the ring (the skipped
//    items pass through empty), so page lane q takes a unit's pages q, q + PL,
//    ... whichever CTA runs it: the output is bit-identical to the
//    one-CTA-per-unit kernel's.
//  * Consumer warps take the records in order.  At a unit's end, with one row
//    column, each page lane keeps its last ring stage and writes its (m, l, O)
//    partial there; the lanes merge through those stages, write the output (one
//    partition) or the split-KV partial, and only then release the kept stages,
//    so the ring keeps streaming the next unit's first pages during the merge.
//    With three row columns the partials go to a merge buffer of their own.
//
// Partitions, partial slots and the merge kernel that follows are those of the
// one-CTA-per-unit kernel; the per-page arithmetic is the same function.
#pragma once

#include "pa_attn.cuh"

namespace pa {

struct StreamUnit {
  int b, g, pg0, npages, slot, direct, vlen, done;
};


template <int D, int NT, int NTW, int PL, bool KV8>
struct StreamSmem {
  using Gm = Geo<D, KV8>;
  static constexpr int kRows = 8 * NT * NTW;
  static constexpr int kQBytes = kRows * Gm::kQStride * 2;        // one query-row buffer
  static constexpr int kQOff = Gm::kNS * Gm::kStageBytes;         // two buffers
  static constexpr int kRecOff = kQOff + 2 * kQBytes;             // two unit records
  static constexpr int kLenOff = kRecOff + 2 * static_cast<int>(sizeof(StreamUnit));
  static constexpr int kPreOff = kLenOff + kStreamMaxSeqs * 4;    // full-unit prefix [B + 1]
  static constexpr int kOrdOff = kPreOff + (kStreamMaxSeqs + 1) * 4;   // last-partition order
  static constexpr int kCntOff = kOrdOff + kStreamMaxSeqs * 4;    // [chunk][size class] counts
  static constexpr int kMetaOff = kCntOff + kStreamMaxSeqs * 4;   // list sizes
  static constexpr int kBarOff = (kMetaOff + 16 + 7) / 8 * 8;
  static constexpr int kNumBars = 2 * Gm::kNS + 5;
  static constexpr int kOkOff = kBarOff + kNumBars * 8;
  static constexpr int kFlagOff = kOkOff + Gm::kNS * 4;
  // merge partial of one (page lane, row column): m[8NT], l[8NT], O[8NT][kOStride].
  // One column: in the page lane's kept ring stage.  Several: in a buffer of their own.
  static constexpr int kMergeFloats = 16 * NT + 8 * NT * Gm::kOStride;
  static constexpr bool kKeepStage = NTW == 1;
  static constexpr int kMergeOff = (kFlagOff + 16 + 15) / 16 * 16;
  static constexpr int kBytes = kMergeOff + (kKeepStage ? 0 : PL * NTW * kMergeFloats * 4);
  static constexpr int kAlloc = kBytes + 1024;                    // room to align the base to 1 KB
  static_assert(!kKeepStage || kMergeFloats * 4 <= Gm::kStageBytes,
                "a page lane's partial fits in one stage");
  static_assert(kQOff % 16 == 0 && Gm::kQStride * 2 % 16 == 0, "16-byte query chunks");
};

// Partitions of a sequence of L tokens (0: no units, an invalid length), with
// its first visible block and its block count.
__device__ __forceinline__ int stream_parts(int L, int T, const AttnParams& p, int& first,
                                            int& nblk) {
  if (L < T || L > p.max_ctx) return 0;
  nblk = (L + kBlockSize - 1) / kBlockSize;
  first = p.window > 0 ? max(0, L - T - p.window + 1) / kBlockSize : 0;
  return (nblk - first + p.ppb - 1) / p.ppb;
}

// The unit list, built by one warp: every full partition of every sequence in
// sequence order (fpre[b]: full units before sequence b), then every
// sequence's last partition, largest first (ord).  Partition 0 of sequences
// b < nb0 is left out (those open the kernel, one per CTA).  Stable counting
// sort into 32 size classes: class = 32 (ppb - pages) / ppb; the classes and
// ranks of every 32-sequence chunk are found at once, then combined.
__device__ __forceinline__ void build_unit_list(const AttnParams& p, int nb0, int lane,
                                                int* slen, int* fpre, int* ord, int* cnt,
                                                int* meta) {
  constexpr int kChunks = kStreamMaxSeqs / 32;
  const int B = p.num_seqs, ppb = p.ppb, T = p.T;
  int L[kChunks], nf[kChunks], cls[kChunks], rnk[kChunks];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int b = lane + 32 * i;
    L[i] = b < B ? __ldg(p.context_lens + b) : 0;
  }
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int b = lane + 32 * i;
    nf[i] = 0;
    cls[i] = 32;                             // 32: no last partition in the list
    if (b < B) {
      slen[b] = L[i];
      int first = 0, nblk = 0;
      const int np = stream_parts(L[i], T, p, first, nblk);
      if (np > 0) {
        const bool opened = b < nb0;         // partition 0 runs as a first unit
        nf[i] = max(0, np - 1 - (opened ? 1 : 0));
        if (!(opened && np == 1)) cls[i] = (ppb - (nblk - first - (np - 1) * ppb)) * 32 / ppb;
      } else {
        bad = true;
      }
    }
    cnt[32 * i + lane] = 0;
  }
  if (__any_sync(0xffffffffu, bad) && blockIdx.x == 0 && lane == 0) atomicOr(&g_pa_err, kErrBounds);
  // full units before each sequence: one warp scan per chunk, then the chunk carries
  int inc[kChunks];
#pragma unroll
  for (int i = 0; i < kChunks; ++i) inc[i] = nf[i];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
      const int y = __shfl_up_sync(0xffffffffu, inc[i], o);
      if (lane >= o) inc[i] += y;
    }
  }
  int carry = 0;
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int b = lane + 32 * i;
    if (b < B) fpre[b] = carry + inc[i] - nf[i];
    carry += __shfl_sync(0xffffffffu, inc[i], 31);
  }
  if (lane == 0) fpre[B] = carry;
  // size-class counts per chunk (one lane per class and chunk writes)
  __syncwarp();
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const unsigned same = __match_any_sync(0xffffffffu, cls[i]);
    rnk[i] = __popc(same & ((1u << lane) - 1u));
    if (cls[i] < 32 && rnk[i] == 0) cnt[32 * i + cls[i]] = __popc(same);
  }
  __syncwarp();
  // lane j: class j's count in earlier chunks (in place), and its total
  int tot = 0;
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int c = cnt[32 * i + lane];
    cnt[32 * i + lane] = tot;
    tot += c;
  }
  int off = tot;                             // classes before this lane's (largest first)
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, off, o);
    if (lane >= o) off += y;
  }
  const int nlast = __shfl_sync(0xffffffffu, off, 31);
  off -= tot;
  __syncwarp();
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int c = cls[i] < 32 ? cls[i] : 0;
    const int base = __shfl_sync(0xffffffffu, off, c);
    if (cls[i] < 32) ord[base + cnt[32 * i + c] + rnk[i]] = lane + 32 * i;
  }
  if (lane == 0) {
    meta[0] = carry;
    meta[1] = nlast;
  }
  __syncwarp();
}

template <int D, class C, bool KV8>
__global__ void __launch_bounds__(C::kThreads, C::MINB)
    paged_attn_stream_kernel(const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
  constexpr int NT = C::NT, NTW = C::NTW, PL = C::PL;
  constexpr int NCW = NTW * PL;              // consumer warps: NTW row columns x PL page lanes
  constexpr int NCT = NCW * 32;
  using Gm = Geo<D, KV8>;
  using Sm = StreamSmem<D, NT, NTW, PL, KV8>;
  constexpr int NS = Gm::kNS;
  constexpr int PPS = Gm::kPPS;              // pages per ring stage
  // ring stages per consumer step (as in the one-CTA-per-unit kernel; FP8 pages:
  // one stage of two pages), and pages per step
  constexpr int TPI = KV8 ? 1 : C::TP;
  constexpr int TP = TPI * PPS;
  static_assert(!Sm::kKeepStage || TPI == 1, "a kept stage ends a one-stage step");
  constexpr int CH = D / 8;                  // 16-byte chunks per query row
  static_assert(NS % PL == 0, "each stage is always consumed by the same page lane");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  __nv_bfloat16* qbuf = reinterpret_cast<__nv_bfloat16*>(smem + Sm::kQOff);
  StreamUnit* rec = reinterpret_cast<StreamUnit*>(smem + Sm::kRecOff);
  int* slen = reinterpret_cast<int*>(smem + Sm::kLenOff);
  int* fpre = reinterpret_cast<int*>(smem + Sm::kPreOff);
  int* ord = reinterpret_cast<int*>(smem + Sm::kOrdOff);
  int* cnt = reinterpret_cast<int*>(smem + Sm::kCntOff);
  int* meta = reinterpret_cast<int*>(smem + Sm::kMetaOff);   // full units, last partitions
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sm::kBarOff);
  uint64_t* empty = full + NS;
  uint64_t* ufull = empty + NS;              // unit record published (2)
  uint64_t* uempty = ufull + 2;              // unit record taken (2)
  uint64_t* lready = uempty + 2;             // unit list built
  int* stage_ok = reinterpret_cast<int*>(smem + Sm::kOkOff);
  // stop flags: s_stop[k & 1] is decided at the start of unit k (a consumer
  // wait that gave up sets it), read by every consumer warp after the barrier
  // that follows
  int* s_stop = reinterpret_cast<int*>(smem + Sm::kFlagOff);

  grid_launch_dependents();                  // the split-KV merge may start its CTAs
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G, T = p.T;
  const int nrows = G * T;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NTW);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ufull[i], 33);              // 32 cp.async arrivals + the record writer
      mbar_init(&uempty[i], NCW);
    }
    mbar_init(lready, 1);
    s_stop[0] = s_stop[1] = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // ------------------------------------------------------------------ producer
  if (warp == NCW) {
    if (lane == 0) {
      tma_prefetch_map(&tmk);
      tma_prefetch_map(&tmv);
    }
    const int B = p.num_seqs, ppb = p.ppb, S = static_cast<int>(gridDim.x);
    const int nb0 = min(B, S / p.Hkv);       // sequences whose first partitions open the kernel
    bool aborted = false;
    bool have_list = false;
    int nfull = 0, nlast = 0;
    auto wait_list = [&]() {
      if (have_list) return;
      if (!mbar_wait(lready, 0, p.timeout_ns)) aborted = true;
      aborted = __any_sync(0xffffffffu, aborted);
      have_list = true;
      nfull = meta[0];
      nlast = meta[1];
    };
    auto fill = [&](StreamUnit& r, int b, int g, int L, int part) {
      int first = 0, nblk = 0;
      const int np = stream_parts(L, T, p, first, nblk);
      r.b = b;
      r.g = g;
      r.pg0 = first + part * ppb;
      r.npages = min(ppb, nblk - r.pg0);
      r.slot = part;
      r.direct = np == 1;
      r.vlen = L;
      r.done = 0;
    };
    // List positions: claimed from the counter (dynamic: an idle CTA takes the
    // next largest unit), or without it position k * S + c (c = this CTA) on even
    // passes k, k * S + S - 1 - c on odd ones, a snake over the largest-first list.
    StreamCtl* ctl = static_cast<StreamCtl*>(p.stream_ctl);
    bool dyn = false;
    if (ctl != nullptr) {
      unsigned long long tag = 0;
      if (lane == 0) tag = *reinterpret_cast<volatile unsigned long long*>(&ctl->tag);
      dyn = __shfl_sync(0xffffffffu, tag == kStreamTag ? 1 : 0, 0) != 0;
    }
    int k_list = 0;
    auto request = [&]() -> long long {      // lane 0's value is the position
      if (dyn) return lane == 0 ? static_cast<long long>(atomicAdd(&ctl->next, 1)) : 0ll;
      const long long pos = static_cast<long long>(k_list) * S +
                            ((k_list & 1) ? S - 1 - static_cast<int>(blockIdx.x)
                                          : static_cast<int>(blockIdx.x));
      ++k_list;
      return pos;
    };
    auto next_from_list = [&](long long req, StreamUnit& r) {
      r.done = 1;
      const long long pos = __shfl_sync(0xffffffffu, req, 0);
      wait_list();
      if (aborted) return;
      if (pos >= static_cast<long long>(nfull + nlast) * p.Hkv) return;
      const int li = static_cast<int>(pos / p.Hkv), g = static_cast<int>(pos % p.Hkv);
      int b, part;
      if (li < nfull) {
        int lo = 0, hi = B - 1;              // last b with fpre[b] <= li
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (fpre[mid] <= li) lo = mid; else hi = mid - 1;
        }
        b = lo;
        part = (b < nb0 ? 1 : 0) + li - fpre[b];
      } else {
        b = ord[li - nfull];
        int first = 0, nblk = 0;
        part = stream_parts(slen[b], T, p, first, nblk) - 1;
      }
      fill(r, b, g, slen[b], part);
    };
    // Query rows of (sequence b, kv head g) into query buffer `buf` by cp.async
    // (rows past the query rows are zero-filled).
    auto copy_q = [&](int buf, int b, int g) {
      __nv_bfloat16* qd = qbuf + buf * (Sm::kRows * Gm::kQStride);
      for (int idx = lane; idx < Sm::kRows * CH; idx += 32) {
        const int n = idx / CH, ch = idx % CH;
        const bool valid = n < nrows;
        const size_t row = valid ? (static_cast<size_t>(b) * T + n / G) * p.Hq + g * G + n % G : 0;
        cp_async_16(smem_u32(qd + n * Gm::kQStride + ch * 8),
                    reinterpret_cast<const uint4*>(p.q) + row * CH + (valid ? ch : 0),
                    valid ? 16u : 0u);
      }
    };
    // The first unit: partition 0 of sequence c / Hkv, kv head c % Hkv.  It needs
    // only that sequence's length, not the list; its query rows and (without a
    // window, when it starts at block 0) its first 32 block ids are requested
    // together with the length.
    StreamUnit cu;
    cu.done = 1;
    int phys_pref = 0;                       // cu's first 32 block ids
    bool have_pref = false, q_first = false;
    if (static_cast<int>(blockIdx.x) < nb0 * p.Hkv) {
      const int b = static_cast<int>(blockIdx.x) / p.Hkv, g = static_cast<int>(blockIdx.x) % p.Hkv;
      copy_q(0, b, g);
      q_first = true;
      if (p.window <= 0 && lane < p.mbs)
        phys_pref = __ldg(p.block_tables + static_cast<size_t>(b) * p.mbs + lane);
      const int L = __ldg(p.context_lens + b);
      int first = 0, nblk = 0;
      if (stream_parts(L, T, p, first, nblk) > 0) {
        fill(cu, b, g, L, 0);
        have_pref = p.window <= 0;
      }
    }
    if (cu.done) next_from_list(request(), cu);
    if (!have_pref) {
      phys_pref = 0;
      if (!cu.done && lane < cu.npages)
        phys_pref = __ldg(p.block_tables + static_cast<size_t>(cu.b) * p.mbs + cu.pg0 + lane);
    }
    constexpr int GP = Gm::kIssueGroup;
    constexpr int IPB = 32 / PPS;            // stages per batch of 32 block ids
    static_assert(GP >= 1 && GP <= NS && IPB % GP == 0, "issue group");
    int k = 0, item0 = 0;
    while (true) {
      // ---- publish unit k (or the end)
      const int buf = k & 1;
      if (!aborted && !mbar_wait(&uempty[buf], ((k >> 1) & 1u) ^ 1u, p.timeout_ns)) aborted = true;
      aborted = __any_sync(0xffffffffu, aborted);
      const bool done = cu.done || aborted;
      if (lane == 0) {
        rec[buf] = cu;
        rec[buf].done = done;
      }
      // The first unit's rows are already on their way; if that unit turned out
      // empty (an invalid length), those copies land before buffer 0 is refilled.
      const bool q_sent = k == 0 && q_first && cu.b == static_cast<int>(blockIdx.x) / p.Hkv &&
                          cu.g == static_cast<int>(blockIdx.x) % p.Hkv && cu.slot == 0;
      if (k == 0 && q_first && !q_sent) asm volatile("cp.async.wait_all;" ::: "memory");
      if (!done && !q_sent) copy_q(buf, cu.b, cu.g);
      cp_async_mbar_arrive(&ufull[buf]);
      if (lane == 0) mbar_arrive(&ufull[buf]);
      ++k;
      if (done) break;

      // Units start on a multiple of PL ring items, so that page lane q takes
      // the unit's items q, q + PL, ... whichever CTA runs it: the arithmetic of
      // a unit, and so its result, does not depend on the schedule.  The items
      // skipped to get there pass through the ring empty.
      {
        const int start = (item0 + PL - 1) / PL * PL;
        if (lane < start - item0) {
          const int it = item0 + lane;
          const int s = it % NS;
          if (!aborted &&
              !mbar_wait(&empty[s], (static_cast<uint32_t>(it / NS) & 1u) ^ 1u, p.timeout_ns))
            aborted = true;
          stage_ok[s] = 0;
          mbar_arrive(&full[s]);
        }
        aborted = __any_sync(0xffffffffu, aborted);
        item0 = start;
      }

      // ---- stream unit cu's pages
      const int b = cu.b, g = cu.g, pg0 = cu.pg0, npages = cu.npages, vlen = cu.vlen;
      const int nitems = (npages + PPS - 1) / PPS;
      const int32_t* trow = p.block_tables + static_cast<size_t>(b) * p.mbs;
      // Query tokens' K/V that land in this unit's pages are stored into the pool
      // (reshape_and_cache fused; FP8 pages quantise on the way), as in the
      // one-CTA-per-unit kernel: after the first group is in flight, with the
      // proxy fence right before the first page that holds a new token.
      int fence_at = npages;
      int jlo = npages, jhi = -1;
      if (p.new_k != nullptr) {
        jlo = max(0, (vlen - T) / kBlockSize - pg0);
        jhi = min(npages - 1, (vlen - 1) / kBlockSize - pg0);
      }
      bool pending = jlo <= jhi;
      auto store_new_tokens = [&]() {
        for (int j = jlo; j <= jhi; ++j) {
          const int phys = __ldg(trow + pg0 + j);
          const int pos0 = (pg0 + j) * kBlockSize;
          const int lo = max(vlen - T, pos0), hi = min(vlen - 1, pos0 + kBlockSize - 1);
          if (lo > hi || static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks))
            continue;                         // out-of-range ids are reported when issued
          fence_at = min(fence_at, j);
          for (int pos = lo; pos <= hi; ++pos) {
            const size_t src = (static_cast<size_t>(b) * T + (pos - (vlen - T))) * p.Hkv + g;
            const size_t page = static_cast<size_t>(phys) * p.Hkv + g;
            const int off = pos & (kBlockSize - 1);
            if constexpr (KV8) {
              const float ks = p.k_scale[g], vs = p.v_scale[g];
              for (int c = lane; c < D / 4; c += 32) {
                const uint2 kx = reinterpret_cast<const uint2*>(p.new_k)[src * (D / 4) + c];
                const uint2 vx = reinterpret_cast<const uint2*>(p.new_v)[src * (D / 4) + c];
                const uint32_t k01 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(kx.x), ks),
                                                     __fdiv_rn(bf16_hi(kx.x), ks));
                const uint32_t k23 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(kx.y), ks),
                                                     __fdiv_rn(bf16_hi(kx.y), ks));
                const uint32_t v01 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(vx.x), vs),
                                                     __fdiv_rn(bf16_hi(vx.x), vs));
                const uint32_t v23 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(vx.y), vs),
                                                     __fdiv_rn(bf16_hi(vx.y), vs));
                uint8_t* kp = static_cast<uint8_t*>(p.k_pool);
                uint8_t* vp = static_cast<uint8_t*>(p.v_pool);
                *reinterpret_cast<uint32_t*>(kp + (page * kBlockSize + off) * D + 4 * c) =
                    k01 | (k23 << 16);
                uint8_t* vrow = vp + (page * D + 4 * c) * kBlockSize + off;
                vrow[0] = static_cast<uint8_t>(v01 & 0xFFu);
                vrow[kBlockSize] = static_cast<uint8_t>(v01 >> 8);
                vrow[2 * kBlockSize] = static_cast<uint8_t>(v23 & 0xFFu);
                vrow[3 * kBlockSize] = static_cast<uint8_t>(v23 >> 8);
              }
            } else {
              const size_t dst = page * kBlockSize + off;
              for (int c = lane; c < 2 * CH; c += 32) {
                const bool isv = c >= CH;
                const int cc = isv ? c - CH : c;
                const uint4 v =
                    reinterpret_cast<const uint4*>(isv ? p.new_v : p.new_k)[src * CH + cc];
                reinterpret_cast<uint4*>(isv ? p.v_pool : p.k_pool)[dst * CH + cc] = v;
              }
            }
          }
        }
        __syncwarp();
        pending = false;
      };
      if (pending && jlo < GP * PPS) store_new_tokens();   // the first group holds a new token

      StreamUnit nu;
      nu.done = 1;
      bool resolved = false, requested = false;
      long long req = 0;
      int phys_cur = phys_pref;              // lane l: block id of page base + l
      for (int base = 0; base < npages; base += 32) {
        const int phys_nb = (base + 32 + lane < npages) ? __ldg(trow + pg0 + base + 32 + lane) : 0;
        const int cnt = min(32, npages - base);
        const int icnt = (cnt + PPS - 1) / PPS;
        int phys_a = phys_cur, phys_b = 0;
        if constexpr (PPS == 2) {
          phys_a = __shfl_sync(0xffffffffu, phys_cur, (2 * lane) & 31);
          phys_b = __shfl_sync(0xffffffffu, phys_cur, (2 * lane + 1) & 31);
        }
        for (int j0 = 0; j0 < icnt; j0 += GP) {
          const int jn = min(j0 + GP, icnt);
          if (min(npages, base + PPS * jn) > fence_at) {
            fence_proxy_async_global();
            __syncwarp();
            fence_at = npages;
          }
          if (lane >= j0 && lane < jn) {
            const int it = item0 + base / PPS + lane;
            const int s = it % NS;
            const uint32_t ph = static_cast<uint32_t>(it / NS) & 1u;
            if (!aborted && !mbar_wait(&empty[s], ph ^ 1u, p.timeout_ns)) aborted = true;
            const bool two = PPS == 2 && base + 2 * lane + 1 < npages;
            const bool ok = static_cast<unsigned>(phys_a) < static_cast<unsigned>(p.num_blocks) &&
                            (!two || static_cast<unsigned>(phys_b) <
                                         static_cast<unsigned>(p.num_blocks));
            if (!ok) atomicOr(&g_pa_err, kErrBounds);
            if (!ok || aborted) {
              stage_ok[s] = 0;
              mbar_arrive(&full[s]);
            } else {
              stage_ok[s] = 1;
              uint8_t* st = stages + s * Gm::kStageBytes;
              if constexpr (KV8) {
                mbar_arrive_expect_tx(&full[s], (two ? 4 : 2) * Gm::kPageBytes);
                tma_load_2d(st, &tmk, &full[s], 0, (phys_a * p.Hkv + g) * kBlockSize);
                tma_load_2d(st + 2 * Gm::kPageBytes, &tmv, &full[s], 0,
                            (phys_a * p.Hkv + g) * (D / 8));
                if (two) {
                  tma_load_2d(st + Gm::kPageBytes, &tmk, &full[s], 0,
                              (phys_b * p.Hkv + g) * kBlockSize);
                  tma_load_2d(st + 3 * Gm::kPageBytes, &tmv, &full[s], 0,
                              (phys_b * p.Hkv + g) * (D / 8));
                }
              } else {
                mbar_arrive_expect_tx(&full[s], Gm::kStageBytes);
                const int row = (phys_a * p.Hkv + g) * kBlockSize;
#pragma unroll
                for (int h = 0; h < Gm::kHalves; ++h)
                  tma_load_2d(st + h * Gm::kHalfBytes, &tmk, &full[s], h * 64, row);
#pragma unroll
                for (int h = 0; h < Gm::kHalves; ++h)
                  tma_load_2d(st + Gm::kPageBytes + h * Gm::kHalfBytes, &tmv, &full[s], h * 64,
                              row);
              }
            }
          }
          aborted = __any_sync(0xffffffffu, aborted);
          if (pending) store_new_tokens();
          if (!requested && base / PPS + jn + 3 * GP >= nitems) {
            requested = true;                // the claim is in flight one group early
            req = request();
          }
          if (!resolved && base / PPS + jn + 2 * GP >= nitems) {
            // At most two groups of this unit are left to issue: take the next
            // unit and request its first block ids.
            resolved = true;
            next_from_list(req, nu);
            phys_pref = 0;
            if (!nu.done && lane < nu.npages)
              phys_pref =
                  __ldg(p.block_tables + static_cast<size_t>(nu.b) * p.mbs + nu.pg0 + lane);
          }
        }
        phys_cur = phys_nb;
      }
      if (!resolved) {                       // a unit without pages (never produced)
        next_from_list(requested ? req : request(), nu);
        phys_pref = 0;
        if (!nu.done && lane < nu.npages)
          phys_pref = __ldg(p.block_tables + static_cast<size_t>(nu.b) * p.mbs + nu.pg0 + lane);
      }
      item0 += nitems;
      cu = nu;
    }
    // Do not leave while copies issued by this warp may still be landing.
    if (lane == 0) {
      for (int it = max(0, item0 - NS); it < item0; ++it)
        mbar_wait(&full[it % NS], static_cast<uint32_t>(it / NS) & 1u, p.timeout_ns);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  if (warp == 0) {
    // The list is needed from the second unit on; page lane 0 builds it while
    // the first units' pages are on their way.
    build_unit_list(p, min(p.num_seqs, static_cast<int>(gridDim.x) / p.Hkv), lane, slen, fpre,
                    ord, cnt, meta);
    if (lane == 0) mbar_arrive(lready);
  }
  const int col = warp % NTW;                // rows 8*NT*col .. 8*NT*(col+1)-1
  const int pl = warp / NTW;                 // page lane: items pl, pl + PL, ... (mod PL)
  const int rbase = 8 * NT * col;
  const int gid = lane >> 2, q4 = lane & 3;
  float sl2 = p.scale_log2;
  float out_scale = 1.f;
  // per-lane ldmatrix row/chunk selectors (as in the one-CTA-per-unit kernel)
  const int mi = lane >> 3, rr = lane & 7;
  const int ktok = rr + ((mi & 1) << 3), kch = mi >> 1;
  const int vtok = rr + ((mi >> 1) << 3), vch = mi & 1;
  uint32_t koff[4], voff[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if constexpr (KV8) {
      koff[k] = page8_off<D>(sigma_row(ktok), 2 * k + kch);
      voff[k] = static_cast<uint32_t>((32 * k + lane) * 16);
    } else {
      koff[k] = page_off(ktok, 2 * k + kch);
      voff[k] = page_off(vtok, 2 * k + vch);
    }
  }
  const int srow0 = KV8 ? sigma_row(gid) : gid;
  const int srow1 = KV8 ? sigma_row(gid + 8) : gid + 8;
  constexpr bool kQRegs = true;
  static_assert(NT <= 2, "query fragments held in registers");

  bool aborted = false;
  int k = 0, item0 = 0;
  while (true) {
    const int buf = k & 1;
    if (!aborted && !mbar_wait(&ufull[buf], static_cast<uint32_t>(k >> 1) & 1u, p.timeout_ns))
      aborted = true;
    if (aborted) s_stop[k & 1] = 1;
    __nv_bfloat16* qb = qbuf + buf * (Sm::kRows * Gm::kQStride);
    if constexpr (KV8) {
      // f16 in place, and inside every 16 dims in the order of the FP8 K bytes
      // (dims 4q, 4q+1 at 2q, 2q+1; 4q+2, 4q+3 at 2q+8, 2q+9): each thread
      // rewrites whole 16-dim groups.
      for (int idx = threadIdx.x; idx < Sm::kRows * (D / 16); idx += NCT) {
        const int n = idx / (D / 16), gq = idx % (D / 16);
        uint4* src = reinterpret_cast<uint4*>(qb + n * Gm::kQStride + gq * 16);
        const uint4 a = src[0], c = src[1];
        uint4 lo, hi;
        lo.x = bf16x2_to_f16x2(a.x);          // dims 0,1 -> 0,1
        hi.x = bf16x2_to_f16x2(a.y);          // dims 2,3 -> 8,9
        lo.y = bf16x2_to_f16x2(a.z);          // dims 4,5 -> 2,3
        hi.y = bf16x2_to_f16x2(a.w);          // dims 6,7 -> 10,11
        lo.z = bf16x2_to_f16x2(c.x);          // dims 8,9 -> 4,5
        hi.z = bf16x2_to_f16x2(c.y);          // dims 10,11 -> 12,13
        lo.w = bf16x2_to_f16x2(c.z);          // dims 12,13 -> 6,7
        hi.w = bf16x2_to_f16x2(c.w);          // dims 14,15 -> 14,15
        src[0] = lo;
        src[1] = hi;
      }
    }
    named_bar_sync(1, NCT);                  // record read by all; stop agreed on
    const StreamUnit r = rec[buf];
    if (s_stop[k & 1] || r.done) break;
    const int g = r.g;
    if constexpr (KV8) {
      sl2 = p.scale_log2 * p.k_scale[g];
      out_scale = p.v_scale[g];
    }
    const uint32_t qrow = smem_u32(qb) + static_cast<uint32_t>(
                                             (rbase + (lane & 7)) * Gm::kQStride * 2 +
                                             (lane >> 3) * 16);
    uint32_t qf[NT][Gm::kKSteps][2];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int ks = 0; ks < Gm::kKSteps; ks += 2)
        ldsm_x4(qf[j][ks][0], qf[j][ks][1], qf[j][ks + 1][0], qf[j][ks + 1][1],
                qrow + static_cast<uint32_t>(j * 8 * Gm::kQStride * 2 + ks * 32));
    __syncwarp();
    if (lane == 0) mbar_arrive(&uempty[buf]);

    // visibility limits of this lane's rows rbase + 8j + 2q4 (+1); padding rows
    // see everything
    int lim0[NT], lim1[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int n0 = rbase + 8 * j + 2 * q4, n1 = n0 + 1;
      lim0[j] = n0 < nrows ? r.vlen - T + (n0 / G) % T : 0x7fffffff;
      lim1[j] = n1 < nrows ? r.vlen - T + (n1 / G) % T : 0x7fffffff;
    }
    int minlim = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < NT; ++j) minlim = min(minlim, min(lim0[j], lim1[j]));
    minlim = __reduce_min_sync(0xffffffffu, minlim);

    StepState<D, NT, TP, KV8> st;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int i = 0; i < Gm::kKSteps; ++i)
        st.acc[j][i][0] = st.acc[j][i][1] = st.acc[j][i][2] = st.acc[j][i][3] = 0.f;
      st.m0[j] = st.m1[j] = -CUDART_INF_F;
      st.l0[j] = st.l1[j] = 0.f;
    }

    // The skipped items before this unit's first (a multiple of PL): this
    // lane's one, if any, is passed through.
    {
      const int start = (item0 + PL - 1) / PL * PL;
      const int gi = item0 + ((pl - item0 % PL) % PL + PL) % PL;
      if (gi < start) {
        const int s = gi % NS;
        if (!aborted && !mbar_wait(&full[s], static_cast<uint32_t>(gi / NS) & 1u, p.timeout_ns))
          aborted = true;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      item0 = start;
    }
    const int nitems = (r.npages + PPS - 1) / PPS;
    const int iend = item0 + nitems;
    // first and last item of page lane q in this unit (none if first >= iend)
    auto lane_first = [&](int q) { return item0 + q; };
    auto lane_last = [&](int q) { return item0 + q + ((nitems - 1 - q) / PL) * PL; };
    const int my_first = lane_first(pl);
    // Steps of TPI items of this lane (gi, gi + PL): one softmax update per step.
    for (int gi = my_first; gi < iend; gi += TPI * PL) {
      const int nstep = (TPI == 2 && gi + PL < iend) ? 2 : 1;
      bool okp[TP];
      uint32_t kb[TP], vb[TP];
      int tok0[TP], sidx[TPI];
#pragma unroll
      for (int si = 0; si < TPI; ++si) {
        sidx[si] = -1;
#pragma unroll
        for (int u = 0; u < PPS; ++u) {
          okp[si * PPS + u] = false;
          kb[si * PPS + u] = vb[si * PPS + u] = 0;
          tok0[si * PPS + u] = 0;
        }
        if (si < nstep) {
          const int item = gi + si * PL;
          const int s = item % NS;
          if (!aborted && !mbar_wait(&full[s], static_cast<uint32_t>(item / NS) & 1u,
                                     p.timeout_ns))
            aborted = true;
          const bool ok = !aborted && stage_ok[s];
          const uint32_t sb = smem_u32(stages + s * Gm::kStageBytes);
          sidx[si] = s;
#pragma unroll
          for (int u = 0; u < PPS; ++u) {
            const int pg = (item - item0) * PPS + u;
            okp[si * PPS + u] = ok && pg < r.npages;
            kb[si * PPS + u] = sb + u * Gm::kPageBytes;
            vb[si * PPS + u] = sb + (PPS + u) * Gm::kPageBytes;
            tok0[si * PPS + u] = (r.pg0 + pg) * kBlockSize;
          }
        }
      }
      attend_step<D, NT, TP, KV8, kQRegs>(st, okp, kb, vb, tok0, qf, qrow, koff, voff, lim0,
                                          lim1, minlim, r.vlen, sl2, srow0, srow1, q4, p);
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int si = 0; si < TPI; ++si) {
          // with one row column the lane's last stage is kept for the merge
          if (si < nstep && !(Sm::kKeepStage && gi + si * PL + PL >= iend))
            mbar_arrive(&empty[sidx[si]]);
        }
      }
    }

    // ---- unit end: merge the page lanes (through their kept stages with one row
    // column, else through the merge buffer)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        st.l0[j] += __shfl_xor_sync(0xffffffffu, st.l0[j], o);
        st.l1[j] += __shfl_xor_sync(0xffffffffu, st.l1[j], o);
      }
    }
    const int held = (Sm::kKeepStage && my_first < iend) ? lane_last(pl) % NS : -1;
    if (my_first < iend) {
      float* mbuf = Sm::kKeepStage
                        ? reinterpret_cast<float*>(stages + held * Gm::kStageBytes)
                        : reinterpret_cast<float*>(smem + Sm::kMergeOff) +
                              (pl * NTW + col) * Sm::kMergeFloats;
      float* ob = mbuf + 16 * NT;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int r0 = 8 * j + 2 * q4;
        if (gid == 0) {
          mbuf[r0] = st.m0[j];
          mbuf[r0 + 1] = st.m1[j];
          mbuf[8 * NT + r0] = st.l0[j];
          mbuf[8 * NT + r0 + 1] = st.l1[j];
        }
#pragma unroll
        for (int mt = 0; mt < Gm::kKSteps; ++mt) {
          ob[r0 * Gm::kOStride + 16 * mt + gid] = st.acc[j][mt][0];
          ob[(r0 + 1) * Gm::kOStride + 16 * mt + gid] = st.acc[j][mt][1];
          ob[r0 * Gm::kOStride + 16 * mt + gid + 8] = st.acc[j][mt][2];
          ob[(r0 + 1) * Gm::kOStride + 16 * mt + gid + 8] = st.acc[j][mt][3];
        }
      }
    }
    if (aborted) s_stop[(k + 1) & 1] = 1;
    named_bar_sync(1, NCT);
    {
      // partials of the page lanes that had pages (row column 0; the merge
      // buffer holds the columns of one page lane side by side)
      const float* mbq[PL];
#pragma unroll
      for (int q = 0; q < PL; ++q) {
        mbq[q] = nullptr;
        if (lane_first(q) < iend)
          mbq[q] = Sm::kKeepStage
                       ? reinterpret_cast<const float*>(stages +
                                                        (lane_last(q) % NS) * Gm::kStageBytes)
                       : reinterpret_cast<const float*>(smem + Sm::kMergeOff) +
                             q * NTW * Sm::kMergeFloats;
      }
      for (int idx = threadIdx.x; idx < nrows * (D / 2); idx += NCT) {
        const int n0 = idx / (D / 2);
        const int d = (idx % (D / 2)) * 2;
        const int c = n0 / (8 * NT), n = n0 % (8 * NT);   // row column, row within it
        const int cofs = c * Sm::kMergeFloats;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int q = 0; q < PL; ++q)
          if (mbq[q] != nullptr) M = fmaxf(M, mbq[q][cofs + n]);
        float Ls = 0.f, o0 = 0.f, o1 = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
          for (int q = 0; q < PL; ++q) {
            if (mbq[q] == nullptr) continue;
            const float* mb = mbq[q] + cofs;
            const float f = exp2f(mb[n] - M);
            Ls += f * mb[8 * NT + n];
            o0 += f * mb[16 * NT + n * Gm::kOStride + d];
            o1 += f * mb[16 * NT + n * Gm::kOStride + d + 1];
          }
        }
        const int t = (n0 / G) % T, hl = n0 % G;
        const size_t orow = (static_cast<size_t>(r.b) * T + t) * p.Hq + g * G + hl;
        if (r.direct) {
          const float inv = out_scale / Ls;
          reinterpret_cast<__nv_bfloat162*>(p.out)[(orow * D + d) >> 1] =
              __floats2bfloat162_rn(o0 * inv, o1 * inv);
        } else {
          const float inv = Ls > 0.f ? out_scale / Ls : 0.f;
          const size_t pidx = orow * p.max_parts + r.slot;
          reinterpret_cast<float2*>(p.part_o)[(pidx * D + d) >> 1] =
              make_float2(o0 * inv, o1 * inv);
          if (d == 0) p.part_ml[pidx] = make_float2(M, Ls);
        }
      }
    }
    // The kept stages were written and read through the generic proxy; the
    // producer's next TMA writes to them come after this fence and the release.
    // (With a merge buffer, the barrier keeps the next unit's partials from
    // overwriting this one's before every thread has read them.)
    if constexpr (Sm::kKeepStage) fence_proxy_async_smem();
    named_bar_sync(1, NCT);
    if (held >= 0 && lane == 0) mbar_arrive(&empty[held]);
    item0 = iend;
    ++k;
  }
}

// Resident CTAs per SM and SMs of the current device, queried once per device.
template <int D, class C, bool KV8>
cudaError_t stream_grid_limit(int* limit) {
  constexpr int smem = StreamSmem<D, C::NT, C::NTW, C::PL, KV8>::kAlloc;
  auto kern = paged_attn_stream_kernel<D, C, KV8>;
  static std::atomic<int> cached[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_acquire);
    if (c > 0) {
      *limit = c;
      return cudaSuccess;
    }
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::kThreads, smem);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int c = std::max(1, per_sm) * std::max(1, sms);
  if (dev >= 0 && dev < 64) cached[dev].store(c, std::memory_order_release);
  *limit = c;
  return cudaSuccess;
}

template <int D, class C, bool KV8>
cudaError_t launch_stream_cfg(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                              long long max_units, bool always, cudaStream_t s, bool* launched) {
  int limit = 0;
  cudaError_t e = stream_grid_limit<D, C, KV8>(&limit);
  if (e != cudaSuccess) return e;
  if (!always && max_units < 4ll * limit) return cudaSuccess;
  const int grid = static_cast<int>(std::min<long long>(std::max(1ll, max_units), limit));
  constexpr int smem = StreamSmem<D, C::NT, C::NTW, C::PL, KV8>::kAlloc;
  paged_attn_stream_kernel<D, C, KV8><<<grid, C::kThreads, smem, s>>>(tk, tv, p);
  e = cudaGetLastError();
  *launched = e == cudaSuccess;
  return e;
}

// `rows` = query rows per kv head: at most 8 (decode; one row column, 3 CTAs
// per SM) or 17-24 (verify; three row columns, 2 CTAs per SM, the layouts of the
// one-CTA-per-unit kernel).  `max_units` bounds the work units (partitions x kv
// heads x sequences); the grid is the smaller of it and the CTAs that fit on
// the device at once.  Unless `always`, the kernel is launched only with at
// least 4 units (bound) per resident CTA: with fewer, long units (bf16 pages at
// 8B shape: 2 per CTA) measured no faster than one CTA per unit.  *launched
// says whether it ran; other row counts never run here.
template <int D, bool KV8>
cudaError_t launch_stream(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                          int rows, long long max_units, bool always, cudaStream_t s,
                          bool* launched) {
  *launched = false;
  if (rows >= 1 && rows <= 8)
    return launch_stream_cfg<D, Cfg<1, 1, 4, 3>, KV8>(tk, tv, p, max_units, always, s, launched);
  if (rows >= 17 && rows <= 24)
    return launch_stream_cfg<D, Cfg<1, 3, 2, 2, 2>, KV8>(tk, tv, p, max_units, always, s,
                                                          launched);
  return cudaSuccess;
}

}  // namespace pa
