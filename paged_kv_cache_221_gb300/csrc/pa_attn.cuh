// Paged decode / verify attention kernel template (sm_103a).
//
// One CTA owns one work unit: (partition of one sequence's pages, kv head) in
// the per-sequence mode, or (partition of a group's shared prefix pages, kv
// head, chunk of group members) in the shared-prefix mode.  The block table
// is resolved on the fly: a producer warp reads the physical block id of each
// logical page and issues two-dimensional TMA loads of the K page and the V
// page (block_size x head_dim bf16 each, contiguous in the pool) into a ring
// of kStages shared-memory stages with 128-byte swizzle.  Consumer warps then
// compute, per page, the scores of all query rows that read this kv head (the
// GQA group x the query tokens, and in shared-prefix mode x the members) on
// the tensor cores, an online softmax in fp32, and the P.V accumulation on the
// tensor cores with P split into two bf16 halves so that P keeps ~16
// significant bits.  Each page is read from HBM once per CTA.
//
// Tile orientation: tokens are the M dimension of the score tile
// (S^T[16 tokens x 8 rows] = K_page[16 x D] . Q^T[D x 8]) and head dims are the
// M dimension of the output tile (O^T[D x 8] += V_page^T[D x 16] . P^T[16 x 8]),
// so a 16-token page is exactly one m16n8k16 step and the query rows of the
// CTA (1 .. 64) fill the N side in n-tiles of 8.  A consumer warp carries NT
// n-tiles, so it reads each K/V page from shared memory once for up to 32 rows;
// NTW warp columns split larger row sets, and PL page lanes split the pages.
//
// FP8 pages (KV8): K pages hold E4M3 codes token-major ([16][D] bytes), V pages
// hold them transposed ([D][16] bytes), with one dequantisation scale per kv
// head for K and for V.  Codes are widened to f16 in registers (exact) and the
// products run on the f16 tensor-core path with fp32 accumulation: Q is
// converted to f16 once per CTA (stored in shared memory in the head-dim order
// of the K bytes), P is one f16 operand (11 significant bits),
// the K scale folds into the softmax scale and the V scale into the output.
// The contraction order inside a 16-wide k step is free, so the operands are
// fed in the order the byte layout delivers them: K rows are fed in the token
// order sigma (below) so that P^T lands in the B registers in the same order
// as the transposed V bytes land in the A registers, and Q is fed in the same
// head-dim order as the K bytes.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include <atomic>
#include <climits>
#include <type_traits>

#include "pa_ptx.cuh"

namespace pa {

template <int D, bool KV8 = false>
struct Geo {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  // A ring stage holds kPPS consecutive pages of the unit: their K pages, then
  // their V pages.  FP8 pages are half the bytes of bf16 pages, so a stage holds
  // two of them and the ring moves the same bytes per barrier round trip.
  static constexpr int kPPS = KV8 ? 2 : 1;              // pages per ring stage
  static constexpr int kNS = kStages;                   // ring stages
  static constexpr int kIssueGroup = 4;                 // stages the producer issues at once
  static constexpr int kHalves = D / 64;                // bf16: 128-byte swizzle rows per token
  static constexpr int kHalfBytes = kBlockSize * 128;   // bf16: one 16 x 64 TMA box
  static constexpr int kPageBytes = kBlockSize * D * (KV8 ? 1 : 2);
  static constexpr int kStageBytes = 2 * kPPS * kPageBytes;
  static constexpr int kQStride = D + 8;                // bf16 per Q row in smem (conflict-free)
  static constexpr int kOStride = D + 4;                // floats per merge row (conflict-free)
  static constexpr int kKSteps = D / 16;
};

// Consumer-warp layout: NT n-tiles of 8 query rows per warp, NTW warp columns
// (rows 8*NT*NTW per CTA), PL page lanes (warps of one column that split the
// pages), and the CTAs per SM the register budget must allow.
// TP: ring stages per softmax step of a consumer warp (2 needs at least four
// ring stages per page lane: two in use, two in flight).  FP8 pages take one
// stage (two pages) per step whatever TP says.
template <int NT_, int NTW_, int PL_, int MINB_, int TP_ = 1>
struct Cfg {
  static constexpr int NT = NT_, NTW = NTW_, PL = PL_, MINB = MINB_, TP = TP_;
  static constexpr int kThreads = (NTW * PL + 1) * 32;
  static_assert(TP == 1 || TP == 2, "one or two pages per softmax step");
};

template <int D, int NT, int NTW, bool KV8 = false>
struct Smem {
  using Gm = Geo<D, KV8>;
  static constexpr int kRows = 8 * NT * NTW;
  static constexpr int kStagesOff = 0;
  static constexpr int kQOff = Gm::kNS * Gm::kStageBytes;
  static constexpr int kLimOff = kQOff + kRows * Gm::kQStride * 2;
  static constexpr int kBarOff = (kLimOff + kRows * 4 + 7) / 8 * 8;
  static constexpr int kOkOff = kBarOff + 2 * Gm::kNS * 8;
  static constexpr int kMemOff = kOkOff + Gm::kNS * 4;
  static constexpr int kBytes = kMemOff + kMaxRows * 4;
  static constexpr int kAlloc = kBytes + 1024;          // room to align the base to 1 KB
  // merge buffer of one (page lane, warp column): m[8NT], l[8NT], O[8NT][kOStride]
  // (reuses the stage ring once every page is consumed)
  static constexpr int kMergeFloats = 16 * NT + 8 * NT * Gm::kOStride;
};

// Byte offset of 16-byte chunk `ch` (of D/8) of token row `tok` inside one
// swizzled page: two-dimensional TMA boxes of 16 rows x 128 bytes, 16-byte
// chunk c of row r stored at chunk c ^ (r % 8).
__device__ __forceinline__ uint32_t page_off(int tok, int ch) {
  return static_cast<uint32_t>((ch >> 3) * (kBlockSize * 128) + tok * 128 +
                               (((ch & 7) ^ (tok & 7)) << 4));
}

// FP8 K page: 16 rows of D bytes, one TMA box, 128-byte swizzle at D = 128
// (16-byte chunk c of row r at chunk c ^ (r % 8)), unswizzled at D = 64.
template <int D>
__device__ __forceinline__ uint32_t page8_off(int tok, int ch) {
  if constexpr (D == 128)
    return static_cast<uint32_t>(tok * 128 + ((ch ^ (tok & 7)) << 4));
  else
    return static_cast<uint32_t>(tok * D + (ch << 4));
}

// FP8 score-tile row m holds token sigma(m): rows 0-7 tokens 0,1,4,5,8,9,12,13
// and rows 8-15 tokens 2,3,6,7,10,11,14,15.  After the P^T transpose lane
// (gid, q) then holds tokens 4q, 4q+1 in its first B register and 4q+2, 4q+3 in
// its second, which is the order of bytes 4q .. 4q+3 of a transposed V row.
__device__ __forceinline__ int sigma_row(int m) {
  return 4 * ((m & 7) >> 1) + (m & 1) + 2 * (m >> 3);
}

// One consumer step: the score tiles of TP staged pages (K_page . Q^T per page
// and n-tile), one online-softmax update of the warp's rows over all of them,
// and the P.V accumulation of every page into the output tile.  okp[k] false
// means page k is absent (its scores are -inf, it adds nothing).
template <int D, int NT, int TP, bool KV8>
struct StepState {
  float acc[NT][D / 16][4];
  float m0[NT], m1[NT], l0[NT], l1[NT];
};

template <int D, int NT, int TP, bool KV8, bool kQRegs>
__device__ __forceinline__ void attend_step(
    StepState<D, NT, TP, KV8>& st, const bool (&okp)[TP], const uint32_t (&kb)[TP],
    const uint32_t (&vb)[TP], const int (&tok0)[TP],
    const uint32_t (&qf)[kQRegs ? NT : 1][kQRegs ? D / 16 : 1][2], uint32_t qrow,
    const uint32_t (&koff)[4], const uint32_t (&voff)[4], const int (&lim0)[NT],
    const int (&lim1)[NT], int minlim, int vlen, float sl2, int srow0, int srow1, int q4,
    const AttnParams& p) {
  using Gm = Geo<D, KV8>;
  auto& acc = st.acc;
  auto& m0 = st.m0;
  auto& m1 = st.m1;
  auto& l0 = st.l0;
  auto& l1 = st.l1;
  // S^T[16 tokens x 8 rows] = K_page . Q^T per page and n-tile (two chains each)
  float sa[TP][NT][4], sb[TP][NT][4];
#pragma unroll
  for (int k = 0; k < TP; ++k)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) sa[k][j][e] = sb[k][j][e] = 0.f;
#pragma unroll
  for (int k = 0; k < TP; ++k) {
    if (!okp[k]) continue;
    if constexpr (KV8) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(r0, r1, r2, r3, kb[k] + koff[c]);
        const uint32_t a00 = e4m3x2_to_f16x2(r0), a02 = e4m3x2_to_f16x2(r0 >> 16);
        const uint32_t a01 = e4m3x2_to_f16x2(r1), a03 = e4m3x2_to_f16x2(r1 >> 16);
        const uint32_t a10 = e4m3x2_to_f16x2(r2), a12 = e4m3x2_to_f16x2(r2 >> 16);
        const uint32_t a11 = e4m3x2_to_f16x2(r3), a13 = e4m3x2_to_f16x2(r3 >> 16);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          uint32_t b00, b01, b10, b11;
          if constexpr (kQRegs) {
            b00 = qf[j][2 * c][0];
            b01 = qf[j][2 * c][1];
            b10 = qf[j][2 * c + 1][0];
            b11 = qf[j][2 * c + 1][1];
          } else {
            ldsm_x4(b00, b01, b10, b11,
                    qrow + static_cast<uint32_t>(j * 8 * Gm::kQStride * 2 + 2 * c * 32));
          }
          mma_f16_16816(sa[k][j], a00, a01, a02, a03, b00, b01);
          mma_f16_16816(sb[k][j], a10, a11, a12, a13, b10, b11);
        }
      }
    } else {
#pragma unroll
    for (int k2 = 0; k2 < Gm::kKSteps; k2 += 2) {
      uint32_t a[2][4];
      ldsm_x4(a[0][0], a[0][1], a[0][2], a[0][3],
              kb[k] + (k2 >> 2) * Gm::kHalfBytes + koff[k2 & 3]);
      ldsm_x4(a[1][0], a[1][1], a[1][2], a[1][3],
              kb[k] + ((k2 + 1) >> 2) * Gm::kHalfBytes + koff[(k2 + 1) & 3]);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        uint32_t b00, b01, b10, b11;
        if constexpr (kQRegs) {
          b00 = qf[j][k2][0];
          b01 = qf[j][k2][1];
          b10 = qf[j][k2 + 1][0];
          b11 = qf[j][k2 + 1][1];
        } else {
          ldsm_x4(b00, b01, b10, b11,
                  qrow + static_cast<uint32_t>(j * 8 * Gm::kQStride * 2 + k2 * 32));
        }
        mma_bf16_16816(sa[k][j], a[0][0], a[0][1], a[0][2], a[0][3], b00, b01);
        mma_bf16_16816(sb[k][j], a[1][0], a[1][1], a[1][2], a[1][3], b10, b11);
      }
    }
    }
  }

  // V rows at or past the context end may hold anything (even NaN): their
  // weight is 0, but 0 * NaN is NaN, so zero them in the operand.
  int nvalid[TP];
  bool interior[TP];
  uint32_t mlo[TP], mhi[TP];
#pragma unroll
  for (int k = 0; k < TP; ++k) {
    nvalid[k] = vlen - tok0[k];
    interior[k] = okp[k] && (tok0[k] + kBlockSize - 1 <= minlim) &&
                  (tok0[k] + p.wspan >= vlen) && (nvalid[k] >= kBlockSize);
    mlo[k] = mhi[k] = 0xffffffffu;
    if (nvalid[k] < kBlockSize) {
      const int nv = nvalid[k];
      // tokens behind the low / high halves of the first and second A register pairs
      const int t0 = KV8 ? 4 * q4 : 2 * q4, t2 = KV8 ? 4 * q4 + 2 : 2 * q4 + 8;
      mlo[k] = (t0 < nv ? 0x0000ffffu : 0u) | (t0 + 1 < nv ? 0xffff0000u : 0u);
      mhi[k] = (t2 < nv ? 0x0000ffffu : 0u) | (t2 + 1 < nv ? 0xffff0000u : 0u);
    }
  }

  uint32_t bh0[TP][NT], bh1[TP][NT], bl0[TP][NT], bl1[TP][NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    // lane holds S^T[j0][n], S^T[j0][n+1], S^T[j0+8][n], S^T[j0+8][n+1] of each
    // page, n = rbase + 8j + 2q4 (t[k][0..3] in that order)
    float t[TP][4];
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int k = 0; k < TP; ++k) {
#pragma unroll
      for (int e = 0; e < 4; ++e) t[k][e] = (sa[k][j][e] + sb[k][j][e]) * sl2;
      if (!okp[k]) {
        t[k][0] = t[k][1] = t[k][2] = t[k][3] = -CUDART_INF_F;
      } else if (!interior[k]) {
        const int j0 = tok0[k] + srow0, j1 = tok0[k] + srow1;
        const unsigned u0 = static_cast<unsigned>(j0), u1 = static_cast<unsigned>(j1);
        t[k][0] = (static_cast<unsigned>(lim0[j]) - u0 < p.wcap) ? t[k][0] : -CUDART_INF_F;
        t[k][1] = (static_cast<unsigned>(lim1[j]) - u0 < p.wcap) ? t[k][1] : -CUDART_INF_F;
        t[k][2] = (static_cast<unsigned>(lim0[j]) - u1 < p.wcap) ? t[k][2] : -CUDART_INF_F;
        t[k][3] = (static_cast<unsigned>(lim1[j]) - u1 < p.wcap) ? t[k][3] : -CUDART_INF_F;
      }
      mx0 = fmaxf(mx0, fmaxf(t[k][0], t[k][2]));
      mx1 = fmaxf(mx1, fmaxf(t[k][1], t[k][3]));
    }

    // online softmax (log2 domain), statistics per row.  The reference max m
    // only moves when a score exceeds it by more than 8 (so every weight
    // 2^(t - m) stays <= 256); the accumulators are rescaled only then.
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const bool up0 = mx0 > m0[j] + 8.f, up1 = mx1 > m1[j] + 8.f;
    if (__any_sync(0xffffffffu, up0 || up1)) {
      const float al0 = up0 ? hw_exp2(m0[j] - mx0) : 1.f;
      const float al1 = up1 ? hw_exp2(m1[j] - mx1) : 1.f;
      if (up0) m0[j] = mx0;
      if (up1) m1[j] = mx1;
      l0[j] *= al0;
      l1[j] *= al1;
#pragma unroll
      for (int mt = 0; mt < Gm::kKSteps; ++mt) {
        acc[j][mt][0] *= al0;
        acc[j][mt][1] *= al1;
        acc[j][mt][2] *= al0;
        acc[j][mt][3] *= al1;
      }
    }
    const float mu0 = (m0[j] == -CUDART_INF_F) ? 0.f : m0[j];
    const float mu1 = (m1[j] == -CUDART_INF_F) ? 0.f : m1[j];
#pragma unroll
    for (int k = 0; k < TP; ++k) {
      const float p0 = hw_exp2(t[k][0] - mu0), p1 = hw_exp2(t[k][1] - mu1);
      const float p2 = hw_exp2(t[k][2] - mu0), p3 = hw_exp2(t[k][3] - mu1);
      l0[j] += p0 + p2;
      l1[j] += p1 + p3;
      if constexpr (KV8) {
        // P^T as one f16 B operand (transposed 8x8 blocks)
        bh0[k][j] = movmatrix_trans(half2_bits(__floats2half2_rn(p0, p1)));
        bh1[k][j] = movmatrix_trans(half2_bits(__floats2half2_rn(p2, p3)));
        continue;
      }
      // P^T as B operands: bf16 high part and bf16 residual, transposed 8x8 blocks
      const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1);
      const __nv_bfloat162 h23 = __floats2bfloat162_rn(p2, p3);
      const float2 f01 = __bfloat1622float2(h01);
      const float2 f23 = __bfloat1622float2(h23);
      const __nv_bfloat162 r01 = __floats2bfloat162_rn(p0 - f01.x, p1 - f01.y);
      const __nv_bfloat162 r23 = __floats2bfloat162_rn(p2 - f23.x, p3 - f23.y);
      bh0[k][j] = movmatrix_trans(bf162_bits(h01));
      bh1[k][j] = movmatrix_trans(bf162_bits(h23));
      bl0[k][j] = movmatrix_trans(bf162_bits(r01));
      bl1[k][j] = movmatrix_trans(bf162_bits(r23));
    }
  }

  // O^T[D x 8] += V_page^T . P^T per page and n-tile
#pragma unroll
  for (int k = 0; k < TP; ++k) {
    if (!okp[k]) continue;
    auto pv = [&](auto tail) {
      if constexpr (KV8) {
        // transposed V: rows are head dims; ldmatrix c covers dims 32c .. 32c+31
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(r0, r1, r2, r3, vb[k] + voff[c]);
          uint32_t a[2][4];
          a[0][0] = e4m3x2_to_f16x2(r0);
          a[0][2] = e4m3x2_to_f16x2(r0 >> 16);
          a[0][1] = e4m3x2_to_f16x2(r1);
          a[0][3] = e4m3x2_to_f16x2(r1 >> 16);
          a[1][0] = e4m3x2_to_f16x2(r2);
          a[1][2] = e4m3x2_to_f16x2(r2 >> 16);
          a[1][1] = e4m3x2_to_f16x2(r3);
          a[1][3] = e4m3x2_to_f16x2(r3 >> 16);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if constexpr (decltype(tail)::value) {
              a[h][0] &= mlo[k];
              a[h][1] &= mlo[k];
              a[h][2] &= mhi[k];
              a[h][3] &= mhi[k];
            }
#pragma unroll
            for (int j = 0; j < NT; ++j)
              mma_f16_16816(acc[j][2 * c + h], a[h][0], a[h][1], a[h][2], a[h][3],
                            bh0[k][j], bh1[k][j]);
          }
        }
      } else {
#pragma unroll
      for (int mt = 0; mt < Gm::kKSteps; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(a0, a1, a2, a3, vb[k] + (mt >> 2) * Gm::kHalfBytes + voff[mt & 3]);
        if constexpr (decltype(tail)::value) {
          a0 &= mlo[k];
          a1 &= mlo[k];
          a2 &= mhi[k];
          a3 &= mhi[k];
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          mma_bf16_16816(acc[j][mt], a0, a1, a2, a3, bh0[k][j], bh1[k][j]);
          mma_bf16_16816(acc[j][mt], a0, a1, a2, a3, bl0[k][j], bl1[k][j]);
        }
      }
      }
    };
    if (nvalid[k] < kBlockSize)
      pv(std::true_type{});
    else
      pv(std::false_type{});
  }
}

template <int D, class C, bool GROUP, bool KV8>
__global__ void __launch_bounds__(C::kThreads, C::MINB)
    paged_attn_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
  constexpr int NT = C::NT, NTW = C::NTW, PL = C::PL;
  constexpr int NCW = NTW * PL;              // consumer warps
  constexpr int NCT = NCW * 32;              // consumer threads
  using Gm = Geo<D, KV8>;
  using Sm = Smem<D, NT, NTW, KV8>;
  constexpr int NS = Gm::kNS;
  constexpr int PPS = Gm::kPPS;              // pages per ring stage
  constexpr int TPI = KV8 ? 1 : C::TP;       // ring stages per consumer step
  constexpr int TP = TPI * PPS;              // pages per consumer step
  static_assert(NS % PL == 0, "each stage is always consumed by the same page lane");
  static_assert(PL * NTW * Sm::kMergeFloats * 4 <= NS * Gm::kStageBytes,
                "merge buffers fit in the stage ring");
  static_assert(TPI == 1 || NS / PL >= 4, "ring too short for two stages per step");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem + Sm::kStagesOff;
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem + Sm::kQOff);
  int* lim = reinterpret_cast<int*>(smem + Sm::kLimOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sm::kBarOff);
  uint64_t* empty = full + NS;
  int* stage_ok = reinterpret_cast<int*>(smem + Sm::kOkOff);
  int* members = reinterpret_cast<int*>(smem + Sm::kMemOff);
  __shared__ int s_nmem;
  __shared__ int s_bad;

  // The kernel launched next may start once every CTA of this grid has started:
  // the per-sequence kernel of the same call after the shared-prefix kernel, the
  // split-KV merge (which waits for this grid's completion) after the per-sequence one.
  grid_launch_dependents();
  if (!GROUP && blockIdx.x == gridDim.x - 1) {
    // When launched alongside a shared-prefix kernel, this grid must not
    // complete before it (the split-KV merge that follows reads both).
    grid_dependency_wait();
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Per-sequence mode: a 1-D grid in partition-major order (every sequence's
  // first partition, then every second one, ...) so that the short, ragged last
  // partitions are dispatched last.  Shared-prefix mode: (partition, head, group chunk).
  const int unit_p = GROUP ? static_cast<int>(blockIdx.x)
                           : static_cast<int>(blockIdx.x / (p.Hkv * p.num_seqs));
  const int g = GROUP ? static_cast<int>(blockIdx.y) : static_cast<int>(blockIdx.x % p.Hkv);
  const int G = p.G, T = p.T;

  // ------------------------------------------------------------------ unit
  int pg0, pg1, slot, nrows, vlen;
  bool direct;
  int b_single = 0;                          // per-sequence mode: the sequence
  if constexpr (!GROUP) {
    const int b = static_cast<int>((blockIdx.x / p.Hkv) % p.num_seqs);
    const int L = p.context_lens[b];
    const int pre = (p.seq_group != nullptr && p.seq_group[b] >= 0)
                        ? p.group_prefix_blocks[p.seq_group[b]] : 0;
    if (L < T || L > p.max_ctx || pre < 0 || pre > p.max_prefix_blocks ||
        pre * kBlockSize > L) {
      if (threadIdx.x == 0 && unit_p == 0) atomicOr(&g_pa_err, kErrBounds);
      return;
    }
    const int nblk = (L + kBlockSize - 1) / kBlockSize;
    // With a sliding window, blocks wholly before the first query's window are skipped.
    const int first = p.window > 0 ? max(pre, max(0, L - T - p.window + 1) / kBlockSize) : pre;
    pg0 = first + unit_p * p.ppb;
    if (pg0 >= nblk) return;                 // partition past this sequence's end
    pg1 = min(pg0 + p.ppb, nblk);
    const int npre = (pre + p.ppb - 1) / p.ppb;
    const int nparts = npre + (nblk - first + p.ppb - 1) / p.ppb;
    slot = npre + unit_p;
    direct = (pre == 0 && nparts == 1);
    nrows = G * T;
    vlen = L;
    b_single = b;
  } else {
    const int gi = blockIdx.z / p.num_chunks;
    const int chunk = blockIdx.z % p.num_chunks;
    const int pre = p.group_prefix_blocks[gi];
    if (pre < 0 || pre > p.max_prefix_blocks) {
      if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(&g_pa_err, kErrBounds);
      return;
    }
    pg0 = blockIdx.x * p.ppb;
    if (pg0 >= pre) return;
    pg1 = min(pg0 + p.ppb, pre);
    slot = blockIdx.x;
    direct = false;
    vlen = 0x7fffffff;                       // prefix pages are full blocks
    const int mc = p.members_per_chunk;
    if (warp == 0) {
      // Members of group gi in ascending sequence order; keep ranks
      // [chunk*mc, chunk*mc + mc).
      int cnt = 0, bad = 0;
      for (int base = 0; base < p.num_seqs; base += 32) {
        const int b = base + lane;
        const bool is = b < p.num_seqs && p.seq_group[b] == gi;
        const unsigned bal = __ballot_sync(0xffffffffu, is);
        if (is) {
          const int r = cnt + __popc(bal & ((1u << lane) - 1)) - chunk * mc;
          if (r >= 0 && r < mc) {
            members[r] = b;
            const int L = p.context_lens[b];
            if (L < T || L > p.max_ctx || L < pre * kBlockSize ||
                (p.new_k != nullptr && L - T < pre * kBlockSize))
              bad = 1;
          }
        }
        cnt += __popc(bal);
      }
      bad = __any_sync(0xffffffffu, bad);
      if (lane == 0) {
        s_nmem = max(0, min(mc, cnt - chunk * mc));
        s_bad = bad;
        if (bad && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(&g_pa_err, kErrBounds);
      }
    }
    __syncthreads();
    if (s_bad || s_nmem == 0) return;
    nrows = s_nmem * G * T;
  }

  // ------------------------------------------------------------------ setup
  const int npages = pg1 - pg0;
  const int nitems = (npages + PPS - 1) / PPS;   // ring stages the unit fills
  const int32_t* trow =
      p.block_tables + static_cast<size_t>(GROUP ? members[0] : b_single) * p.mbs;
  int phys_first = 0;                        // first 32 block ids, loaded before the sync
  if (warp == NCW) {
    if (lane < npages) phys_first = __ldg(trow + pg0 + lane);
    if (lane == 0) {
      tma_prefetch_map(&tmk);
      tma_prefetch_map(&tmv);
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NTW);
    }
    fence_barrier_init();
  }
  __syncthreads();                           // barriers initialised before anyone uses them

  // ------------------------------------------------------------------ producer
  // Starts streaming pages at once; the consumers gather the query rows meanwhile.
  // Stages are issued in groups of GP: lane j of the group waits for its own
  // stage and issues its own page(s), so one pass of the loop puts GP stages in
  // flight (the per-stage cost of waiting and issuing is paid once per group).
  if (warp == NCW) {
    constexpr int GP = Gm::kIssueGroup;
    constexpr int IPB = 32 / PPS;             // stages per batch of 32 block ids
    static_assert(GP >= 1 && GP <= NS && IPB % GP == 0, "issue group");
    bool aborted = false;
    // Query tokens' K/V that land in this unit's pages are stored into the pool
    // first (reshape_and_cache fused; FP8 pages quantise on the way).  The stores
    // are issued once the first group of pages is in flight (before it, if that
    // group holds a new token), and the proxy fence only right before the first
    // page that holds a new token is issued, so the stores have long landed and
    // neither the stores nor the fence stall the stream.
    int fence_at = npages;                    // first unit page that holds a new token
    int jlo = npages, jhi = -1;               // unit pages that hold new tokens
    if constexpr (!GROUP) {
      if (p.new_k != nullptr) {
        jlo = max(0, (vlen - T) / kBlockSize - pg0);
        jhi = min(npages - 1, (vlen - 1) / kBlockSize - pg0);
      }
    }
    bool pending = jlo <= jhi;
    auto store_new_tokens = [&]() {
      for (int j = jlo; j <= jhi; ++j) {
        const int phys = __ldg(trow + pg0 + j);
        const int pos0 = (pg0 + j) * kBlockSize;
        const int lo = max(vlen - T, pos0), hi = min(vlen - 1, pos0 + kBlockSize - 1);
        if (lo > hi || static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks))
          continue;                           // out-of-range ids are reported when issued
        fence_at = min(fence_at, j);
        for (int pos = lo; pos <= hi; ++pos) {
          const size_t src = (static_cast<size_t>(b_single) * T + (pos - (vlen - T))) * p.Hkv + g;
          const size_t page = static_cast<size_t>(phys) * p.Hkv + g;
          const int off = pos & (kBlockSize - 1);
          if constexpr (KV8) {
            // lane c: head dims 4c .. 4c+3; K row bytes contiguous, V bytes one per
            // transposed row
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
            constexpr int CH = D / 8;           // 16-byte chunks per row
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
    for (int base = 0; base < npages; base += 32) {
      const int phys_l = base == 0 ? phys_first
                                   : ((base + lane < npages) ? __ldg(trow + pg0 + base + lane) : 0);
      const int cnt = min(32, npages - base);
      const int icnt = (cnt + PPS - 1) / PPS;   // stages of this batch
      // lane i takes pages base + PPS*i .. base + PPS*i + PPS - 1 (lanes below IPB)
      int phys_a = phys_l, phys_b = 0;
      if constexpr (PPS == 2) {
        phys_a = __shfl_sync(0xffffffffu, phys_l, (2 * lane) & 31);
        phys_b = __shfl_sync(0xffffffffu, phys_l, (2 * lane + 1) & 31);
      }
      for (int j0 = 0; j0 < icnt; j0 += GP) {
        const int jn = min(j0 + GP, icnt);
        if (min(npages, base + PPS * jn) > fence_at) {
          // the stores must be visible to the TMA reads of the pages that hold them
          fence_proxy_async_global();
          __syncwarp();
          fence_at = npages;
        }
        if (lane >= j0 && lane < jn) {
          const int it = base / PPS + lane;
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
              // K pages at 0 and kPageBytes, V pages at 2 and 3 kPageBytes
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
        // a wait that gave up on any lane ends the streaming of the whole warp
        aborted = __any_sync(0xffffffffu, aborted);
        if (pending) store_new_tokens();            // the first group is in flight
      }
    }
    // Do not leave while copies issued by this warp may still be landing.
    if (lane == 0) {
      for (int it = max(0, nitems - NS); it < nitems; ++it)
        mbar_wait(&full[it % NS], static_cast<uint32_t>(it / NS) & 1u, p.timeout_ns);
    }
    return;
  }

  // ------------------------------------------------------------------ query rows
  {
    // Gather the query rows of this unit into smem (zero rows pad to 8*NTW).
    constexpr int CH = D / 8;                 // 16-byte chunks per row
    for (int idx = threadIdx.x; idx < Sm::kRows * CH; idx += NCT) {
      const int n = idx / CH, ch = idx % CH;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (n < nrows) {
        const int m = n / (G * T), t = (n / G) % T, hl = n % G;
        const int b = GROUP ? members[m] : b_single;
        const size_t row = (static_cast<size_t>(b) * T + t) * p.Hq + g * G + hl;
        v = reinterpret_cast<const uint4*>(p.q)[row * CH + ch];
      }
      if constexpr (KV8) {
        // f16, and inside every 16 dims in the order of the FP8 K bytes: dims
        // 4q, 4q+1 at positions 2q, 2q+1 and dims 4q+2, 4q+3 at 2q+8, 2q+9, so
        // that the usual B-operand ldmatrix hands lane q the dims its K bytes hold.
        uint32_t* dst = reinterpret_cast<uint32_t*>(qs + n * Gm::kQStride + (ch >> 1) * 16 +
                                                    4 * (ch & 1));
        dst[0] = bf16x2_to_f16x2(v.x);        // dims 8h, 8h+1      -> 4h, 4h+1
        dst[4] = bf16x2_to_f16x2(v.y);        // dims 8h+2, 8h+3    -> 4h+8, 4h+9
        dst[1] = bf16x2_to_f16x2(v.z);        // dims 8h+4, 8h+5    -> 4h+2, 4h+3
        dst[5] = bf16x2_to_f16x2(v.w);        // dims 8h+6, 8h+7    -> 4h+10, 4h+11
      } else {
        *reinterpret_cast<uint4*>(qs + n * Gm::kQStride + ch * 8) = v;
      }
    }
    for (int n = threadIdx.x; n < Sm::kRows; n += NCT) {
      // Padding rows (query 0) see every position: their columns of the tiles
      // are never written out, and treating them as unmasked lets interior
      // pages skip masking altogether.
      int lm = 0x7fffffff;
      if (n < nrows) {
        const int m = n / (G * T), t = (n / G) % T;
        lm = (GROUP ? p.context_lens[members[m]] : vlen) - T + t;
      }
      lim[n] = lm;
    }
    named_bar_sync(1, NCT);
  }

  // ------------------------------------------------------------------ consumers
  const int col = warp % NTW;                // rows 8*NT*col .. 8*NT*(col+1)-1
  const int pl = warp / NTW;                 // page lane: pages pl, pl+PL, ...
  const int gid = lane >> 2, q4 = lane & 3;
  const int rbase = 8 * NT * col;
  float sl2 = p.scale_log2;
  float out_scale = 1.f;
  if constexpr (KV8) {
    sl2 *= p.k_scale[g];
    out_scale = p.v_scale[g];
  }
  int lim0[NT], lim1[NT];                    // this lane's rows rbase+8j+2q4 (+1)
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    lim0[j] = lim[rbase + 8 * j + 2 * q4];
    lim1[j] = lim[rbase + 8 * j + 2 * q4 + 1];
  }
  // Position j is visible to a row with last position lim iff 0 <= lim - j < p.wcap:
  // wcap is the window, or 2^31 (every earlier position) without one.  Padding
  // rows (lim = INT_MAX) then see everything without a window and nothing with
  // one; their columns are never written either way.
  // Q^T B operands: held in registers for NT <= 2, re-read from smem per page otherwise.
  constexpr bool kQRegs = NT <= 2;
  const uint32_t qrow = smem_u32(qs) +
                        static_cast<uint32_t>((rbase + (lane & 7)) * Gm::kQStride * 2 +
                                              (lane >> 3) * 16);
  uint32_t qf[kQRegs ? NT : 1][kQRegs ? Gm::kKSteps : 1][2];
  if constexpr (kQRegs) {
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int ks = 0; ks < Gm::kKSteps; ks += 2)
        ldsm_x4(qf[j][ks][0], qf[j][ks][1], qf[j][ks + 1][0], qf[j][ks + 1][1],
                qrow + static_cast<uint32_t>(j * 8 * Gm::kQStride * 2 + ks * 32));
  }

  StepState<D, NT, TP, KV8> st;
  auto& acc = st.acc;
  auto& m0 = st.m0;
  auto& m1 = st.m1;
  auto& l0 = st.l0;
  auto& l1 = st.l1;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
#pragma unroll
    for (int i = 0; i < Gm::kKSteps; ++i)
      acc[j][i][0] = acc[j][i][1] = acc[j][i][2] = acc[j][i][3] = 0.f;
    m0[j] = m1[j] = -CUDART_INF_F;
    l0[j] = l1[j] = 0.f;
  }
  bool aborted = false;

  // per-lane ldmatrix row/chunk selectors
  const int mi = lane >> 3, rr = lane & 7;
  const int ktok = rr + ((mi & 1) << 3), kch = mi >> 1;     // K: A operand (tokens x dims)
  const int vtok = rr + ((mi >> 1) << 3), vch = mi & 1;     // V: A operand (dims x tokens)
  // Swizzled byte offsets of this lane's ldmatrix rows for 16-byte chunks
  // 2k + sel (k = 0..3) of the first 64 head dims; the second 64 add one box.
  uint32_t koff[4], voff[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if constexpr (KV8) {
      // k: 16-byte chunk pair (2k, 2k+1) = head dims 32k .. 32k+31, rows fed as sigma
      koff[k] = page8_off<D>(sigma_row(ktok), 2 * k + kch);
      voff[k] = static_cast<uint32_t>((32 * k + lane) * 16);   // transposed V: d rows
    } else {
      koff[k] = page_off(ktok, 2 * k + kch);
      voff[k] = page_off(vtok, 2 * k + vch);
    }
  }
  // FP8: tokens of score rows gid and gid + 8
  const int srow0 = KV8 ? sigma_row(gid) : gid;
  const int srow1 = KV8 ? sigma_row(gid + 8) : gid + 8;
  // Smallest visibility limit of this warp's rows: pages wholly below it (and
  // below the context end) need no masking.
  // With a window, pages must also start at or after vlen - window, the first
  // position the sequence's last query token sees (no row's window starts later).
  int minlim = 0x7fffffff;
#pragma unroll
  for (int j = 0; j < NT; ++j) minlim = min(minlim, min(lim0[j], lim1[j]));
  minlim = __reduce_min_sync(0xffffffffu, minlim);

  // Each step handles TPI stages of this lane (it, it + PL, ...), TP pages in
  // all: one score tile per page, one softmax update over all of them, one P.V
  // per page.
  for (int it = pl; it < nitems; it += TPI * PL) {
    int nstep = 1;
    if (TPI == 2 && it + PL < nitems) nstep = 2;
    bool okp[TP];
    uint32_t kb[TP], vb[TP];
    int tok0[TP], sidx[TPI];
#pragma unroll
    for (int k = 0; k < TP; ++k) {
      okp[k] = false;
      kb[k] = vb[k] = 0;
      tok0[k] = 0;
    }
#pragma unroll
    for (int si = 0; si < TPI; ++si) {
      sidx[si] = 0;
      if (si < nstep) {
        const int item = it + si * PL;
        const int s = item % NS;
        const uint32_t ph = static_cast<uint32_t>(item / NS) & 1u;
        if (!aborted && !mbar_wait(&full[s], ph, p.timeout_ns)) aborted = true;
        const bool ok = !aborted && stage_ok[s];
        sidx[si] = s;
        const uint32_t sb = smem_u32(stages + s * Gm::kStageBytes);
#pragma unroll
        for (int u = 0; u < PPS; ++u) {
          const int k = si * PPS + u, pg = item * PPS + u;
          okp[k] = ok && pg < npages;
          kb[k] = sb + u * Gm::kPageBytes;
          vb[k] = sb + (PPS + u) * Gm::kPageBytes;
          tok0[k] = (pg0 + pg) * kBlockSize;
        }
      }
    }

    attend_step<D, NT, TP, KV8, kQRegs>(st, okp, kb, vb, tok0, qf, qrow, koff, voff, lim0, lim1,
                                        minlim, vlen, sl2, srow0, srow1, q4, p);
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int si = 0; si < TPI; ++si)
        if (si < nstep) mbar_arrive(&empty[sidx[si]]);
    }
  }

  // ------------------------------------------------------------------ merge + write
#pragma unroll
  for (int j = 0; j < NT; ++j) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0[j] += __shfl_xor_sync(0xffffffffu, l0[j], o);
      l1[j] += __shfl_xor_sync(0xffffffffu, l1[j], o);
    }
  }
  named_bar_sync(1, NCT);                    // every page consumed: stage ring is free
  {
    float* mbuf = reinterpret_cast<float*>(stages) + (pl * NTW + col) * Sm::kMergeFloats;
    float* ob = mbuf + 16 * NT;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int r0 = 8 * j + 2 * q4;          // row within this warp's 8*NT rows
      if (gid == 0) {
        mbuf[r0] = m0[j];
        mbuf[r0 + 1] = m1[j];
        mbuf[8 * NT + r0] = l0[j];
        mbuf[8 * NT + r0 + 1] = l1[j];
      }
#pragma unroll
      for (int mt = 0; mt < Gm::kKSteps; ++mt) {
        ob[r0 * Gm::kOStride + 16 * mt + gid] = acc[j][mt][0];
        ob[(r0 + 1) * Gm::kOStride + 16 * mt + gid] = acc[j][mt][1];
        ob[r0 * Gm::kOStride + 16 * mt + gid + 8] = acc[j][mt][2];
        ob[(r0 + 1) * Gm::kOStride + 16 * mt + gid + 8] = acc[j][mt][3];
      }
    }
  }
  named_bar_sync(1, NCT);

  const float* mb0 = reinterpret_cast<const float*>(stages);
  for (int idx = threadIdx.x; idx < nrows * (D / 2); idx += NCT) {
    const int n = idx / (D / 2);
    const int d = (idx % (D / 2)) * 2;
    const int c = n / (8 * NT), nn = n % (8 * NT);
    float M = -CUDART_INF_F;
#pragma unroll
    for (int q = 0; q < PL; ++q) M = fmaxf(M, mb0[(q * NTW + c) * Sm::kMergeFloats + nn]);
    float Ls = 0.f, o0 = 0.f, o1 = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int q = 0; q < PL; ++q) {
        const float* mbq = mb0 + (q * NTW + c) * Sm::kMergeFloats;
        const float f = exp2f(mbq[nn] - M);
        Ls += f * mbq[8 * NT + nn];
        o0 += f * mbq[16 * NT + nn * Gm::kOStride + d];
        o1 += f * mbq[16 * NT + nn * Gm::kOStride + d + 1];
      }
    }
    const int m = n / (G * T), t = (n / G) % T, hl = n % G;
    const int b = GROUP ? members[m] : b_single;
    const size_t orow = (static_cast<size_t>(b) * T + t) * p.Hq + g * G + hl;
    if (direct) {
      const float inv = out_scale / Ls;
      reinterpret_cast<__nv_bfloat162*>(p.out)[(orow * D + d) >> 1] =
          __floats2bfloat162_rn(o0 * inv, o1 * inv);
    } else {
      const float inv = Ls > 0.f ? out_scale / Ls : 0.f;
      const size_t pidx = orow * p.max_parts + slot;
      reinterpret_cast<float2*>(p.part_o)[(pidx * D + d) >> 1] = make_float2(o0 * inv, o1 * inv);
      if (d == 0) {
        p.part_ml[pidx] = make_float2(M, Ls);
      }
    }
  }
}

template <int D, class C, bool GROUP, bool KV8>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                       dim3 grid, cudaStream_t s, bool overlap_previous) {
  constexpr int smem = Smem<D, C::NT, C::NTW, KV8>::kAlloc;
  auto kern = paged_attn_kernel<D, C, GROUP, KV8>;
  // The shared-memory attribute is per device: one bit per device (ids below 64)
  // records that it has been set.  Host threads driving different devices may
  // race here; setting the attribute twice is harmless, and a failed attempt
  // records nothing, so the next call tries again.
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
  if (!overlap_previous) {
    kern<<<grid, C::kThreads, smem, s>>>(tk, tv, p);
    return cudaGetLastError();
  }
  // Programmatic stream serialisation: may start while the previous kernel runs.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

// `rows` = query rows per CTA (1..64).  One n-tile per warp keeps registers low
// and many warps resident (latency hiding); warp columns split the rows.
template <int D, bool GROUP, bool KV8 = false>
cudaError_t launch_dispatch(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                            int rows, dim3 grid, cudaStream_t s, bool overlap_previous) {
  const bool o = overlap_previous;
  if (rows <= 0) return cudaErrorInvalidValue;
  if (rows <= 8) return launch_one<D, Cfg<1, 1, 4, 3>, GROUP, KV8>(tk, tv, p, grid, s, o);
  if (rows <= 16) return launch_one<D, Cfg<1, 2, 2, 3>, GROUP, KV8>(tk, tv, p, grid, s, o);
  if (rows <= 24) return launch_one<D, Cfg<1, 3, 2, 2, 2>, GROUP, KV8>(tk, tv, p, grid, s, o);
  if (rows <= 32) return launch_one<D, Cfg<1, 4, 2, 2>, GROUP, KV8>(tk, tv, p, grid, s, o);
  if (rows <= 64) return launch_one<D, Cfg<2, 4, 1, 2>, GROUP, KV8>(tk, tv, p, grid, s, o);
  return cudaErrorInvalidValue;
}

inline cudaError_t take_error_word(unsigned* bits) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_pa_err, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_pa_err, &zero, sizeof(zero));
  *bits |= v;
  return e;
}

}  // namespace pa
