// Shared pieces of the tensor-core kernels (bf16 I/O, G = 4).
//
// A warp owns 4 consecutive query positions x the 4 query heads of one KV
// group = 16 mma rows (row r = 4 h + p).  Keys are raw RoPE-rotated K' rows
// and raw V rows staged per CTA by TMA as shifted slabs: a stage holds a K'
// region and a V region of two 40-row boxes each (128-byte rows, 128B
// swizzle, rows outside the sequence zero-filled by the TMA unit).
//  * window chunk s_lo (12 distances): rows = positions i0 - 12 - s_lo + r,
//    r < 80; warp w reads rows 4w .. 4w + 15 (16 key columns).
//  * rung pair: box x holds positions i0 - c_x + r, r < 40; B column
//    n = 2 p + e of warp w is row 4w + p + e of the box, so the lane with
//    tig = p holds both raw logits (floor and floor-plus-one) of position p.
#pragma once

#include "sfa_device.cuh"
#include "sfa_mma.cuh"
#include "sfa_tma.cuh"

namespace sfa {

constexpr int kTcTQ = 32;                     // query positions per CTA (two CTAs per SM)
constexpr int kTcWarps = kTcTQ / 4;           // 8 warps
constexpr int kTcThreads = kTcWarps * 32;     // 256
constexpr int kTcBoxRows = 40;                // rows per TMA box (5 KB, 1024-byte multiple)
constexpr int kTcBoxB = kTcBoxRows * 128;
constexpr int kTcRegionB = 2 * kTcBoxB;       // K' (or V) part of a stage
constexpr int kTcStageB = 2 * kTcRegionB;
constexpr int kTcStages = 5;
constexpr int kTcWC = 12;                     // window distances per chunk
constexpr size_t kFwdTcSmem = (size_t)kTcStages * kTcStageB + 1024;  // + alignment slack

// q' fragments of a warp's 16 rows: rows gid (head gid>>2) and gid+8 (head
// 2 + (gid>>2)), position i, scaled by `scale`; RoPE pairs (d, d + 32) sit in
// k-steps kk and kk + 2 of the same lane.
__device__ __forceinline__ void load_q_frags(const bf16* q0, const bf16* q1, const float2* rope,
                                             int i, float scale, uint32_t (*qa)[4]) {
  const int tig = threadIdx.x & 3;
  float x[2][4][4];  // [row][kk][e]: e = dims 2tig, 2tig+1, 2tig+8, 2tig+9 of k-step kk
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const bf16* q = rr ? q1 : q0;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float2 u = unpack_bf16(*reinterpret_cast<const uint32_t*>(q + 16 * kk + 2 * tig));
      const float2 v = unpack_bf16(*reinterpret_cast<const uint32_t*>(q + 16 * kk + 2 * tig + 8));
      x[rr][kk][0] = u.x;
      x[rr][kk][1] = u.y;
      x[rr][kk][2] = v.x;
      x[rr][kk][3] = v.y;
    }
  }
  if (rope) {
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(rope + (int64_t)i * 32 + 16 * kk + 2 * tig));
      const float4 b = __ldg(reinterpret_cast<const float4*>(rope + (int64_t)i * 32 + 16 * kk + 2 * tig + 8));
      const float cs[4] = {a.x, a.z, b.x, b.z}, sn[4] = {a.y, a.w, b.y, b.w};
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = x[rr][kk][e], hi = x[rr][kk + 2][e];
          x[rr][kk][e] = lo * cs[e] - hi * sn[e];
          x[rr][kk + 2][e] = lo * sn[e] + hi * cs[e];
        }
    }
  }
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    qa[kk][0] = pack_bf16(x[0][kk][0] * scale, x[0][kk][1] * scale);
    qa[kk][1] = pack_bf16(x[1][kk][0] * scale, x[1][kk][1] * scale);
    qa[kk][2] = pack_bf16(x[0][kk][2] * scale, x[0][kk][3] * scale);
    qa[kk][3] = pack_bf16(x[1][kk][2] * scale, x[1][kk][3] * scale);
  }
}

// S[16 x 8] += q' . K'^T for the 8 key rows of a region; lane l supplies
// row `row` (its key column l & 7).
__device__ __forceinline__ void qk_tile(const uint32_t (*qa)[4], uint32_t region, int row, float* s) {
  const int mi = (threadIdx.x & 31) >> 3;
  uint32_t b[8];
  ldsm_x4(region + swz(row, mi), b[0], b[1], b[2], b[3]);
  ldsm_x4(region + swz(row, 4 + mi), b[4], b[5], b[6], b[7]);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) mma_bf16(s, qa[kk], b[2 * kk], b[2 * kk + 1]);
}

// O[16 x 64] += P[16 x 16] . V[16 keys x 64]; lane l supplies the row of key
// (l & 7) of k-half ((l >> 3) & 1): row_lo for keys 0..7, row_hi for 8..15.
__device__ __forceinline__ void pv_tile(const uint32_t* pa, uint32_t region, int row_lo, int row_hi,
                                        float (*o)[4]) {
  const int mi = (threadIdx.x & 31) >> 3;
  const int row = (mi & 1) ? row_hi : row_lo;
#pragma unroll
  for (int nd = 0; nd < 8; nd += 2) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(region + swz(row, nd + (mi >> 1)), b0, b1, b2, b3);
    mma_bf16(o[nd], pa, b0, b1);
    mma_bf16(o[nd + 1], pa, b2, b3);
  }
}

// Issue the TMA loads of group `grp` (a window chunk, then rung pairs) into
// a stage (thread 0 only).  An unpaired rung reloads its partner's slab: its
// probabilities are zero, and the rows stay finite.
__device__ __forceinline__ void tc_issue_group(const CUtensorMap* mk, const CUtensorMap* mv,
                                               const Plan& P, int bg, int i0, int nwc, int nr,
                                               int grp, uint32_t st, uint32_t bar) {
  int y0, y1;
  if (grp < nwc) {
    y0 = i0 - kTcWC - kTcWC * grp;
    y1 = y0 + kTcBoxRows;
  } else {
    const int r0 = 2 * (grp - nwc);
    y0 = i0 - P.c[r0];
    y1 = (r0 + 1 < nr) ? i0 - P.c[r0 + 1] : y0;
  }
  mbar_expect_tx(bar, kTcStageB);
  tma_load_3d(st, mk, 0, y0, bg, bar);
  tma_load_3d(st + kTcBoxB, mk, 0, y1, bg, bar);
  tma_load_3d(st + kTcRegionB, mv, 0, y0, bg, bar);
  tma_load_3d(st + kTcRegionB + kTcBoxB, mv, 0, y1, bg, bar);
}

// The staged pipeline shared by the forward and the query-side backward:
// NST stages in flight, one mbarrier each, consumed in order.  compute(grp,
// kst, vst) runs on every warp.  Returns false (uniformly across the CTA)
// if a wait timed out; the status word then holds SFA_ERR_TIMEOUT.
template <typename ComputeFn>
__device__ __forceinline__ bool tc_pipeline(const CUtensorMap* mk, const CUtensorMap* mv,
                                            const Plan& P, int bg, int i0, int nwc, int nr, int NG,
                                            uint32_t sbase, uint64_t* bars, int* status,
                                            ComputeFn compute) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < kTcStages && s < NG; ++s)
      tc_issue_group(mk, mv, P, bg, i0, nwc, nr, s, sbase + s * kTcStageB, smem_u32(&bars[s]));
  for (int grp = 0; grp < NG; ++grp) {
    const int s = grp % kTcStages;
    const bool ok = mbar_wait_bounded(smem_u32(&bars[s]), (grp / kTcStages) & 1);
    // One barrier per group: it makes the timeout decision uniform and, as
    // every thread has finished group grp - 1, frees that group's stage.
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        record_status(status, SFA_ERR_TIMEOUT);
        for (int g2 = grp; g2 < NG && g2 < grp + kTcStages - 1; ++g2)  // loads still in flight
          mbar_wait_bounded(smem_u32(&bars[g2 % kTcStages]), (g2 / kTcStages) & 1);
      }
      return false;
    }
    if (tid == 0 && grp > 0 && grp - 1 + kTcStages < NG) {
      const int sp = (grp - 1) % kTcStages;
      tc_issue_group(mk, mv, P, bg, i0, nwc, nr, grp - 1 + kTcStages, sbase + sp * kTcStageB,
                     smem_u32(&bars[sp]));
    }
    const uint32_t kst = sbase + s * kTcStageB;
    compute(grp, kst, kst + kTcRegionB);
  }
  __syncthreads();  // the caller may reuse shared memory
  return true;
}

// Host: tensor map over [B*H, T, 64] bf16 rows with a (64, box_rows, box_h)
// box and 128B swizzle (sfa_api.cu).
int make_rows_map(CUtensorMap* m, const void* base, int64_t planes, int T, int box_rows, int box_h);
// Host: tensor map over the key-side coefficient records [B*Hkv, T, NS, 8
// words], box (8, box_slots, box_q, 1), no swizzle.
int make_coef_map(CUtensorMap* m, const void* base, int64_t planes, int T, int NS, int box_slots,
                  int box_q);

}  // namespace sfa
