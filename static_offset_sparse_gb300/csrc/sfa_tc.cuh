// Shared pieces of the rung tensor-core kernels (bf16 I/O, G = 4, 8 or 16: the
// query heads of a KV head in groups of 4).
//
// A warp owns 4 consecutive query positions x the 4 query heads of one KV
// group = 16 mma rows (row r = 4 h + p).  Keys are raw RoPE-rotated K' rows
// and raw V rows staged per CTA by TMA as shifted slabs: a stage holds a K'
// region and a V region of two 24-row boxes each (128-byte rows, 128B
// swizzle, rows outside the sequence zero-filled by the TMA unit).
//  * window chunk s_lo (12 distances): rows = positions i0 - 12 - s_lo + r,
//    r < 48; warp w reads rows 4w .. 4w + 15 (16 key columns).
//  * rung pair: box x holds positions i0 - c_x + r, r < 24; B column
//    n = 2 p + e of warp w is row 4w + p + e of the box, so the lane with
//    tig = p holds both raw logits (floor and floor-plus-one) of position p.
#pragma once

#include "sfa_device.cuh"
#include "sfa_launch.cuh"
#include "sfa_mma.cuh"
#include "sfa_tma.cuh"

namespace sfa {

constexpr int kTcTQ = 16;                     // query positions per CTA (four CTAs per SM)
constexpr int kTcWarps = kTcTQ / 4;           // 4 warps
constexpr int kTcThreads = kTcWarps * 32;     // 128
constexpr int kTcBoxRows = 24;                // rows per TMA box (3 KB, 1024-byte multiple)
constexpr int kTcBoxB = kTcBoxRows * 128;
constexpr int kTcRegionB = 2 * kTcBoxB;       // K' (or V) part of a stage
constexpr int kTcStageB = 2 * kTcRegionB;
constexpr int kTcStages = 2;
constexpr int kTcWC = 12;                     // window distances per chunk

// Number of rungs with c <= x (the plan's c are ascending): binary search.
__device__ __forceinline__ int rungs_upto(const Plan& P, int x) {
  int lo = 0, hi = P.n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (P.c[mid] <= x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
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

// Integer rung pairs (w = 0: one row per position and rung): the 8 B columns
// of one tile are (rung x, position p) = (n >> 2, n & 3), raw row 4w + p of
// box x, so one product serves both rungs; the lane of position p's row holds
// rung tig >> 1 at column 2 tig + (p & 1) when tig & 1 == p >> 1.
__device__ __forceinline__ int int_pair_row(int warp) {
  const int n = threadIdx.x & 7;
  return (n >> 2) * kTcBoxRows + 4 * warp + (n & 3);
}

// O[16 x 64] += P[16 x 8] . V[8 keys x 64] (k = 8): P in the C-fragment
// positions of an integer rung pair's tile, V rows as int_pair_row gives them.
__device__ __forceinline__ void pv_tile_k8(const uint32_t* pa, uint32_t region, int row,
                                           float (*o)[4]) {
  const int mi = (threadIdx.x & 31) >> 3;
#pragma unroll
  for (int nd = 0; nd < 8; nd += 4) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(region + swz(row, nd + mi), b0, b1, b2, b3);
    mma_bf16_k8(o[nd], pa, b0);
    mma_bf16_k8(o[nd + 1], pa, b1);
    mma_bf16_k8(o[nd + 2], pa, b2);
    mma_bf16_k8(o[nd + 3], pa, b3);
  }
}

// Issue the TMA loads of group `grp` (a window chunk, then rung pairs) into
// a stage (thread 0 only).  An unpaired rung reloads its partner's slab: its
// probabilities are zero, and the rows stay finite.
//
// skip (test injection only, AttnArgs::debug_skip): issue neither the
// expect_tx nor the loads, so the stage's barrier never completes and its
// consumers' bounded wait runs out with nothing in flight.
__device__ __forceinline__ void tc_issue_group(const CUtensorMap* mk, const CUtensorMap* mv,
                                               const Plan& P, int bg, int i0, int nwc, int nr,
                                               int grp, uint32_t st, uint32_t bar, bool skip) {
  if (skip) return;
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

// Per-CTA query tiles: Q (and dO) of the tile's 16 positions x 4 heads come in
// by one TMA box each, [4 heads][20 rows][128 B] (the 20-row plane stride is
// 4 mod 8, so the 16 rows of a warp's fragments sit on distinct swizzle
// phases); outputs leave through [4 heads][16 rows][128 B] tiles and one TMA
// store each (rows past the sequence end are not written).
constexpr int kTcQRows = 20;
constexpr int kTcQTileB = 4 * kTcQRows * 128;  // 10240, a 1024-byte multiple
constexpr int kTcORows = 16;
// shared memory: [query tiles][stages] from a 1024-aligned base (+ alignment slack)
constexpr size_t kFwdTcSmem = (size_t)kTcQTileB + (size_t)kTcStages * kTcStageB + 1024;
constexpr size_t kBwdQTcSmem = (size_t)3 * kTcQTileB + (size_t)kTcStages * kTcStageB + 1024;

// Barriers: one per stage, then one for the query tiles.  Thread 0 issues
// the query-tile loads (nq boxes from the maps in qmaps, at coordinates
// (0, i0, plane)) and the first stages.
//
// skip_grp: the group whose loads this CTA never issues (test injection
// through AttnArgs::debug_skip, for CTA (0, 0) only), or -1.
__device__ __forceinline__ void tc_start(const CUtensorMap* mk, const CUtensorMap* mv,
                                         const CUtensorMap* const* qmaps, int nq, uint32_t qtile,
                                         int qplane, const Plan& P, int bg, int i0, int nwc, int nr,
                                         int NG, uint32_t sbase, uint64_t* bars, int skip_grp) {
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s <= kTcStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();  // the previous kernel's outputs (K', Q, ...) are complete from here on
  if (threadIdx.x == 0) {
    const uint32_t qb = smem_u32(&bars[kTcStages]);
    mbar_expect_tx(qb, nq * kTcQTileB);
    for (int x = 0; x < nq; ++x) tma_load_3d(qtile + x * kTcQTileB, qmaps[x], 0, i0, qplane, qb);
    for (int s = 0; s < kTcStages && s < NG; ++s)
      tc_issue_group(mk, mv, P, bg, i0, nwc, nr, s, sbase + s * kTcStageB, smem_u32(&bars[s]),
                     s == skip_grp);
  }
}

// Wait (bounded) for the query tiles; uniform across the CTA.
__device__ __forceinline__ bool tc_wait_qtiles(uint64_t* bars, const AttnArgs& a) {
  const bool ok = mbar_wait_bounded(smem_u32(&bars[kTcStages]), 0, a.wait_cycles);
  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) record_status(a.status, SFA_ERR_TIMEOUT);
    return false;
  }
  return true;
}

// The staged loop shared by the forward and the query-side backward: NST
// stages in flight, one mbarrier each, consumed in order; compute(grp, kst,
// vst) runs on every warp.  Returns false (uniformly across the CTA) if a
// wait timed out; the status word then holds SFA_ERR_TIMEOUT.
template <typename ComputeFn>
__device__ __forceinline__ bool tc_run(const CUtensorMap* mk, const CUtensorMap* mv, const Plan& P,
                                       int bg, int i0, int nwc, int nr, int NG, uint32_t sbase,
                                       uint64_t* bars, const AttnArgs& a, int skip_grp,
                                       ComputeFn compute) {
  const int tid = threadIdx.x;
  for (int grp = 0; grp < NG; ++grp) {
    const int s = grp % kTcStages;
    const bool ok = mbar_wait_bounded(smem_u32(&bars[s]), (grp / kTcStages) & 1, a.wait_cycles);
    // One barrier per group: it makes the timeout decision uniform and, as
    // every thread has finished group grp - 1, frees that group's stage.
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        record_status(a.status, SFA_ERR_TIMEOUT);
        for (int g2 = grp; g2 < NG && g2 < grp + kTcStages - 1; ++g2)  // loads still in flight
          mbar_wait_bounded(smem_u32(&bars[g2 % kTcStages]), (g2 / kTcStages) & 1, a.wait_cycles);
      }
      return false;
    }
    if (tid == 0 && grp > 0 && grp - 1 + kTcStages < NG) {
      const int sp = (grp - 1) % kTcStages;
      tc_issue_group(mk, mv, P, bg, i0, nwc, nr, grp - 1 + kTcStages, sbase + sp * kTcStageB,
                     smem_u32(&bars[sp]), grp - 1 + kTcStages == skip_grp);
    }
    const uint32_t kst = sbase + s * kTcStageB;
    compute(grp, kst, kst + kTcRegionB);
  }
  __syncthreads();  // the caller may reuse shared memory
  return true;
}

// The RoPE (cos, sin) pairs a lane's fragments need at position i (pairs
// 16 kk + 2 tig + {0, 1, 8, 9}, kk = 0, 1), as four float4: loaded while the
// query tile is still in flight.
__device__ __forceinline__ void load_frag_rope(const float2* rope, int i, float4* rp) {
  const int tig = threadIdx.x & 3;
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    rp[2 * kk] = __ldg(reinterpret_cast<const float4*>(rope + (int64_t)i * 32 + 16 * kk + 2 * tig));
    rp[2 * kk + 1] = __ldg(reinterpret_cast<const float4*>(rope + (int64_t)i * 32 + 16 * kk + 2 * tig + 8));
  }
}

// A fragments of a warp's 16 rows (row r = 4 h + p: head h, position 4w + p)
// for the 4 k-steps, from a query tile; with transform they are unpacked,
// rotated by the RoPE pairs rp of load_frag_rope (none if rp is nullptr),
// scaled and repacked.
__device__ __forceinline__ void tile_frags(uint32_t tile, int warp, const float4* rp, float scale,
                                           bool transform, uint32_t (*qa)[4]) {
  const int lane = threadIdx.x & 31;
  const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int srow = (r >> 2) * kTcQRows + 4 * warp + (r & 3);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    ldsm_x4(tile + swz(srow, 2 * kk + (lane >> 4)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
  if (!transform) return;
  float x[2][4][4];  // [row gid / gid + 8][kk][dims 2tig, 2tig+1, 2tig+8, 2tig+9]
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const float2 a0 = unpack_bf16(qa[kk][0]), a1 = unpack_bf16(qa[kk][1]);
    const float2 a2 = unpack_bf16(qa[kk][2]), a3 = unpack_bf16(qa[kk][3]);
    x[0][kk][0] = a0.x; x[0][kk][1] = a0.y; x[0][kk][2] = a2.x; x[0][kk][3] = a2.y;
    x[1][kk][0] = a1.x; x[1][kk][1] = a1.y; x[1][kk][2] = a3.x; x[1][kk][3] = a3.y;
  }
  // scale is a power of two (1/8 or 1), so folding it into cos and sin gives
  // the same bits as scaling the rotated values
  if (rp) {
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const float4 a = rp[2 * kk], b = rp[2 * kk + 1];
      const float cs[4] = {a.x * scale, a.z * scale, b.x * scale, b.z * scale};
      const float sn[4] = {a.y * scale, a.w * scale, b.y * scale, b.w * scale};
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = x[rr][kk][e], hi = x[rr][kk + 2][e];
          x[rr][kk][e] = lo * cs[e] - hi * sn[e];
          x[rr][kk + 2][e] = lo * sn[e] + hi * cs[e];
        }
    }
  } else {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[rr][kk][e] *= scale;
  }
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    qa[kk][0] = pack_bf16(x[0][kk][0], x[0][kk][1]);
    qa[kk][1] = pack_bf16(x[1][kk][0], x[1][kk][1]);
    qa[kk][2] = pack_bf16(x[0][kk][2], x[0][kk][3]);
    qa[kk][3] = pack_bf16(x[1][kk][2], x[1][kk][3]);
  }
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}

// Byte address in an output tile of the bf16 pair (dim d, d + 1) of warp row
// r (head r >> 2, position 4w + (r & 3)); d even.
__device__ __forceinline__ uint32_t otile_addr(uint32_t tile, int warp, int r, int d) {
  const int srow = (r >> 2) * kTcORows + 4 * warp + (r & 3);
  return tile + swz(srow, d >> 3) + (d & 7) * 2;
}

// stmatrix: four 8x8 b16 tiles to shared memory (lanes 8t..8t+7 give tile
// t's row addresses; register t holds the lane's pair of tile t, row lane / 4,
// columns 2 (lane % 4), + 1: the mma fragment layout).
__device__ __forceinline__ void stsm_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                        uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(addr),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

// A warp's 16 x 64 rows of an output tile (row r = 4 h + p) from packed bf16
// pairs pk[nd][x]: row gid (x = 0) or gid + 8 (x = 1), dims 8 nd + 2 tig, + 1.
// Four stmatrix, each two 16-row chunks nd, nd + 1.
__device__ __forceinline__ void store_otile(uint32_t tile, int warp, const uint32_t (*pk)[2]) {
  const int lane = threadIdx.x & 31, mi = lane >> 3;
  const int r = 8 * (mi & 1) + (lane & 7);
  const int srow = (r >> 2) * kTcORows + 4 * warp + (r & 3);
#pragma unroll
  for (int nd = 0; nd < 8; nd += 2)
    stsm_x4(tile + swz(srow, nd + (mi >> 1)), pk[nd][0], pk[nd][1], pk[nd + 1][0], pk[nd + 1][1]);
}

// Store an output tile (thread 0; after every thread's fence + a barrier).
__device__ __forceinline__ void tc_store_tile(const CUtensorMap* map, uint32_t tile, int i0,
                                              int plane) {
  tma_store_3d(map, 0, i0, plane, tile);
  bulk_commit();
}

// Host: tensor map over [B*H, T, 64] bf16 rows with a (64, box_rows, box_h)
// box, 128B swizzle unless swizzle is false (sfa_api.cu).
int make_rows_map(CUtensorMap* m, const void* base, int64_t planes, int T, int box_rows, int box_h,
                  bool swizzle = true);
// Host: tensor map over [planes, T, 64] bf16 rows viewed as [planes][T /
// delta][delta][64] (delta divides T): coordinates (dim, residue class,
// compressed index, plane), box (64, 1, box_rows, box_planes), 128B swizzle.
int make_band_map(CUtensorMap* m, const void* base, int64_t planes, int T, int delta, int box_rows,
                  int box_planes);
// Host: tensor map over the key-side coefficient records [planes, T, NS,
// words] (uint32 words), box (words, box_slots, box_q, 1), no swizzle.
int make_coef_map(CUtensorMap* m, const void* base, int64_t planes, int T, int NS, int words,
                  int box_slots, int box_q);

}  // namespace sfa
