// Shared pieces of the tensor-core kernels (bf16 I/O, G = 4).
//
// A warp owns 4 consecutive query positions x the 4 query heads of one KV
// group = 16 mma rows (row r = 4 h + p).  Keys are raw RoPE-rotated K' rows
// and raw V rows staged per CTA as shifted slabs: a window chunk covers 12
// distances (16 key columns per warp), a rung slab holds the TQ + 1 rows that
// the floor and floor-plus-one reads of the tile's positions touch.  For a
// rung, B column n = 2 p + e is row p + e of the warp's part of the slab, so
// the lane with tig = p holds both raw logits of position p.
#pragma once

#include "sfa_device.cuh"
#include "sfa_mma.cuh"

namespace sfa {

constexpr int kTcTQ = 64;                  // query positions per CTA
constexpr int kTcWarps = kTcTQ / 4;        // 16 warps
constexpr int kTcThreads = kTcWarps * 32;  // 512
constexpr int kTcRowB = 144;               // smem bytes per staged row (128 + 16 pad)
constexpr int kTcRegion = 2 * (kTcTQ + 1); // rows per K (or V) region of a stage
constexpr int kTcStageB = 2 * kTcRegion * kTcRowB;
constexpr int kTcStages = 3;
constexpr int kTcWC = 12;                  // window distances per chunk (16 key columns)
constexpr size_t kFwdTcSmem = (size_t)kTcStages * kTcStageB;

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

// S[16 x 8] += q' . K'^T for the 8 key rows whose smem row addresses lane
// (l & 7) supplies in `rowaddr` (byte address of the row start).
__device__ __forceinline__ void qk_tile(const uint32_t (*qa)[4], uint32_t rowaddr, float* s) {
  const int mi = (threadIdx.x & 31) >> 3;
  uint32_t b[8];
  ldsm_x4(rowaddr + mi * 16, b[0], b[1], b[2], b[3]);
  ldsm_x4(rowaddr + 64 + mi * 16, b[4], b[5], b[6], b[7]);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) mma_bf16(s, qa[kk], b[2 * kk], b[2 * kk + 1]);
}

// O[16 x 64] += P[16 x 16] . V[16 keys x 64]; lane l supplies the address of
// key row (l & 7) of k-half ((l >> 3) & 1): rowaddr_lo for keys 0..7,
// rowaddr_hi for keys 8..15.
__device__ __forceinline__ void pv_tile(const uint32_t* pa, uint32_t rowaddr_lo, uint32_t rowaddr_hi,
                                        float (*o)[4]) {
  const int mi = (threadIdx.x & 31) >> 3;
  const uint32_t base = (mi & 1) ? rowaddr_hi : rowaddr_lo;
#pragma unroll
  for (int nd = 0; nd < 8; nd += 2) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(base + (nd + (mi >> 1)) * 16, b0, b1, b2, b3);
    mma_bf16(o[nd], pa, b0, b1);
    mma_bf16(o[nd + 1], pa, b2, b3);
  }
}

// Stage one group (a window chunk or a rung pair) of K' and V rows.
//   window chunk s_lo: rows = positions i0 - 12 - s_lo + r, r < 76
//   rung pair r0:      region a (a = 0, 1) rows = positions i0 - c_{r0+a} + r, r < 65
// Rows outside [0, T) (and the second region of an unpaired rung) are zeros.
__device__ __forceinline__ void tc_load_group(const bf16* Kr, const bf16* Vb, const Plan& P, int T,
                                              int i0, int nwc, int nr, int grp, uint32_t kst,
                                              uint32_t vst) {
  const bool win = grp < nwc;
  const int nrows = win ? kTcTQ + kTcWC : kTcRegion;
  const int r0 = 2 * (grp - nwc);
  for (int it = threadIdx.x; it < nrows * 16; it += kTcThreads) {
    const int r = it >> 4, ch = it & 15;
    int pos;
    bool ok;
    if (win) {
      pos = i0 - kTcWC - kTcWC * grp + r;
      ok = true;
    } else {
      const int a = r >= kTcTQ + 1;
      const int rg = r0 + a;
      ok = rg < nr;
      pos = i0 - (ok ? P.c[rg] : 0) + (r - a * (kTcTQ + 1));
    }
    ok = ok && pos >= 0 && pos < T;
    const bf16* src = (ch < 8 ? Kr : Vb) + (ok ? (int64_t)pos * kD : 0) + (ch & 7) * 8;
    const uint32_t dst = (ch < 8 ? kst : vst) + r * kTcRowB + (ch & 7) * 16;
    cp_async16(dst, src, ok ? 16 : 0);
  }
}

}  // namespace sfa
