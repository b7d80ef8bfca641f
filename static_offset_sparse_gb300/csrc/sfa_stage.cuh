// Slab staging shared by the forward and the query-side backward kernels.
//
// Offsets are shared by all queries, so the key/value rows one query tile
// needs through one window chunk or one rung form a contiguous, shifted slab
// of the sequence.  These helpers copy such slabs into shared memory as fp32,
// applying RoPE to K at each row's own position and, for a rung, the two-row
// interpolation (1 - w) row[i - c] + w row[i - c + 1].
#pragma once

#include "sfa_device.cuh"

namespace sfa {

constexpr int kSlab = 144;      // staged rows per tensor (K and V)
constexpr int kWinChunk = 16;   // window distances per batch
constexpr int kMaxBatch = 16;   // slots per batch

// Stage rows [pos_lo, pos_lo + nrows) of K (rotated) and V into sK / sV.
// T and status serve the bounds-checked build only.
template <typename TIO>
__device__ __forceinline__ void stage_rows(const TIO* Kb, const TIO* Vb, const float2* rope,
                                           int pos_lo, int nrows, float* sK, float* sV, int T,
                                           int* status) {
  for (int it = threadIdx.x; it < nrows * 4; it += kThreads) {
    const int r = it >> 2, pc = it & 3;
    const int pos = pos_lo + r;
    if (pos < 0) continue;  // never read: a slot needs i - s >= 0
    if (!dbg_in(pos, T, status) || !dbg_in(r, kSlab, status)) continue;
    float lo[8], hi[8];
    load_pair_chunk(Kb + (int64_t)pos * kD, pc, rope, pos, lo, hi);
    st_smem8(sK + r * kRowPad + 8 * pc, lo);
    st_smem8(sK + r * kRowPad + 32 + 8 * pc, hi);
    load_pair_chunk<TIO>(Vb + (int64_t)pos * kD, pc, nullptr, pos, lo, hi);
    st_smem8(sV + r * kRowPad + 8 * pc, lo);
    st_smem8(sV + r * kRowPad + 32 + 8 * pc, hi);
  }
}

// Stage the rung slabs of rungs r0 .. r0+nb-1 for the tile's TQ positions:
// slab a, row rr holds the interpolated (rotated) K and V row seen by query
// i0 + rr through rung r0 + a.
template <typename TIO, bool INTERP>
__device__ __forceinline__ void stage_rungs(const TIO* Kb, const TIO* Vb, const float2* rope,
                                            const Plan& P, int r0, int nb, int i0, int TQ, int T,
                                            float* sK, float* sV, int* status) {
  const int per = TQ * 4;
  for (int it = threadIdx.x; it < nb * per; it += kThreads) {
    const int a = it / per, rem = it - a * per;
    const int rr = rem >> 2, pc = rem & 3;
    const int iq = i0 + rr;
    const int p0 = iq - P.c[r0 + a];
    if (iq >= T || p0 < 0 || p0 >= T) continue;  // rung absent for this query
    if (!dbg_in(a * TQ + rr, kSlab, status)) continue;
    float* dk = sK + (a * TQ + rr) * kRowPad;
    float* dv = sV + (a * TQ + rr) * kRowPad;
    float klo[8], khi[8], vlo[8], vhi[8];
    load_pair_chunk(Kb + (int64_t)p0 * kD, pc, rope, p0, klo, khi);
    load_pair_chunk<TIO>(Vb + (int64_t)p0 * kD, pc, nullptr, p0, vlo, vhi);
    if (INTERP) {
      const float w = P.w[r0 + a];
      if (w != 0.0f && dbg_in(p0 + 1, T, status)) {  // p0 + 1 <= iq: inside the sequence
        float k2l[8], k2h[8], v2l[8], v2h[8];
        load_pair_chunk(Kb + (int64_t)(p0 + 1) * kD, pc, rope, p0 + 1, k2l, k2h);
        load_pair_chunk<TIO>(Vb + (int64_t)(p0 + 1) * kD, pc, nullptr, p0 + 1, v2l, v2h);
        const float u = 1.0f - w;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          klo[e] = fmaf(w, k2l[e], u * klo[e]);
          khi[e] = fmaf(w, k2h[e], u * khi[e]);
          vlo[e] = fmaf(w, v2l[e], u * vlo[e]);
          vhi[e] = fmaf(w, v2h[e], u * vhi[e]);
        }
      }
    }
    st_smem8(dk + 8 * pc, klo);
    st_smem8(dk + 32 + 8 * pc, khi);
    st_smem8(dv + 8 * pc, vlo);
    st_smem8(dv + 32 + 8 * pc, vhi);
  }
}

}  // namespace sfa
