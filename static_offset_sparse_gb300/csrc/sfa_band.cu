// Tensor-core kernels for integer distance sets made of long arithmetic runs
// (bf16 I/O, G = 1, 2, 4 or 8 query heads per KV head).
//
// "Christoffel-Balanced Sparse Attention" builds its offsets from a carry
// word with m ones per period k; when m divides k they are 0 and
// k/m - 1 + t k/m, one arithmetic run, and a dense causal window is one run
// of step 1.  With delta the runs' common step and i = r + delta u
// (r = i mod delta), run m (distances a_m + delta t, t < len_m) sends query
// class r to key class rho = (r - a_m) mod delta at compressed keys
// v in [u + e - len_m + 1, u + e], e = floor((r - a_m) / delta): a band.  The
// keys of query i are still exactly i - s for s in the set (the integer path
// of "Depth-Staggered Fibonacci Spacing for Sparse Attention"); only the
// order of the work changes.
//
// A CTA owns 64 query rows, G heads x 64 / G consecutive compressed positions
// of one class (row h (64 / G) + u), and walks, run by run, the 64-key tiles
// of its band.  Rows come in as TMA boxes of a [plane][T / delta][delta][64]
// view (the class is a coordinate of stride one row, the compressed index
// one of stride delta rows; rows outside the sequence are zero-filled).
// Products are mma.sync m16n8k16 (bf16 in, fp32 accumulate) on dense
// 16 x 64 per-warp tiles, masked only at the band's edges:
//  * band_fwd:    S = q~.K'^T (q~ = q'/8 in bf16, as the backward has it),
//                 online softmax in base 2, O += P.V; O, LSE.
//  * band_bwd_q:  S and dP = dO.V^T recomputed, P = exp(S - LSE),
//                 dS = P (dP - delta_i), dQ += dS.K'; writes dQ = R(-phi) dQ'
//                 / 8, q~ = q'/8 and per row (LSE log2(e), sum_j P dP).
//  * band_bwd_kv: per 64-key tile, the query tiles of each run that reach
//                 it, keys on the mma M side: S^T = K'.q~^T, dP^T = V.dO^T,
//                 dV += P^T.dO, dK' += dS^T.q~; dK = R(-phi) dK'.  Each key
//                 row is written once (no atomics).
#include <math.h>

#include "sfa_tc.cuh"
#include "sfa_umma.cuh"

namespace sfa {

constexpr int kBR = 64;                 // rows of every tile: queries (G heads x 64/G) or keys
constexpr int kBThreads = 128;          // 4 warps x 16 rows
constexpr int kBTileB = kBR * 128;      // 8 KB, a 1024-byte multiple (128B swizzle)
constexpr int kBStages = 2;
constexpr int kBStageB = 2 * kBTileB;   // K' + V, or q~ + dO
constexpr size_t kBandFwdSmem = (size_t)kBTileB + (size_t)kBStages * kBStageB + 1024;
constexpr size_t kBandBwdQSmem = (size_t)3 * kBTileB + (size_t)kBStages * kBStageB + 1024;
constexpr size_t kBandBwdKvSmem = (size_t)2 * kBTileB + (size_t)kBStages * kBStageB + 1024;

// Class and shift of run m for query class r: r - a_m = rho + delta e.
__device__ __forceinline__ void run_shift(const BandPlan& P, int m, int r, int& rho, int& e) {
  const int x = r - P.a[m];
  e = x >= 0 ? x / P.delta : -((P.delta - 1 - x) / P.delta);
  rho = x - e * P.delta;
}

// Key tiles of a query tile (class r, compressed positions u0 .. ul): run by
// run, the band [u0 + e - len + 1, ul + e] clipped to the sequence's Uc
// compressed keys (a negative distance, e > 0, reads later keys), from its
// low end in steps of 64.
struct QWalk {
  int m, vs, vhi, rho, e;
};
__device__ __forceinline__ bool qwalk_seek(const BandPlan& P, int r, int u0, int ul, int Uc,
                                           QWalk& w) {
  for (; w.m < P.nruns; ++w.m) {
    run_shift(P, w.m, r, w.rho, w.e);
    const int lo = max(0, u0 + w.e - P.len[w.m] + 1), hi = min(ul + w.e, Uc - 1);
    if (lo <= hi) {
      w.vs = lo;
      w.vhi = hi;
      return true;
    }
  }
  return false;
}
__device__ __forceinline__ bool qwalk_next(const BandPlan& P, int r, int u0, int ul, int Uc,
                                           QWalk& w) {
  w.vs += kBR;
  if (w.vs <= w.vhi) return true;
  ++w.m;
  return qwalk_seek(P, r, u0, ul, Uc, w);
}

// Query tiles that reach a key tile (class rho, compressed keys v0 .. vl):
// run by run, query class r = (rho + a) mod delta at positions
// [v0 - e, vl - e + len - 1] (clipped to the sequence at both ends), in steps
// of bu.
struct KWalk {
  int m, us, uhi, r, e;
};
__device__ __forceinline__ bool kwalk_seek(const BandPlan& P, int rho, int v0, int vl, int Uc,
                                           KWalk& w) {
  for (; w.m < P.nruns; ++w.m) {
    w.r = ((rho + P.a[w.m]) % P.delta + P.delta) % P.delta;  // a < 0 for a signed run
    int rho2;
    run_shift(P, w.m, w.r, rho2, w.e);
    const int lo = max(0, v0 - w.e), hi = min(Uc - 1, vl - w.e + P.len[w.m] - 1);
    if (lo <= hi) {
      w.us = lo;
      w.uhi = hi;
      return true;
    }
  }
  return false;
}
__device__ __forceinline__ bool kwalk_next(const BandPlan& P, int rho, int v0, int vl, int Uc, int bu,
                                           KWalk& w) {
  w.us += bu;
  if (w.us <= w.uhi) return true;
  ++w.m;
  return kwalk_seek(P, rho, v0, vl, Uc, w);
}

// The RoPE (cos, sin) pairs of rows gid (x = 0) and gid + 8 at positions
// pos[x] that band_frags needs (pairs 16 kk + 2 tig + {0, 1, 8, 9}), loaded
// while the tile is still in flight.
__device__ __forceinline__ void band_rope_pairs(const float2* rope, const int* pos, float4 (*rp)[4]) {
  const int tig = threadIdx.x & 3;
#pragma unroll
  for (int x = 0; x < 2; ++x)
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const float2* tab = rope + (int64_t)pos[x] * 32 + 16 * kk + 2 * tig;
      rp[x][2 * kk] = __ldg(reinterpret_cast<const float4*>(tab));
      rp[x][2 * kk + 1] = __ldg(reinterpret_cast<const float4*>(tab + 8));
    }
}

// A fragments of rows row0 .. row0 + 15 of a 64-row tile for the 4 k-steps.
// With transform they are unpacked, rotated by the RoPE pairs rp of
// band_rope_pairs (none if rp is nullptr), scaled and repacked.
__device__ __forceinline__ void band_frags(uint32_t tile, int row0, const float4 (*rp)[4],
                                           float scale, bool transform, uint32_t (*qa)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    ldsm_x4(tile + swz(row0 + (lane & 15), 2 * kk + (lane >> 4)), qa[kk][0], qa[kk][1], qa[kk][2],
            qa[kk][3]);
  if (!transform) return;
  float x[2][4][4];  // [row gid / gid + 8][kk][dims 2tig, 2tig+1, 2tig+8, 2tig+9]
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const float2 a0 = unpack_bf16(qa[kk][0]), a1 = unpack_bf16(qa[kk][1]);
    const float2 a2 = unpack_bf16(qa[kk][2]), a3 = unpack_bf16(qa[kk][3]);
    x[0][kk][0] = a0.x; x[0][kk][1] = a0.y; x[0][kk][2] = a2.x; x[0][kk][3] = a2.y;
    x[1][kk][0] = a1.x; x[1][kk][1] = a1.y; x[1][kk][2] = a3.x; x[1][kk][3] = a3.y;
  }
  if (rp) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const float4 a = rp[rr][2 * kk], b = rp[rr][2 * kk + 1];
        const float cs[4] = {a.x, a.z, b.x, b.z}, sn[4] = {a.y, a.w, b.y, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = x[rr][kk][e], hi = x[rr][kk + 2][e];
          x[rr][kk][e] = lo * cs[e] - hi * sn[e];
          x[rr][kk + 2][e] = lo * sn[e] + hi * cs[e];
        }
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

// Byte address of the bf16 pair (dims 8 nd + 2 tig, + 1) of tile row `row`.
__device__ __forceinline__ uint32_t band_out_addr(uint32_t tile, int row, int nd) {
  return tile + swz(row, nd) + 4 * (threadIdx.x & 3);
}

// Rows gid (x = 0) and gid + 8 (x = 1) of a warp's accumulator v[8][4]
// (dims 8 nd + 2 tig, + 1), scaled, optionally rotated back by RoPE
// (R(-phi) at positions pos[x]), into a 64-row output tile.
__device__ __forceinline__ void band_store_rows(uint32_t tile, int row0, const float (*v)[4],
                                                const float* scale, const float2* rope,
                                                const int* pos) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    float w[8][2];
#pragma unroll
    for (int nd = 0; nd < 8; ++nd) {
      w[nd][0] = v[nd][2 * x] * scale[x];
      w[nd][1] = v[nd][2 * x + 1] * scale[x];
    }
    if (rope) {
#pragma unroll
      for (int nd = 0; nd < 4; ++nd) {
        const float4 cs =
            __ldg(reinterpret_cast<const float4*>(rope + (int64_t)pos[x] * 32 + 8 * nd + 2 * tig));
        const float c2[2] = {cs.x, cs.z}, s2[2] = {cs.y, cs.w};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float lo = w[nd][e], hi = w[nd + 4][e];
          w[nd][e] = lo * c2[e] + hi * s2[e];
          w[nd + 4][e] = hi * c2[e] - lo * s2[e];
        }
      }
    }
#pragma unroll
    for (int nd = 0; nd < 8; ++nd)
      st_shared_u32(band_out_addr(tile, row0 + gid + 8 * x, nd), pack_bf16(w[nd][0], w[nd][1]));
  }
}

// acc[nt] += A . rows(row0 + 8 nt .. + 7)^T for four n-tiles, k-step outer:
// consecutive products go to different accumulators (qk_tile's four
// products chain on one).  B fragments of two k-steps are live at a time.
__device__ __forceinline__ void qk_tiles4(const uint32_t (*qa)[4], uint32_t region, int row0,
                                          float (*acc)[4]) {
  const int lane = threadIdx.x & 31, mi = lane >> 3;
#pragma unroll
  for (int hk = 0; hk < 2; ++hk) {  // dims 32 hk .. 32 hk + 31: k-steps 2 hk, 2 hk + 1
    uint32_t b[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
      ldsm_x4(region + swz(row0 + 8 * nt + (lane & 7), 4 * hk + mi), b[nt][0], b[nt][1], b[nt][2],
              b[nt][3]);
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) mma_bf16(acc[nt], qa[2 * hk + k2], b[nt][2 * k2], b[nt][2 * k2 + 1]);
  }
}

// x as bf16 hi + lo pairs (hi = bf16(x), lo = bf16(x - hi)): about 16
// mantissa bits for the key side's sums over many queries.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x0, x1);
  const float2 h = unpack_bf16(hi);
  lo = pack_bf16(x0 - h.x, x1 - h.y);
}

// acc[16 x 64] += (A_hi + A_lo)[16 x 16] . rows[16 x 64] (as pv_tile, one set
// of B loads for both parts).
__device__ __forceinline__ void pv_tile2(const uint32_t* ah, const uint32_t* al, uint32_t region,
                                         int row_lo, int row_hi, float (*acc)[4]) {
  const int mi = (threadIdx.x & 31) >> 3;
  const int row = (mi & 1) ? row_hi : row_lo;
#pragma unroll
  for (int nd = 0; nd < 8; nd += 2) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(region + swz(row, nd + (mi >> 1)), b0, b1, b2, b3);
    mma_bf16(acc[nd], ah, b0, b1);
    mma_bf16(acc[nd + 1], ah, b2, b3);
    mma_bf16(acc[nd], al, b0, b1);
    mma_bf16(acc[nd + 1], al, b2, b3);
  }
}

// acc0 += A0 . rows and acc1 += A1 . rows for one set of B loads.
__device__ __forceinline__ void pv_tile2(const uint32_t* a0, const uint32_t* a1, uint32_t region,
                                         int row_lo, int row_hi, float (*acc0)[4],
                                         float (*acc1)[4]) {
  const int mi = (threadIdx.x & 31) >> 3;
  const int row = (mi & 1) ? row_hi : row_lo;
#pragma unroll
  for (int nd = 0; nd < 8; nd += 2) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(region + swz(row, nd + (mi >> 1)), b0, b1, b2, b3);
    mma_bf16(acc0[nd], a0, b0, b1);
    mma_bf16(acc0[nd + 1], a0, b2, b3);
    mma_bf16(acc1[nd], a1, b0, b1);
    mma_bf16(acc1[nd + 1], a1, b2, b3);
  }
}

// Barriers: kBStages stage barriers, then one for the CTA's own tiles; the
// dependent-launch handshake (no global access before it).
__device__ __forceinline__ void band_init_bars(uint64_t* bars) {
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s <= kBStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();  // the previous kernel's outputs are complete from here on
}

// Bounded wait on a barrier, uniform across the CTA (false: timed out, the
// status word holds SFA_ERR_TIMEOUT).
__device__ __forceinline__ bool band_wait(uint64_t* bar, uint32_t parity, const AttnArgs& a) {
  const bool ok = mbar_wait_bounded(smem_u32(bar), parity, a.wait_cycles);
  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) record_status(a.status, SFA_ERR_TIMEOUT);
    return false;
  }
  return true;
}

// The staged loop: tile t waits on stage t % kBStages; once every thread has
// passed the barrier of tile t, the stage of tile t - 1 is refilled with tile
// t - 1 + kBStages by issue(stage) (thread 0, in tile order).  compute(t,
// stage address) runs on every thread.  False (uniformly) on a timeout,
// after thread 0 has waited out the loads still in flight.
template <typename IssueFn, typename ComputeFn>
__device__ __forceinline__ bool band_loop(int NT, uint32_t stages, uint64_t* bars, const AttnArgs& a,
                                          IssueFn issue, ComputeFn compute) {
  for (int t = 0; t < NT; ++t) {
    const int s = t % kBStages;
    const bool ok = mbar_wait_bounded(smem_u32(&bars[s]), (t / kBStages) & 1, a.wait_cycles);
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) {
        record_status(a.status, SFA_ERR_TIMEOUT);
        for (int t2 = t; t2 < NT && t2 < t + kBStages - 1; ++t2)
          mbar_wait_bounded(smem_u32(&bars[t2 % kBStages]), (t2 / kBStages) & 1, a.wait_cycles);
      }
      return false;
    }
    if (threadIdx.x == 0 && t > 0 && t - 1 + kBStages < NT) issue((t - 1) % kBStages);
    compute(t, stages + s * kBStageB);
  }
  __syncthreads();  // every stage is consumed: shared memory may be reused
  return true;
}

// Thread 0 waits out the first stages' loads after the CTA's own tiles timed
// out (nothing may land in shared memory after the CTA has left).
__device__ __forceinline__ void band_drain(uint64_t* bars, int NT, const AttnArgs& a) {
  if (threadIdx.x == 0)
    for (int s = 0; s < kBStages && s < NT; ++s) mbar_wait_bounded(smem_u32(&bars[s]), 0, a.wait_cycles);
}

// Online softmax over N keys of a tile for rows gid (x = 0) and gid + 8 of a
// lane: s[x][N] holds base-2 logits (invalid = -inf) and comes back as
// p = 2^(s - m).  The running maximum m is refreshed only when some logit
// of the warp exceeds it by more than 8: between refreshes p stays below
// 2^8, and O = sum p v / sum p and LSE = m + log2 l hold for any m.  m stays
// uniform over a row's quad (it changes only through the quad reduction).
template <int N>
__device__ __forceinline__ void band_softmax(float (*s)[N], float* m, float* l, float (*o)[4]) {
  constexpr float kMargin = 8.0f;
  float mx[2];
  bool need = false;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    mx[x] = s[x][0];
#pragma unroll
    for (int e = 1; e < N; ++e) mx[x] = fmaxf(mx[x], s[x][e]);
    need |= mx[x] > m[x] + kMargin;  // m = -inf: any valid logit
  }
  if (__any_sync(0xffffffffu, need)) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      mx[x] = fmaxf(mx[x], __shfl_xor_sync(0xffffffffu, mx[x], 1));
      mx[x] = fmaxf(mx[x], __shfl_xor_sync(0xffffffffu, mx[x], 2));
      if (mx[x] > m[x]) {
        const float corr = ex2(m[x] - mx[x]);  // 0 while the row had no key
        m[x] = mx[x];
        l[x] *= corr;
#pragma unroll
        for (int nd = 0; nd < 8; ++nd) {
          o[nd][2 * x] *= corr;
          o[nd][2 * x + 1] *= corr;
        }
      }
    }
  }
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const float mm = m[x] == -INFINITY ? 0.0f : m[x];
#pragma unroll
    for (int e = 0; e < N; ++e) {
      const float pe = ex2(s[x][e] - mm);  // ex2(-inf) = 0
      s[x][e] = pe;
      l[x] += pe;
    }
  }
}

// Whether every row of the warp reads all 32 key columns c0 .. c0 + 31 of the
// current tile (lo, hi: this lane's two rows' column ranges; a row past the
// sequence has hi = -1 and never qualifies).  Warp-uniform.
__device__ __forceinline__ bool band_half_full(const int* lo, const int* hi, int c0) {
  return __all_sync(0xffffffffu, lo[0] <= c0 && lo[1] <= c0 && hi[0] >= c0 + 31 && hi[1] >= c0 + 31);
}

// Query-tile geometry shared by the forward and the query-side backward.
template <int G>
struct QTile {
  static constexpr int BU = kBR / G;
  int delta, Uc, r, u0, ul, qplane, bg;
  int hh[2], uu[2], pos[2];  // rows gid, gid + 8 of the lane's warp: head, position, i
  // reverse: planes in reverse launch order (the query-side backward starts on
  // the planes the forward ended on, whose O and LSE are the likeliest to be
  // in L2, and ends on those the key side starts on)
  __device__ __forceinline__ QTile(const AttnArgs& a, const BandPlan& P, bool reverse) {
    const int warp = threadIdx.x >> 5, gid = (threadIdx.x & 31) >> 2;
    delta = P.delta;
    Uc = a.T / delta;
    const int nqt = (Uc + BU - 1) / BU;
    r = blockIdx.x / nqt;
    u0 = (blockIdx.x - r * nqt) * BU;
    ul = min(u0 + BU - 1, Uc - 1);
    bg = reverse ? gridDim.y - 1 - blockIdx.y : blockIdx.y;
    const int b = bg / a.Hkv, g = bg - b * a.Hkv;
    qplane = b * a.Hq + g * G;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int row = 16 * warp + gid + 8 * x;
      hh[x] = row / BU;
      uu[x] = u0 + row % BU;
      pos[x] = r + delta * min(uu[x], Uc - 1);
    }
  }
  __device__ __forceinline__ int count(const BandPlan& P) const {
    int n = 0;
    QWalk w{0, 0, 0, 0, 0};
    if (qwalk_seek(P, r, u0, ul, Uc, w)) do ++n; while (qwalk_next(P, r, u0, ul, Uc, w));
    return n;
  }
  // Positions of this warp's 16 rows: one head's 16 consecutive positions
  // (64 / G >= 16) or the same 8 positions of two heads (G = 8).
  __device__ __forceinline__ void warp_span(int& umin, int& umax) const {
    const int warp = threadIdx.x >> 5;
    umin = u0 + (BU >= 16 ? (16 * warp) % BU : 0);
    umax = min(umin + (BU >= 16 ? 15 : BU - 1), Uc - 1);
  }
  // The n-tiles (8 key columns each) of the current tile that hold a key of
  // some row of the warp (bit nt); warp-uniform, 0 when none does.
  __device__ __forceinline__ unsigned ntmask(const BandPlan& P, const QWalk& w, int umin,
                                             int umax) const {
    const int cl = max(0, umin + w.e - P.len[w.m] + 1 - w.vs);
    const int ch = min(kBR - 1, min(umax + w.e, Uc - 1) - w.vs);
    if (umin > umax || cl > ch) return 0u;
    return ((2u << (ch >> 3)) - 1u) & ~((1u << (cl >> 3)) - 1u);
  }
  // Tile columns [lo, hi] of row x that are keys of the current run.
  __device__ __forceinline__ void cols(const BandPlan& P, const QWalk& w, int* lo, int* hi) const {
    const int len = P.len[w.m];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      lo[x] = uu[x] + w.e - len + 1 - w.vs;
      // rows past the sequence take no key; keys past it do not exist
      hi[x] = uu[x] < Uc ? min(uu[x] + w.e, Uc - 1) - w.vs : -1;
    }
  }
};

template <int G>
__global__ void __launch_bounds__(kBThreads, 5)
    band_fwd_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mq,
                    const __grid_constant__ CUtensorMap mo, const __grid_constant__ BandPlan P) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bars[kBStages + 1];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tig = lane & 3;
  const QTile<G> q(a, P, false);
  const uint32_t qtile = sbase, stages = sbase + kBTileB;
  const int NT = q.count(P);
  band_init_bars(bars);
  QWalk iw{0, 0, 0, 0, 0};
  auto issue = [&](int s) {
    const uint32_t st = stages + s * kBStageB, bar = smem_u32(&bars[s]);
    mbar_expect_tx(bar, kBStageB);
    tma_load_4d(st, &mk, 0, iw.rho, iw.vs, q.bg, bar);
    tma_load_4d(st + kBTileB, &mv, 0, iw.rho, iw.vs, q.bg, bar);
    qwalk_next(P, q.r, q.u0, q.ul, q.Uc, iw);
  };
  if (threadIdx.x == 0) {
    const uint32_t qb = smem_u32(&bars[kBStages]);
    mbar_expect_tx(qb, kBTileB);
    tma_load_4d(qtile, &mq, 0, q.r, q.u0, q.qplane, qb);
    qwalk_seek(P, q.r, q.u0, q.ul, q.Uc, iw);
    for (int s = 0; s < kBStages && s < NT; ++s) issue(s);
  }
  const float2* rope = static_cast<const float2*>(a.rope);
  float4 rp[2][4];
  if (rope) band_rope_pairs(rope, q.pos, rp);  // while the Q tile is in flight
  if (!band_wait(&bars[kBStages], 0, a)) {
    band_drain(bars, NT, a);
    return;
  }
  // q~ = q'/8 rounded exactly as the backward rounds it, log2(e) applied to
  // the fp32 logits: the backward's P = exp(S - LSE) then recomputes this
  // kernel's logits bit for bit and stays normalised
  uint32_t qa[4][4];
  band_frags(qtile, 16 * warp, rope ? rp : nullptr, 0.125f, true, qa);
  float o[8][4];
#pragma unroll
  for (int nd = 0; nd < 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.0f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
  QWalk cw{0, 0, 0, 0, 0};
  qwalk_seek(P, q.r, q.u0, q.ul, q.Uc, cw);

  const bool ok = band_loop(NT, stages, bars, a, issue, [&](int, uint32_t kst) {
    // every warp computes the whole tile (skipping the n-tiles outside its
    // rows' bands measured slower: it breaks up the load and product batches
    // the scheduler overlaps), in two halves of 32 keys with one softmax step
    // each, which keeps four CTAs per SM within the register file
    int lo[2], hi[2];
    q.cols(P, cw, lo, hi);
    const uint32_t vst = kst + kBTileB;
    if (P.len[cw.m] == 1) {
      // a one-distance run (distance 0 in the Christoffel sets): each row reads
      // one key, and a warp's 16 rows read at most 16 consecutive columns, so
      // the warp computes the three n-tiles nb .. nb + 2 around them (a
      // CTA-uniform path: the n-tile base only moves shared-memory addresses)
      int umin, umax;
      q.warp_span(umin, umax);
      const int nb = min(max(0, umin + cw.e - cw.vs) >> 3, 5);
      float acc[3][4];
#pragma unroll
      for (int nt = 0; nt < 3; ++nt) {
        acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
        qk_tile(qa, kst, 8 * (nb + nt) + (lane & 7), acc[nt]);
      }
      float s[2][6];
#pragma unroll
      for (int nt = 0; nt < 3; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int x = e >> 1, col = 8 * (nb + nt) + 2 * tig + (e & 1);
          s[x][2 * nt + (e & 1)] = (col >= lo[x] && col <= hi[x]) ? acc[nt][e] * kLog2e : -INFINITY;
        }
      band_softmax<6>(s, m, l, o);
      const uint32_t pa0[4] = {pack_bf16(s[0][0], s[0][1]), pack_bf16(s[1][0], s[1][1]),
                               pack_bf16(s[0][2], s[0][3]), pack_bf16(s[1][2], s[1][3])};
      const uint32_t pa1[4] = {pack_bf16(s[0][4], s[0][5]), pack_bf16(s[1][4], s[1][5]), 0u, 0u};
      const int rl = 8 * nb + (lane & 7);
      pv_tile(pa0, vst, rl, rl + 8, o);
      pv_tile(pa1, vst, rl + 16, rl + 16, o);  // keys 8 nb + 24 .. are not read (zero P)
      qwalk_next(P, q.r, q.u0, q.ul, q.Uc, cw);
      return;
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      float acc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
      qk_tiles4(qa, kst, 32 * hf, acc);
      float s[2][8];
      // inside the band: every row of the warp reads all 32 keys of the half,
      // so the per-element mask (which would pass them all) is skipped
      if (band_half_full(lo, hi, 32 * hf)) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[e >> 1][2 * nt + (e & 1)] = acc[nt][e] * kLog2e;
      } else {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int x = e >> 1, col = 32 * hf + 8 * nt + 2 * tig + (e & 1);
            s[x][2 * nt + (e & 1)] = (col >= lo[x] && col <= hi[x]) ? acc[nt][e] * kLog2e : -INFINITY;
          }
      }
      band_softmax<8>(s, m, l, o);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint32_t pa[4] = {pack_bf16(s[0][4 * kk], s[0][4 * kk + 1]),
                                pack_bf16(s[1][4 * kk], s[1][4 * kk + 1]),
                                pack_bf16(s[0][4 * kk + 2], s[0][4 * kk + 3]),
                                pack_bf16(s[1][4 * kk + 2], s[1][4 * kk + 3])};
        const int rl = 32 * hf + 16 * kk + (lane & 7);
        pv_tile(pa, vst, rl, rl + 8, o);
      }
    }
    qwalk_next(P, q.r, q.u0, q.ul, q.Uc, cw);
  });
  if (!ok) return;

  float inv[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    l[x] += __shfl_xor_sync(0xffffffffu, l[x], 1);
    l[x] += __shfl_xor_sync(0xffffffffu, l[x], 2);
    inv[x] = 1.0f / l[x];
    if (tig == 0 && q.uu[x] < q.Uc)
      a.out_lse[(int64_t)(q.qplane + q.hh[x]) * a.T + q.pos[x]] = (m[x] + log2f(l[x])) * kLn2;
  }
  band_store_rows(qtile, 16 * warp, o, inv, nullptr, q.pos);
  fence_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    tma_store_4d(&mo, 0, q.r, q.u0, q.qplane, qtile);
    bulk_commit();
    bulk_wait_read();
  }
}

template <int G>
__global__ void __launch_bounds__(kBThreads, 3)
    band_bwd_q_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mq,
                      const __grid_constant__ CUtensorMap mdo, const __grid_constant__ CUtensorMap mo,
                      const __grid_constant__ CUtensorMap mqt,
                      const __grid_constant__ CUtensorMap mdq, float2* __restrict__ stat,
                      const __grid_constant__ BandPlan P) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bars[kBStages + 1];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gid = lane >> 2, tig = lane & 3;
  const QTile<G> q(a, P, true);
  const uint32_t qtile = sbase, dotile = sbase + kBTileB, otile = sbase + 2 * kBTileB;
  const uint32_t stages = sbase + 3 * kBTileB;
  const float2* rope = static_cast<const float2*>(a.rope);
  const int NT = q.count(P);
  band_init_bars(bars);
  QWalk iw{0, 0, 0, 0, 0};
  auto issue = [&](int s) {
    const uint32_t st = stages + s * kBStageB, bar = smem_u32(&bars[s]);
    mbar_expect_tx(bar, kBStageB);
    tma_load_4d(st, &mk, 0, iw.rho, iw.vs, q.bg, bar);
    tma_load_4d(st + kBTileB, &mv, 0, iw.rho, iw.vs, q.bg, bar);
    qwalk_next(P, q.r, q.u0, q.ul, q.Uc, iw);
  };
  if (threadIdx.x == 0) {
    const uint32_t qb = smem_u32(&bars[kBStages]);
    mbar_expect_tx(qb, 3 * kBTileB);
    tma_load_4d(qtile, &mq, 0, q.r, q.u0, q.qplane, qb);
    tma_load_4d(dotile, &mdo, 0, q.r, q.u0, q.qplane, qb);
    tma_load_4d(otile, &mo, 0, q.r, q.u0, q.qplane, qb);
    qwalk_seek(P, q.r, q.u0, q.ul, q.Uc, iw);
    for (int s = 0; s < kBStages && s < NT; ++s) issue(s);
  }
  float lse2[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) lse2[x] = a.lse[(int64_t)(q.qplane + q.hh[x]) * a.T + q.pos[x]] * kLog2e;
  float4 rp[2][4];
  if (rope) band_rope_pairs(rope, q.pos, rp);  // while the query tiles are in flight
  if (!band_wait(&bars[kBStages], 0, a)) {
    band_drain(bars, NT, a);
    return;
  }
  uint32_t qa[4][4], da[4][4];
  band_frags(qtile, 16 * warp, rope ? rp : nullptr, 0.125f, true, qa);
  band_frags(dotile, 16 * warp, nullptr, 1.0f, false, da);
  float dlt[2];
  {  // delta_i = dO . O per row from this lane's 16 dims of each, then the quad
    uint32_t oa[4][4];
    band_frags(otile, 16 * warp, nullptr, 1.0f, false, oa);
    float acc[2] = {0.0f, 0.0f};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float2 u = unpack_bf16(da[kk][x]), v = unpack_bf16(oa[kk][x]);
        acc[x & 1] = fmaf(u.x, v.x, fmaf(u.y, v.y, acc[x & 1]));  // x even: row gid, odd: gid + 8
      }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      acc[x] += __shfl_xor_sync(0xffffffffu, acc[x], 1);
      acc[x] += __shfl_xor_sync(0xffffffffu, acc[x], 2);
      dlt[x] = acc[x];
    }
  }
  __syncthreads();  // the O tile is read: it now carries q~ = q'/8 out for the key side
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    st_shared_u32(band_out_addr(otile, 16 * warp + gid, 2 * kk), qa[kk][0]);
    st_shared_u32(band_out_addr(otile, 16 * warp + gid + 8, 2 * kk), qa[kk][1]);
    st_shared_u32(band_out_addr(otile, 16 * warp + gid, 2 * kk + 1), qa[kk][2]);
    st_shared_u32(band_out_addr(otile, 16 * warp + gid + 8, 2 * kk + 1), qa[kk][3]);
  }
  fence_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    tma_store_4d(&mqt, 0, q.r, q.u0, q.qplane, otile);
    bulk_commit();
  }
  float dq[8][4];
#pragma unroll
  for (int nd = 0; nd < 8; ++nd) dq[nd][0] = dq[nd][1] = dq[nd][2] = dq[nd][3] = 0.0f;
  // delta_i is dO . O from the stored (bf16) O; the exact value is
  // sum_j P_ij dP_ij (fp32 here), and with |dP| in the tens the difference
  // shifts dS visibly.  The loop uses the O value and also sums
  // psum = sum_j P_ij dP_ij and kbar = sum_j P_ij K'_j; at the end
  // dQ' += (delta - psum) kbar makes dQ' = sum_j P_ij (dP_ij - psum) K'_j, and
  // the key side reads psum.
  float psum[2] = {0.0f, 0.0f};
  float kbar[8][4];
#pragma unroll
  for (int nd = 0; nd < 8; ++nd) kbar[nd][0] = kbar[nd][1] = kbar[nd][2] = kbar[nd][3] = 0.0f;
  QWalk cw{0, 0, 0, 0, 0};
  qwalk_seek(P, q.r, q.u0, q.ul, q.Uc, cw);
  int umin, umax;
  q.warp_span(umin, umax);

  const bool ok = band_loop(NT, stages, bars, a, issue, [&](int, uint32_t kst) {
    const uint32_t vst = kst + kBTileB;
    int lo[2], hi[2];
    q.cols(P, cw, lo, hi);
    const unsigned msk = q.ntmask(P, cw, umin, umax);  // n-tiles the warp's rows read
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {  // keys 32 hf .. 32 hf + 31 of the tile
      const unsigned mh = (msk >> (4 * hf)) & 15u;
      if (!mh) continue;
      float sc[4][4], dp[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.0f;
        dp[nt][0] = dp[nt][1] = dp[nt][2] = dp[nt][3] = 0.0f;
        if (!((mh >> nt) & 1u)) continue;
        const int row = 32 * hf + 8 * nt + (lane & 7);
        qk_tile(qa, kst, row, sc[nt]);
        qk_tile(da, vst, row, dp[nt]);
      }
      float ds[4][4], pp[4][4];
      if (mh == 15u && band_half_full(lo, hi, 32 * hf)) {  // no key of the half is masked
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) pp[nt][e] = ex2(fmaf(sc[nt][e], kLog2e, -lse2[e >> 1]));
      } else {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int x = e >> 1, col = 32 * hf + 8 * nt + 2 * tig + (e & 1);
            pp[nt][e] = ((mh >> nt) & 1u) && col >= lo[x] && col <= hi[x]
                            ? ex2(fmaf(sc[nt][e], kLog2e, -lse2[x]))
                            : 0.0f;
          }
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int x = e >> 1;
          ds[nt][e] = pp[nt][e] * (dp[nt][e] - dlt[x]);
          psum[x] = fmaf(pp[nt][e], dp[nt][e], psum[x]);
        }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        if (!((mh >> (2 * ks)) & 3u)) continue;
        const uint32_t sa[4] = {pack_bf16(ds[2 * ks][0], ds[2 * ks][1]),
                                pack_bf16(ds[2 * ks][2], ds[2 * ks][3]),
                                pack_bf16(ds[2 * ks + 1][0], ds[2 * ks + 1][1]),
                                pack_bf16(ds[2 * ks + 1][2], ds[2 * ks + 1][3])};
        const uint32_t pa[4] = {pack_bf16(pp[2 * ks][0], pp[2 * ks][1]),
                                pack_bf16(pp[2 * ks][2], pp[2 * ks][3]),
                                pack_bf16(pp[2 * ks + 1][0], pp[2 * ks + 1][1]),
                                pack_bf16(pp[2 * ks + 1][2], pp[2 * ks + 1][3])};
        const int rl = 32 * hf + 16 * ks + (lane & 7);
        pv_tile2(sa, pa, kst, rl, rl + 8, dq, kbar);
      }
    }
    qwalk_next(P, q.r, q.u0, q.ul, q.Uc, cw);
  });
  if (!ok) {
    if (threadIdx.x == 0) bulk_wait_read();
    return;
  }
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    psum[x] += __shfl_xor_sync(0xffffffffu, psum[x], 1);
    psum[x] += __shfl_xor_sync(0xffffffffu, psum[x], 2);
    if (tig == 0 && q.uu[x] < q.Uc)
      stat[(int64_t)(q.qplane + q.hh[x]) * a.T + q.pos[x]] = make_float2(lse2[x], psum[x]);
    const float corr = dlt[x] - psum[x];
#pragma unroll
    for (int nd = 0; nd < 8; ++nd) {
      dq[nd][2 * x] = fmaf(corr, kbar[nd][2 * x], dq[nd][2 * x]);
      dq[nd][2 * x + 1] = fmaf(corr, kbar[nd][2 * x + 1], dq[nd][2 * x + 1]);
    }
  }
  const float eighth[2] = {0.125f, 0.125f};
  band_store_rows(qtile, 16 * warp, dq, eighth, rope, q.pos);  // dQ = R(-phi) dQ' / 8
  fence_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    tma_store_4d(&mdq, 0, q.r, q.u0, q.qplane, qtile);
    bulk_commit();
    bulk_wait_read();  // the q~ and dQ tiles have been read
  }
}

template <int G>
__global__ void __launch_bounds__(kBThreads, 3)
    band_bwd_kv_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mqt,
                       const __grid_constant__ CUtensorMap mdo, const __grid_constant__ CUtensorMap mdk,
                       const __grid_constant__ CUtensorMap mdv, const float2* __restrict__ stat,
                       const __grid_constant__ BandPlan P) {
  constexpr int BU = kBR / G;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bars[kBStages + 1];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gid = lane >> 2, tig = lane & 3;
  const int T = a.T, delta = P.delta, Uc = T / delta;
  const int nkt = (Uc + kBR - 1) / kBR;
  const int rho = blockIdx.x / nkt, v0 = (blockIdx.x - rho * nkt) * kBR;
  const int vl = min(v0 + kBR - 1, Uc - 1);
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int qplane = b * a.Hq + g * G;
  const int kv[2] = {v0 + 16 * warp + gid, v0 + 16 * warp + gid + 8};  // this lane's key rows
  const uint32_t ktile = sbase, vtile = sbase + kBTileB, stages = sbase + 2 * kBTileB;
  int NT = 0;
  {
    KWalk w{0, 0, 0, 0, 0};
    if (kwalk_seek(P, rho, v0, vl, Uc, w)) do ++NT; while (kwalk_next(P, rho, v0, vl, Uc, BU, w));
  }
  band_init_bars(bars);
  KWalk iw{0, 0, 0, 0, 0};
  auto issue = [&](int s) {
    const uint32_t st = stages + s * kBStageB, bar = smem_u32(&bars[s]);
    mbar_expect_tx(bar, kBStageB);
    tma_load_4d(st, &mqt, 0, iw.r, iw.us, qplane, bar);
    tma_load_4d(st + kBTileB, &mdo, 0, iw.r, iw.us, qplane, bar);
    kwalk_next(P, rho, v0, vl, Uc, BU, iw);
  };
  if (threadIdx.x == 0) {
    const uint32_t kb = smem_u32(&bars[kBStages]);
    mbar_expect_tx(kb, 2 * kBTileB);
    tma_load_4d(ktile, &mk, 0, rho, v0, bg, kb);
    tma_load_4d(vtile, &mv, 0, rho, v0, bg, kb);
    kwalk_seek(P, rho, v0, vl, Uc, iw);
    for (int s = 0; s < kBStages && s < NT; ++s) issue(s);
  }
  if (!band_wait(&bars[kBStages], 0, a)) {
    band_drain(bars, NT, a);
    return;
  }
  float dk[8][4], dv[8][4];
#pragma unroll
  for (int nd = 0; nd < 8; ++nd) {
    dk[nd][0] = dk[nd][1] = dk[nd][2] = dk[nd][3] = 0.0f;
    dv[nd][0] = dv[nd][1] = dv[nd][2] = dv[nd][3] = 0.0f;
  }
  KWalk cw{0, 0, 0, 0, 0};
  kwalk_seek(P, rho, v0, vl, Uc, cw);
  // keys of this warp's 16 rows (none past the sequence)
  const int vmin = v0 + 16 * warp, vmax = min(vmin + 15, Uc - 1);

  const bool ok = band_loop(NT, stages, bars, a, issue, [&](int, uint32_t qst) {
    const uint32_t dst = qst + kBTileB;
    const int len = P.len[cw.m];
    // query u of column n reaches key v of row x iff t = u - v + e is in [0, len)
    int tb[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) tb[x] = kv[x] < Uc ? cw.e - kv[x] : -(1 << 30);
    // n-tiles (8 columns = 8 positions of one head) holding a query that reads
    // one of the warp's keys: positions [vmin - e, vmax - e + len - 1]; whole
    // halves of 32 columns are skipped
    unsigned msk = 0u;
    {
      const int ua = max(vmin - cw.e, 0) - cw.us, ub = min(vmax - cw.e + len - 1, Uc - 1) - cw.us;
      if (vmin <= vmax && ua <= ub)
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
          const int c0 = (8 * g8) % BU;
          if (c0 <= ub && c0 + 7 >= ua) msk |= 1u << g8;
        }
    }
#pragma unroll
    for (int hq = 0; hq < 2; ++hq) {  // query rows 32 hq .. 32 hq + 31 of the tile
      const unsigned mh = (msk >> (4 * hq)) & 15u;
      if (!mh) continue;
      float2 sd[4][2];
      int uq[4][2];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int n = 32 * hq + 8 * nt + 2 * tig + c;
          const int u = cw.us + n % BU;
          uq[nt][c] = u < Uc ? u : -(1 << 30);
          sd[nt][c] = __ldg(stat + (int64_t)(qplane + n / BU) * T + cw.r + delta * min(u, Uc - 1));
        }
      float st[4][4], dpt[4][4];
      {
        // the warp's K' and V rows as A fragments, from the CTA's tiles (kept
        // in shared memory rather than in 32 registers for the whole CTA)
        uint32_t ka[4][4], va[4][4];
        band_frags(ktile, 16 * warp, nullptr, 1.0f, false, ka);
        band_frags(vtile, 16 * warp, nullptr, 1.0f, false, va);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.0f;
          dpt[nt][0] = dpt[nt][1] = dpt[nt][2] = dpt[nt][3] = 0.0f;
        }
        qk_tiles4(ka, qst, 32 * hq, st);
        qk_tiles4(va, dst, 32 * hq, dpt);
      }
      // the half's query positions are ua .. ub (each head's, for G > 2); when
      // every one of them reads every key row of the warp through the run, the
      // per-element test (which would pass them all) is skipped
      const int ua = cw.us + (BU >= 32 ? (32 * hq) % BU : 0), ub = ua + min(BU, 32) - 1;
      const bool full = mh == 15u && vmin + 15 < Uc && ub < Uc && ua - (vmin + 15) + cw.e >= 0 &&
                        ub - vmin + cw.e <= len - 1;
      float pp[4][4], ds[4][4];
      if (full) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) pp[nt][e] = ex2(fmaf(st[nt][e], kLog2e, -sd[nt][e & 1].x));
      } else {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int x = e >> 1, c = e & 1;
            const bool valid = (unsigned)(uq[nt][c] + tb[x]) < (unsigned)len;
            pp[nt][e] = valid ? ex2(fmaf(st[nt][e], kLog2e, -sd[nt][c].x)) : 0.0f;
          }
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) ds[nt][e] = pp[nt][e] * (dpt[nt][e] - sd[nt][e & 1].y);
      // a key row sums P and dS over up to G x len (query, head) pairs, with
      // sum P above 1 for the early keys: both go in as bf16 hi + lo
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t ph[4], pl[4], sh[4], sl[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int nt = 2 * ks + (y >> 1), e = 2 * (y & 1);
          split_bf16(pp[nt][e], pp[nt][e + 1], ph[y], pl[y]);
          split_bf16(ds[nt][e], ds[nt][e + 1], sh[y], sl[y]);
        }
        const int rl = 32 * hq + 16 * ks + (lane & 7);
        pv_tile2(ph, pl, dst, rl, rl + 8, dv);
        pv_tile2(sh, sl, qst, rl, rl + 8, dk);
      }
    }
    kwalk_next(P, rho, v0, vl, Uc, BU, cw);
  });
  if (!ok) return;
  // dK = R(-phi_j) dK' at j = rho + delta v; dV as accumulated
  const int kpos[2] = {rho + delta * min(kv[0], Uc - 1), rho + delta * min(kv[1], Uc - 1)};
  const float one[2] = {1.0f, 1.0f};
  band_store_rows(ktile, 16 * warp, dk, one, static_cast<const float2*>(a.rope), kpos);
  band_store_rows(vtile, 16 * warp, dv, one, nullptr, kpos);
  fence_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    tma_store_4d(&mdk, 0, rho, v0, bg, ktile);
    tma_store_4d(&mdv, 0, rho, v0, bg, vtile);
    bulk_commit();
    bulk_wait_read();
  }
}

// ---- forward on the fifth-generation tensor cores (tcgen05, TMEM) -------------
//
// The same band walk with 128 query rows per CTA (G heads x 128 / G
// positions), one row per thread, and both products issued by one thread as
// tcgen05.mma with the accumulators in tensor memory:
//  * S = q~ . K'^T (M = 128, N = 64 keys, K = 64): A is the CTA's query tile,
//    rotated and scaled in shared memory once, B the staged K' tile (both
//    K-major, 128B swizzle as the TMA unit writes them); S lands in TMEM
//    columns 0..63.
//  * Each thread reads its row of S (tcgen05.ld), masks it to its band,
//    takes the online-softmax step in base 2 (the running maximum refreshed
//    only when the row's maximum exceeds it by more than 8, as in the mma.sync
//    forward), and writes its row of P in bf16 to a shared-memory tile (K-major,
//    128B swizzle).  A refresh rescales the warp's rows of O in TMEM (ld,
//    scale, st: warp-collective instructions, so every lane of the warp takes
//    part, the rows without a refresh scaled by 1).
//  * O += P . V (M = 128, N = 64 dims, K = 64 keys): B is the staged V tile,
//    MN-major; O stays in TMEM columns 64..127 until the epilogue.
// Two K'/V stages (three CTAs per SM: 65 KB of shared memory and 128 TMEM
// columns each); a stage is refilled once the P . V product that last read it
// has completed.  All waits are bounded.

constexpr int kUR = 128;                 // query rows per CTA: the TMEM lanes of M = 128
constexpr int kUStages = 2;
constexpr int kUTileB = kUR * 128;       // 16 KB: the query (then output) tile, the P tile
constexpr size_t kBandFwdTc05Smem = (size_t)2 * kUTileB + (size_t)kUStages * kBStageB + 1024;
constexpr uint32_t kUColS = 0, kUColO = 64, kUCols = 128;

template <int G>
__global__ void __launch_bounds__(kBThreads, 3)
    band_fwd_tc05_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mq,
                         const __grid_constant__ CUtensorMap mo, const __grid_constant__ BandPlan P) {
  constexpr int BU = kUR / G;  // positions per head in the tile
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bars[kUStages + 3];  // stages, query tile, S done, P.V done
  __shared__ uint32_t tmem_base;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t qtile = sbase, ptile = sbase + kUTileB, stages = sbase + 2 * kUTileB;
  const int tid = threadIdx.x, warp = tid >> 5;
  uint64_t* const qbar = &bars[kUStages];
  uint64_t* const sbar = &bars[kUStages + 1];
  uint64_t* const pvbar = &bars[kUStages + 2];

  // tile geometry: class r, compressed positions u0 .. ul; this thread's row
  const int delta = P.delta, Uc = a.T / delta, nqt = (Uc + BU - 1) / BU;
  const int r = blockIdx.x / nqt, u0 = (blockIdx.x - r * nqt) * BU, ul = min(u0 + BU - 1, Uc - 1);
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv, qplane = b * a.Hq + g * G;
  const int hrow = tid / BU, urow = u0 + tid % BU;
  const bool live = urow < Uc;
  const int pos = r + delta * min(urow, Uc - 1);
  int NT = 0;
  {
    QWalk w{0, 0, 0, 0, 0};
    if (qwalk_seek(P, r, u0, ul, Uc, w)) do ++NT; while (qwalk_next(P, r, u0, ul, Uc, w));
  }

  pdl_launch_dependents();
  if (tid == 0) {
    for (int x = 0; x < kUStages + 3; ++x) mbar_init(smem_u32(&bars[x]), 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), kUCols);
    tmem_relinquish();
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  const uint32_t tm = tmem_base;
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;  // this warp's TMEM lanes
  pdl_wait();  // the previous kernel's outputs are complete from here on

  QWalk iw{0, 0, 0, 0, 0};
  // thread 0's bookkeeping for a clean exit after a timeout: tiles issued and
  // consumed, and the last S and P . V products committed (-1: none)
  int n_issued = 0, n_consumed = 0, last_s = -1, last_pv = -1;
  auto issue = [&](int st) {
    const uint32_t sa = stages + st * kBStageB, bar = smem_u32(&bars[st]);
    mbar_expect_tx(bar, kBStageB);
    tma_load_4d(sa, &mk, 0, iw.rho, iw.vs, bg, bar);
    tma_load_4d(sa + kBTileB, &mv, 0, iw.rho, iw.vs, bg, bar);
    qwalk_next(P, r, u0, ul, Uc, iw);
    ++n_issued;
  };
  if (tid == 0) {
    mbar_expect_tx(smem_u32(qbar), kUTileB);
    tma_load_4d(qtile, &mq, 0, r, u0, qplane, smem_u32(qbar));
    qwalk_seek(P, r, u0, ul, Uc, iw);
    for (int st = 0; st < kUStages && st < NT; ++st) issue(st);
  }
  bool ok = true;
  // the query row: RoPE at its position, times 1/8, rounded to bf16 in place
  // (the rounding the backward uses for q~)
  const float2* rope = static_cast<const float2*>(a.rope);
  ok = mbar_wait_bounded(smem_u32(qbar), 0, a.wait_cycles);
  if (ok) {
    unsigned char* row = sgen + (size_t)tid * 128;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      uint4* plo = reinterpret_cast<uint4*>(row + ((ch ^ (tid & 7)) << 4));
      uint4* phi = reinterpret_cast<uint4*>(row + (((ch + 4) ^ (tid & 7)) << 4));
      uint4 lo = *plo, hi = *phi;
      uint32_t* l4 = reinterpret_cast<uint32_t*>(&lo);
      uint32_t* h4 = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 x = unpack_bf16(l4[e]), y = unpack_bf16(h4[e]);
        if (rope) {
          const float4 cs = __ldg(reinterpret_cast<const float4*>(rope + (int64_t)pos * 32 + 8 * ch + 2 * e));
          const float x0 = x.x * cs.x - y.x * cs.y, y0 = x.x * cs.y + y.x * cs.x;
          const float x1 = x.y * cs.z - y.y * cs.w, y1 = x.y * cs.w + y.y * cs.z;
          x = make_float2(x0, x1);
          y = make_float2(y0, y1);
        }
        l4[e] = pack_bf16(x.x * 0.125f, x.y * 0.125f);
        h4[e] = pack_bf16(y.x * 0.125f, y.y * 0.125f);
      }
      *plo = lo;
      *phi = hi;
    }
  }
  fence_async_smem();
  tc05_fence_before();
  ok = !__syncthreads_or(!ok);
  tc05_fence_after();

  constexpr uint32_t idS = idesc_bf16(kUR, 64, false, false);
  constexpr uint32_t idPV = idesc_bf16(kUR, 64, false, true);
  float m = -INFINITY, l = 0.0f;
  QWalk cw{0, 0, 0, 0, 0};
  qwalk_seek(P, r, u0, ul, Uc, cw);
  // S_t = q~ . K'_t^T into TMEM columns 0..63 (thread 0).  S_{t+1} is issued
  // right after P_t . V_t: every thread holds S_t in registers by then, and
  // the tensor cores run both products while the threads go on.
  auto issue_s = [&](int t) {
    const int st = t % kUStages;
    const uint32_t kst = stages + st * kBStageB;
    if (!mbar_wait_bounded(smem_u32(&bars[st]), (t / kUStages) & 1, a.wait_cycles)) {
      record_status(a.status, SFA_ERR_TIMEOUT);  // the S wait of every thread then runs out
      return;
    }
    n_consumed = t + 1;
    tc05_fence_after();
#pragma unroll
    for (int k = 0; k < 4; ++k)
      umma_bf16(tm + kUColS, smem_desc_sw128(qtile + 32 * k, 16, 1024),
                smem_desc_sw128(kst + 32 * k, 16, 1024), idS, k > 0);
    umma_commit(smem_u32(sbar));
    last_s = t;
  };
  if (tid == 0 && ok && NT > 0) issue_s(0);
  for (int t = 0; t < NT && ok; ++t) {
    const uint32_t vst = stages + (t % kUStages) * kBStageB + kBTileB;
    bool okw = mbar_wait_bounded(smem_u32(sbar), t & 1, a.wait_cycles);
    tc05_fence_after();
    // this row's keys in the tile: columns lo .. hi of the current run; a
    // 16-column chunk no row of the warp reads is neither loaded nor
    // exponentiated (warp-uniform: the TMEM loads are warp-collective)
    const int len = P.len[cw.m];
    const int lo = urow + cw.e - len + 1 - cw.vs, hi = live ? min(urow + cw.e, Uc - 1) - cw.vs : -1;
    bool chunk[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) chunk[q] = __any_sync(0xffffffffu, lo <= 16 * q + 15 && hi >= 16 * q);
    float sv[64];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (chunk[q]) tmem_ld16(tm + lane_base + kUColS + 16 * q, sv + 16 * q);
    tmem_wait_ld();
    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      sv[c] = (chunk[c >> 4] && c >= lo && c <= hi) ? sv[c] * kLog2e : -INFINITY;
      mx4[c & 3] = fmaxf(mx4[c & 3], sv[c]);
    }
    const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
    // the previous P . V has finished: O is stable and the P tile is free
    if (t > 0) {
      okw &= mbar_wait_bounded(smem_u32(pvbar), (t - 1) & 1, a.wait_cycles);
      tc05_fence_after();
      // its K'/V stage is free: refill it with tile t - 1 + kUStages
      if (tid == 0 && t - 1 + kUStages < NT) issue((t - 1) % kUStages);
    }
    // refresh the running maximum (m = -inf: any valid logit); the TMEM
    // moves are warp-collective, so a warp rescales its rows of O when any of
    // them refreshes (by 1 for the others)
    const bool refresh = mx > m + 8.0f;
    float corr = 1.0f;
    if (refresh) {
      corr = ex2(m - mx);  // 0 while the row had no key
      l *= corr;
      m = mx;
    }
    if (t > 0 && __any_sync(0xffffffffu, refresh)) {
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        float ov[16];
        tmem_ld16(tm + lane_base + kUColO + c, ov);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) ov[e] *= corr;
        tmem_st16(tm + lane_base + kUColO + c, ov);
      }
      tmem_wait_st();
    }
    const float mm = m == -INFINITY ? 0.0f : m;
    unsigned char* prow = sgen + kUTileB + (size_t)tid * 128;
    float lt[2] = {0.0f, 0.0f};
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      uint32_t w4[4] = {0u, 0u, 0u, 0u};
      if (chunk[ch >> 1]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2(sv[8 * ch + 2 * e] - mm), p1 = ex2(sv[8 * ch + 2 * e + 1] - mm);
          lt[e & 1] += p0 + p1;
          w4[e] = pack_bf16(p0, p1);
        }
      }
      *reinterpret_cast<uint4*>(prow + ((ch ^ (tid & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    l += lt[0] + lt[1];
    fence_async_smem();
    tc05_fence_before();
    ok = !__syncthreads_or(!okw);
    if (!ok) {
      if (tid == 0) record_status(a.status, SFA_ERR_TIMEOUT);
      break;
    }
    // O += P . V into TMEM columns 64..127 (V MN-major: 16 keys = two 8-row
    // groups), then S_{t+1}
    if (tid == 0) {
      tc05_fence_after();
#pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_bf16(tm + kUColO, smem_desc_sw128(ptile + 32 * k, 16, 1024),
                  smem_desc_sw128(vst + 2048 * k, 8192, 1024), idPV, t > 0 || k > 0);
      umma_commit(smem_u32(pvbar));
      last_pv = t;
      if (t + 1 < NT) issue_s(t + 1);
    }
    qwalk_next(P, r, u0, ul, Uc, cw);
  }
  if (ok && NT > 0) ok = mbar_wait_bounded(smem_u32(pvbar), (NT - 1) & 1, a.wait_cycles);
  ok = !__syncthreads_or(!ok);
  tc05_fence_after();
  if (ok) {
    // O = acc / l and LSE; the row goes out through the query tile's space
    float ov[64];
#pragma unroll
    for (int c = 0; c < 64; c += 16) tmem_ld16(tm + lane_base + kUColO + c, ov + c);
    tmem_wait_ld();
    const float inv = NT > 0 ? 1.0f / l : 0.0f;
    if (live)
      a.out_lse[(int64_t)(qplane + hrow) * a.T + pos] = NT > 0 ? (m + log2f(l)) * kLn2 : -INFINITY;
    unsigned char* orow = sgen + (size_t)tid * 128;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      uint32_t w4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) w4[e] = pack_bf16(ov[8 * ch + 2 * e] * inv, ov[8 * ch + 2 * e + 1] * inv);
      *reinterpret_cast<uint4*>(orow + ((ch ^ (tid & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    fence_async_smem();
  } else if (tid == 0) {
    record_status(a.status, SFA_ERR_TIMEOUT);
    // wait (bounded) for the loads still in flight (at most one per stage) and
    // the last products committed, before the TMEM and the CTA go away
    for (int x = n_consumed; x < n_issued; ++x)
      mbar_wait_bounded(smem_u32(&bars[x % kUStages]), (x / kUStages) & 1, a.wait_cycles);
    if (last_s >= 0) mbar_wait_bounded(smem_u32(sbar), last_s & 1, a.wait_cycles);
    if (last_pv >= 0) mbar_wait_bounded(smem_u32(pvbar), last_pv & 1, a.wait_cycles);
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  if (warp == 0) tmem_dealloc(tm, kUCols);
  if (ok && tid == 0) {
    tma_store_4d(&mo, 0, r, u0, qplane, qtile);
    bulk_commit();
    bulk_wait_read();
  }
}

// ---- launchers ---------------------------------------------------------------

template <int G>
static int band_fwd_launch(const AttnArgs& a, const BandPlan& p, const void* kr, cudaStream_t s) {
  if (a.band_tc05) {  // tcgen05 forward: 128 query rows per CTA
    constexpr int BU = kUR / G;
    CUtensorMap mk, mv, mq, mo;
    const int64_t planes = (int64_t)a.B * a.Hkv, qplanes = (int64_t)a.B * a.Hq;
    if (make_band_map(&mk, kr, planes, a.T, p.delta, kBR, 1) != SFA_OK ||
        make_band_map(&mv, a.v, planes, a.T, p.delta, kBR, 1) != SFA_OK ||
        make_band_map(&mq, a.q, qplanes, a.T, p.delta, BU, G) != SFA_OK ||
        make_band_map(&mo, a.out_o, qplanes, a.T, p.delta, BU, G) != SFA_OK)
      return SFA_ERR_CUDA;
    if (cudaFuncSetAttribute(band_fwd_tc05_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kBandFwdTc05Smem) != cudaSuccess)
      return SFA_ERR_CUDA;
    const int Uc = a.T / p.delta;
    dim3 grid((unsigned)(p.delta * ((Uc + BU - 1) / BU)), (unsigned)(a.B * a.Hkv));
    LaunchTimer tm(SFA_KERNEL_FWD, s);
    return launch_pdl(band_fwd_tc05_kernel<G>, grid, dim3(kBThreads), kBandFwdTc05Smem, s, a, mk, mv,
                      mq, mo, p) == cudaSuccess
               ? SFA_OK
               : SFA_ERR_CUDA;
  }
  constexpr int BU = kBR / G;
  CUtensorMap mk, mv, mq, mo;
  const int64_t planes = (int64_t)a.B * a.Hkv, qplanes = (int64_t)a.B * a.Hq;
  if (make_band_map(&mk, kr, planes, a.T, p.delta, kBR, 1) != SFA_OK ||
      make_band_map(&mv, a.v, planes, a.T, p.delta, kBR, 1) != SFA_OK ||
      make_band_map(&mq, a.q, qplanes, a.T, p.delta, BU, G) != SFA_OK ||
      make_band_map(&mo, a.out_o, qplanes, a.T, p.delta, BU, G) != SFA_OK)
    return SFA_ERR_CUDA;
  if (cudaFuncSetAttribute(band_fwd_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kBandFwdSmem) != cudaSuccess)
    return SFA_ERR_CUDA;
  const int Uc = a.T / p.delta;
  dim3 grid((unsigned)(p.delta * ((Uc + BU - 1) / BU)), (unsigned)(a.B * a.Hkv));
  LaunchTimer tm(SFA_KERNEL_FWD, s);
  return launch_pdl(band_fwd_kernel<G>, grid, dim3(kBThreads), kBandFwdSmem, s, a, mk, mv, mq, mo,
                    p) == cudaSuccess
             ? SFA_OK
             : SFA_ERR_CUDA;
}

int launch_band_forward(const AttnArgs& a, const BandPlan& p, const void* kr, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  switch (a.lgG) {
    case 0: return band_fwd_launch<1>(a, p, kr, s);
    case 1: return band_fwd_launch<2>(a, p, kr, s);
    case 2: return band_fwd_launch<4>(a, p, kr, s);
    case 3: return band_fwd_launch<8>(a, p, kr, s);
    default: return SFA_ERR_UNSUPPORTED;
  }
}

size_t band_backward_workspace_bytes(const sfa_desc* d, size_t* off_kr, size_t* off_qt,
                                     size_t* off_stat) {
  const size_t qrows = (size_t)d->B * d->Hq * d->T;
  *off_kr = 0;
  *off_qt = kr_bytes(d);
  *off_stat = *off_qt + align256(qrows * 64 * 2);
  return *off_stat + align256(qrows * sizeof(float2));
}

template <int G>
static int band_bwd_launch(const AttnArgs& a, const BandPlan& p, const void* kr, void* qt,
                           void* stat, cudaStream_t s) {
  constexpr int BU = kBR / G;
  CUtensorMap mk, mv, mq, mdo, mo, mqt, mdq, mdk, mdv;
  const int64_t planes = (int64_t)a.B * a.Hkv, qplanes = (int64_t)a.B * a.Hq;
  const int T = a.T, dl = p.delta;
  if (make_band_map(&mk, kr, planes, T, dl, kBR, 1) != SFA_OK ||
      make_band_map(&mv, a.v, planes, T, dl, kBR, 1) != SFA_OK ||
      make_band_map(&mq, a.q, qplanes, T, dl, BU, G) != SFA_OK ||
      make_band_map(&mdo, a.dO, qplanes, T, dl, BU, G) != SFA_OK ||
      make_band_map(&mo, a.o, qplanes, T, dl, BU, G) != SFA_OK ||
      make_band_map(&mqt, qt, qplanes, T, dl, BU, G) != SFA_OK ||
      make_band_map(&mdq, a.dq, qplanes, T, dl, BU, G) != SFA_OK ||
      make_band_map(&mdk, a.dk, planes, T, dl, kBR, 1) != SFA_OK ||
      make_band_map(&mdv, a.dv, planes, T, dl, kBR, 1) != SFA_OK)
    return SFA_ERR_CUDA;
  if (cudaFuncSetAttribute(band_bwd_q_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kBandBwdQSmem) != cudaSuccess ||
      cudaFuncSetAttribute(band_bwd_kv_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kBandBwdKvSmem) != cudaSuccess)
    return SFA_ERR_CUDA;
  const int Uc = T / dl;
  float2* st = static_cast<float2*>(stat);
  {
    dim3 grid((unsigned)(dl * ((Uc + BU - 1) / BU)), (unsigned)(a.B * a.Hkv));
    LaunchTimer tm(SFA_KERNEL_BWD_Q, s);
    if (launch_pdl(band_bwd_q_kernel<G>, grid, dim3(kBThreads), kBandBwdQSmem, s, a, mk, mv, mq, mdo,
                   mo, mqt, mdq, st, p) != cudaSuccess)
      return SFA_ERR_CUDA;
  }
  dim3 grid((unsigned)(dl * ((Uc + kBR - 1) / kBR)), (unsigned)(a.B * a.Hkv));
  LaunchTimer tm(SFA_KERNEL_BWD_KV, s);
  return launch_pdl(band_bwd_kv_kernel<G>, grid, dim3(kBThreads), kBandBwdKvSmem, s, a, mk, mv, mqt,
                    mdo, mdk, mdv, static_cast<const float2*>(st), p) == cudaSuccess
             ? SFA_OK
             : SFA_ERR_CUDA;
}

int launch_band_backward(const AttnArgs& a, const BandPlan& p, const void* kr, void* qt,
                         void* stat, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  switch (a.lgG) {
    case 0: return band_bwd_launch<1>(a, p, kr, qt, stat, s);
    case 1: return band_bwd_launch<2>(a, p, kr, qt, stat, s);
    case 2: return band_bwd_launch<4>(a, p, kr, qt, stat, s);
    case 3: return band_bwd_launch<8>(a, p, kr, qt, stat, s);
    default: return SFA_ERR_UNSUPPORTED;
  }
}

}  // namespace sfa
