// Tensor-core backward (bf16 I/O, G = 4, 8 or 16 in groups of 4 query heads;
// the key side sums the groups of its KV head): gradients of L = sum(O * dO) for
// the key set of "Depth-Staggered Fibonacci Spacing for Sparse Attention"
// (method section), the same quantities as the SIMT backward.
//
// bwd_q_tc (per query tile, the forward's warp layout and slab staging):
//   S = q~.K'^T and dP = dO.V^T from raw rows (a rung's two raw values are
//   interpolated on the fragment), P = exp(S - LSE), dS = P (dP - delta);
//   dQ += dS~.K' (dS~ = dS split (1 - w, w) over a rung's two rows), then
//   dQ = R(-phi) dQ / 8.  dL/dd_k = dS (q~.K'[i-c] - q~.K'[i-c+1])
//   + P (dO.V[i-c] - dO.V[i-c+1]) comes from the same raw fragments.  For
//   the key side it writes q~ = q'/8 (bf16) and, per (query, slot, head),
//   the pair (P, dS) as a key-side-ready record (bf16 at G = 4, bf16 hi + lo
//   at G > 4; a rung gets one record per role: weight 1 - w for key i - c, w
//   for key i - c + 1).
// bwd_kv_tc (per key tile): dK^T and dV^T accumulate as [64 dims x 8 keys]
//   mma tiles per warp: A = q~^T or dO^T (TMA-staged slabs) of the (query,
//   head) pairs that read the warp's 8 key rows, B = their (dS, P)
//   coefficients (the records, also TMA-staged): a window
//   slot s reaches key i - s; a rung (c, w) reaches key i - c with weight
//   1 - w and key i - c + 1 with weight w.  Each key row is written by one
//   warp: no atomics.
#include <math.h>

#include <type_traits>

#include "sfa_tc.cuh"

namespace sfa {

// A record of key-side coefficients for a (query, slot) is two halves, one
// per head pair (0, 2) and (1, 3), each word holding the pair's two heads
// (lower head in the low half).  With G = 4 a half is 8 bytes, the pair's
// wt * dS and wt * P in bf16 (words: dS, P).  With G > 4 (LO) a key sums G
// heads' coefficients, and a half is 16 bytes, both as bf16 hi + lo
// (hi = bf16(x), lo = bf16(x - hi); words: dS hi, dS lo, P hi, P lo).  The
// lane whose fragment rows are the pair's two heads writes its half
// directly.
template <bool LO>
struct CoefFmt {
  using Half = typename std::conditional<LO, uint4, uint2>::type;
  static constexpr int kHalfWords = LO ? 4 : 2;
  static constexpr int kRecWords = 2 * kHalfWords;
  static constexpr int kRecBytes = 4 * kRecWords;
};
__device__ __forceinline__ void write_coef_half(uint4* dst, float wt, float ds0, float ds1, float p0,
                                                float p1) {
  const float a0 = wt * ds0, a1 = wt * ds1, b0 = wt * p0, b1 = wt * p1;
  const uint32_t dh = pack_bf16(a0, a1), ph = pack_bf16(b0, b1);
  const float2 dhf = unpack_bf16(dh), phf = unpack_bf16(ph);
  *dst = make_uint4(dh, pack_bf16(a0 - dhf.x, a1 - dhf.y), ph, pack_bf16(b0 - phf.x, b1 - phf.y));
}
__device__ __forceinline__ void write_coef_half(uint2* dst, float wt, float ds0, float ds1, float p0,
                                                float p1) {
  *dst = make_uint2(pack_bf16(wt * ds0, wt * ds1), pack_bf16(wt * p0, wt * p1));
}

// PSI (G > 4): also sum psi = sum_j P_ij dP_ij per row and write delta - psi
// for the key side's correction (a.dcorr); records carry hi + lo words.
template <bool INTERP, bool PSI>
__global__ void __launch_bounds__(kTcThreads, 4)
    bwd_q_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mq,
                    const __grid_constant__ CUtensorMap mdo, const __grid_constant__ CUtensorMap mo,
                    const __grid_constant__ CUtensorMap mqt,
                    const __grid_constant__ CUtensorMap mdq, uint32_t* coef, int NS,
                    const __grid_constant__ Plan P) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bars[kTcStages + 1];
  __shared__ double red[kTcWarps];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  // qy = (batch, group g of 4 query heads); with G = 4m query heads per KV head
  // the group reads KV head g / m; its records form plane qy.  Planes run in
  // reverse launch order: the forward ended on the last planes, whose O and
  // LSE are the likeliest to be still in L2, and the key side, which starts
  // on the first planes, finds their records there
  const int qy = gridDim.y - 1 - blockIdx.y;
  const int ng4 = a.Hq >> 2, b = qy / ng4, g = qy - b * ng4;
  const int bg = b * a.Hkv + (g >> (a.lgG - 2));
  const int T = a.T;
  const int i0 = blockIdx.x * kTcTQ, i0w = i0 + 4 * warp;
  const int p = gid & 3, i = i0w + p;
  const int ic = min(i, T - 1);
  const bool act = i < T;
  const int imax = min(T - 1, i0 + kTcTQ - 1);
  const int hA = g * 4 + (gid >> 2), hB = hA + 2;
  const int64_t rowA = (int64_t)(b * a.Hq + hA) * T + ic, rowB = (int64_t)(b * a.Hq + hB) * T + ic;
  const float2* rope = static_cast<const float2*>(a.rope);

  const int wmax = min(P.W, imax);
  const int nwc = wmax >= 0 ? wmax / kTcWC + 1 : 0;
  const int nr = rungs_upto(P, imax);
  const int NG = nwc + (nr + 1) / 2;
  const uint32_t qtile = sbase, dotile = sbase + kTcQTileB, otile = sbase + 2 * kTcQTileB;
  const uint32_t stages = sbase + 3 * kTcQTileB;
  const int qplane = b * a.Hq + g * 4;
  const int skip_grp = (blockIdx.x | blockIdx.y) == 0 ? a.debug_skip : -1;  // test injection
  const CUtensorMap* qmaps[3] = {&mq, &mdo, &mo};
  tc_start(&mk, &mv, qmaps, 3, qtile, qplane, P, bg, i0, nwc, nr, NG, stages, bars, skip_grp);

  uint32_t qa[4][4], da[4][4];
  float delta[2], lse2[2];
  lse2[0] = a.lse[rowA] * kLog2e;
  lse2[1] = a.lse[rowB] * kLog2e;
  float4 rp[4];
  if (rope) load_frag_rope(rope, ic, rp);  // while the query tiles are in flight
  if (!tc_wait_qtiles(bars, a)) return;
  tile_frags(qtile, warp, rope ? rp : nullptr, 0.125f, true, qa);
  tile_frags(dotile, warp, nullptr, 1.0f, false, da);
  {  // delta = dO . O per row: the diagonal of dO . O^T over the warp's 16 rows, by
     // two tensor-core tiles (columns = rows 0..7 and 8..15 of the O tile); the
     // diagonal element of row gid (gid + 8) sits in lane 4 gid + gid / 2, column
     // gid & 1 of the first (second) tile
    float dd[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int r = 8 * nt + (lane & 7);
      qk_tile(da, otile, (r >> 2) * kTcQRows + 4 * warp + (r & 3), dd[nt]);
    }
    const float mine0 = (gid & 1) ? dd[0][1] : dd[0][0], mine1 = (gid & 1) ? dd[1][3] : dd[1][2];
    const int src = 4 * gid + (gid >> 1);
    delta[0] = __shfl_sync(0xffffffffu, mine0, src);
    delta[1] = __shfl_sync(0xffffffffu, mine1, src);
  }
  __syncthreads();  // the dO tile is read: it now carries q~ = q'/8 out for the key side
  {  // the A fragments are the output layout: k-step kk holds dims 16 kk .. 16 kk + 15
    const uint32_t pk[8][2] = {{qa[0][0], qa[0][1]}, {qa[0][2], qa[0][3]}, {qa[1][0], qa[1][1]},
                               {qa[1][2], qa[1][3]}, {qa[2][0], qa[2][1]}, {qa[2][2], qa[2][3]},
                               {qa[3][0], qa[3][1]}, {qa[3][2], qa[3][3]}};
    store_otile(dotile, warp, pk);
  }
  fence_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) tc_store_tile(&mqt, dotile, i0, qplane);
  float dq[8][4];
#pragma unroll
  for (int nd = 0; nd < 8; ++nd) dq[nd][0] = dq[nd][1] = dq[nd][2] = dq[nd][3] = 0.0f;
  float dacc = 0.0f;
  // psi = sum_j P_ij dP_ij per row (this lane's keys), equal to dO . O for the
  // exact O: the key side of G > 4 corrects its dS by P (delta - psi)
  float psi[2] = {0.0f, 0.0f};
  // records of query i: [slot][2 halves]; this lane's rows gid, gid + 8 are
  // heads hA, hA + 2 of position p, i.e. half gid >> 2 of each record
  using Half = typename CoefFmt<PSI>::Half;
  Half* crow = reinterpret_cast<Half*>(coef) + ((int64_t)qy * T + ic) * NS * 2 + (gid >> 2);

  const int colrow = 4 * warp + ((lane & 7) >> 1) + (lane & 1);
  const int colrow2 = 4 * warp + ((((lane & 7) >> 1) + 2) & 3) + (lane & 1);

  const bool ok = tc_run(&mk, &mv, P, bg, i0, nwc, nr, NG, stages, bars, a, skip_grp,
                              [&](int grp, uint32_t kst, uint32_t vst) {
    uint32_t sa[4];
    if (grp < nwc) {
      const int s_lo = kTcWC * grp, s_hi = min(s_lo + kTcWC - 1, P.W);
      float sc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}}, dp[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int row = 4 * warp + 8 * nt + (lane & 7);
        qk_tile(qa, kst, row, sc[nt]);
        qk_tile(da, vst, row, dp[nt]);
      }
      float ds[2][4], pp[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = e >> 1;
          const int dist = p + 12 + s_lo - (8 * nt + 2 * tig + (e & 1));
          const bool v = act && dist >= s_lo && dist <= s_hi && dist <= i;
          const float pr = v ? ex2(fmaf(sc[nt][e], kLog2e, -lse2[r])) : 0.0f;
          ds[r][2 * nt + (e & 1)] = pr * (dp[nt][e] - delta[r]);
          pp[r][2 * nt + (e & 1)] = pr;
          if (PSI) psi[r] = fmaf(pr, dp[nt][e], psi[r]);
        }
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int dist = p + 12 + s_lo - (8 * (cc >> 1) + 2 * tig + (cc & 1));
        if (act && dist >= s_lo && dist <= s_hi && dist <= i)
          write_coef_half(crow + 2 * dist, 1.0f, ds[0][cc], ds[1][cc], pp[0][cc], pp[1][cc]);
      }
      sa[0] = pack_bf16(ds[0][0], ds[0][1]);
      sa[1] = pack_bf16(ds[1][0], ds[1][1]);
      sa[2] = pack_bf16(ds[0][2], ds[0][3]);
      sa[3] = pack_bf16(ds[1][2], ds[1][3]);
      pv_tile(sa, kst, 4 * warp + (lane & 7), 4 * warp + 8 + (lane & 7), dq);
    } else if (!INTERP) {
      // integer rung pair (w = 0): one tile per product, column (rung x,
      // position p') = raw row 4w + p' of box x (the forward's layout); the
      // lane of this row's position p holds rung tig >> 1 at column p & 1 when
      // tig & 1 == p >> 1.  Role 0 only: the key side reads no role 1
      const int r0 = 2 * (grp - nwc), rg = r0 + (tig >> 1), e = p & 1;
      float sc[4] = {0, 0, 0, 0}, dpv[4] = {0, 0, 0, 0};
      qk_tile(qa, kst, int_pair_row(warp), sc);
      qk_tile(da, vst, int_pair_row(warp), dpv);
      const bool v = act && (tig & 1) == (p >> 1) && rg < nr && i >= P.c[min(rg, P.n - 1)];
      float ds[2], prr[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float a0 = e ? sc[2 * r + 1] : sc[2 * r], b0 = e ? dpv[2 * r + 1] : dpv[2 * r];
        const float pr = v ? ex2(fmaf(a0, kLog2e, -lse2[r])) : 0.0f;
        ds[r] = pr * (b0 - delta[r]);
        prr[r] = pr;
        if (PSI) psi[r] = fmaf(pr, b0, psi[r]);
      }
      if (v) write_coef_half(crow + 2 * (P.W + 1 + 2 * rg), 1.0f, ds[0], ds[1], prr[0], prr[1]);
      const uint32_t sk8[2] = {pack_bf16(e ? 0.0f : ds[0], e ? ds[0] : 0.0f),
                               pack_bf16(e ? 0.0f : ds[1], e ? ds[1] : 0.0f)};
      pv_tile_k8(sk8, kst, int_pair_row(warp), dq);
    } else {
      // rung pair; box 1's B columns rotate positions by two, so the lane of
      // position p holding a rung's raw pair is tig == p (box 0) or
      // tig == p + 2 (box 1): one pass of the per-rung work serves both
      const int r0 = 2 * (grp - nwc);
      float sc0[4] = {0, 0, 0, 0}, dp0[4] = {0, 0, 0, 0}, sc1[4] = {0, 0, 0, 0}, dp1[4] = {0, 0, 0, 0};
      qk_tile(qa, kst, colrow, sc0);
      qk_tile(da, vst, colrow, dp0);
      qk_tile(qa, kst, kTcBoxRows + colrow2, sc1);
      qk_tile(da, vst, kTcBoxRows + colrow2, dp1);
      const bool own0 = tig == p, own1 = tig == ((p + 2) & 3);
      const int rg = own1 ? r0 + 1 : r0;
      const float w0 = (INTERP && r0 < nr) ? P.w[r0] : 0.0f;
      const float w1 = (INTERP && r0 + 1 < nr) ? P.w[r0 + 1] : 0.0f;
      const float f0 = (INTERP && r0 < nr) ? P.f[r0] : 0.0f;
      const float f1 = (INTERP && r0 + 1 < nr) ? P.f[r0 + 1] : 0.0f;
      const float w = own1 ? w1 : w0, f = own1 ? f1 : f0;
      const bool v = act && (own0 || own1) && rg < nr && i >= P.c[min(rg, P.n - 1)];
      float ds[2], prr[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float a0 = own1 ? sc1[2 * r] : sc0[2 * r], a1 = own1 ? sc1[2 * r + 1] : sc0[2 * r + 1];
        const float b0 = own1 ? dp1[2 * r] : dp0[2 * r], b1 = own1 ? dp1[2 * r + 1] : dp0[2 * r + 1];
        const float sr = fmaf(w, a1, (1.0f - w) * a0);
        const float dpi = fmaf(w, b1, (1.0f - w) * b0);
        const float pr = v ? ex2(fmaf(sr, kLog2e, -lse2[r])) : 0.0f;
        const float d = pr * (dpi - delta[r]);
        ds[r] = d;
        prr[r] = pr;
        if (PSI) psi[r] = fmaf(pr, dpi, psi[r]);
        if (INTERP && v) dacc = fmaf(f, fmaf(d, a0 - a1, pr * (b0 - b1)), dacc);
      }
      if (v) {  // role 0: key i - c (weight 1 - w); role 1: key i - c + 1 (weight w)
        write_coef_half(crow + 2 * (P.W + 1 + 2 * rg), 1.0f - w, ds[0], ds[1], prr[0], prr[1]);
        if (INTERP)  // an integer rung has no role 1 (w = 0); the key side does not read it
          write_coef_half(crow + 2 * (P.W + 2 + 2 * rg), w, ds[0], ds[1], prr[0], prr[1]);
      }
      const uint32_t lo = pack_bf16(ds[0] * (1.0f - w), ds[0] * w);
      const uint32_t hi = pack_bf16(ds[1] * (1.0f - w), ds[1] * w);
      sa[0] = own1 ? 0u : lo;  // k 0..7: box 0 (zero when the lane owns neither)
      sa[1] = own1 ? 0u : hi;
      sa[2] = own1 ? lo : 0u;  // k 8..15: box 1
      sa[3] = own1 ? hi : 0u;
      pv_tile(sa, kst, colrow, kTcBoxRows + colrow2, dq);
    }
  });
  if (!ok) return;

  if (PSI) {  // delta - psi per (row, head), for the key side's correction
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      psi[r] += __shfl_xor_sync(0xffffffffu, psi[r], 1);
      psi[r] += __shfl_xor_sync(0xffffffffu, psi[r], 2);
    }
    if (tig == 0 && act) {
      a.dcorr[rowA] = delta[0] - psi[0];
      a.dcorr[rowB] = delta[1] - psi[1];
    }
  }

  if (INTERP && a.dalpha_out) {
    // per-CTA partial of dL/dalpha; the key-side kernel, which runs after this
    // one, sums the partials in a fixed order (deterministic)
    double d = (double)dacc;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_down_sync(0xffffffffu, d, off);
    if (lane == 0) red[warp] = d;
    __syncthreads();
    if (threadIdx.x == 0) {
      double sum = 0.0;
      for (int x = 0; x < kTcWarps; ++x) sum += red[x];
      a.dalpha_part[(int64_t)qy * gridDim.x + blockIdx.x] = sum;
    }
  }
  // dQ = R(-phi) dq / 8 (dims d in tile nd and d + 32 in tile nd + 4 share a
  // lane), out through the Q tile's space and one TMA store
  uint32_t pk[8][2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float v[8][2];
#pragma unroll
    for (int nd = 0; nd < 8; ++nd) {
      v[nd][0] = dq[nd][2 * r] * 0.125f;
      v[nd][1] = dq[nd][2 * r + 1] * 0.125f;
    }
    if (rope) {
#pragma unroll
      for (int nd = 0; nd < 4; ++nd) {
        const float4 cs = rp[nd];  // the pairs 8 nd + 2 tig (+1) loaded for the fragments
        const float c2[2] = {cs.x, cs.z}, s2[2] = {cs.y, cs.w};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float lo = v[nd][e], hi = v[nd + 4][e];
          v[nd][e] = lo * c2[e] + hi * s2[e];
          v[nd + 4][e] = hi * c2[e] - lo * s2[e];
        }
      }
    }
#pragma unroll
    for (int nd = 0; nd < 8; ++nd) pk[nd][r] = pack_bf16(v[nd][0], v[nd][1]);
  }
  store_otile(qtile, warp, pk);
  fence_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    tc_store_tile(&mdq, qtile, i0, qplane);
    bulk_wait_read();  // the q~ and dQ tiles have been read
  }
}

constexpr int kKvTK = 32;                     // key rows per CTA
constexpr int kKvThreads = 128;               // 4 warps: 8 key rows each, all 64 dims
constexpr int kKvMT = 4;                      // dK / dV m-tiles per warp (16 dims each)
// A rung group reaches queries j + c - 1 .. j + c + 31 (33 rows); 34 rows keep
// the plane stride at 2 (mod 8), so the 128B swizzle puts the 8 (query, head)
// rows of one ldmatrix tile on distinct banks.  Each warp reads 12 of them (3
// k-steps), from row min(8 kw, 22) on, which covers its keys' 9 queries
// 8 kw .. 8 kw + 8.
constexpr int kKvQR = kKvTK + 2;
constexpr int kKvStages = 2;

// Stage layout of the key side.  A window chunk of WC = 9 distances reaches
// queries j0 + s_lo .. j0 + 31 + s_lo + 8, staged as Q = 42 rows per head plane
// (Q = 2 mod 8 again); a warp reads WKS = 4 k-steps of them from row
// min(8 kw, Q - 4 WKS) on.  A rung group stages 34 rows ([4 heads][34][128 B]
// for q~ and for dO) and its records.
//
// G = 4 (16-byte records, SPLIT): a window chunk runs as two pipeline groups,
// its q~ slab with the records (the dK products; the lane's dV coefficients
// are kept in registers) and then its dO slab (the dV products), so every
// stage fits in 36 KB (a rung group: 2 x 17 KB + 1 KB of records) and three
// CTAs (12 warps) stay on an SM, while the window's rows are staged once.
// G > 4 (32-byte records) stages a window chunk's two slabs and records
// together in 54 KB stages, two CTAs per SM.
template <bool MULTI>
struct KvLayout {
  static constexpr bool SPLIT = !MULTI;
  static constexpr int WC = 9;
  static constexpr int Q = kKvTK + 10;
  static constexpr int WKS = 4;
  static constexpr int PlaneB = Q * 4 * 128;                       // a window slab (q~ or dO)
  static constexpr int WRecB = Q * WC * CoefFmt<MULTI>::kRecBytes;  // a window chunk's records
  static constexpr int RDoff = MULTI ? PlaneB : kKvQR * 4 * 128;   // a rung group's dO slab
  static constexpr int StageB = MULTI ? 2 * PlaneB + 12288 : 36864;
  static constexpr int MinBlocks = MULTI ? 2 : 3;
  static constexpr size_t Smem = (size_t)kKvStages * StageB + 1024;
  static_assert(Q % 8 == 2 && kKvQR % 8 == 2, "slab strides 2 (mod 8)");
  static_assert((SPLIT ? PlaneB : 2 * PlaneB) + WRecB <= StageB, "window chunk fits a stage");
  static_assert(2 * RDoff + kKvQR * 2 * CoefFmt<MULTI>::kRecBytes <= StageB, "rung group fits a stage");
  static_assert(PlaneB % 1024 == 0 && RDoff % 1024 == 0 && StageB % 1024 == 0,
                "swizzled boxes sit on 1024-byte periods");
};

// Bits m of the query offsets ql = m + t1 (t1 = tig >> 1) with lo <= ql <= hi.
__device__ __forceinline__ uint32_t ql_mask(int lo, int hi, int t1) {
  lo = max(lo - t1, 0);
  hi = min(hi - t1, 31);
  return lo > hi ? 0u : (0xffffffffu >> (31 - hi)) & (0xffffffffu << lo);
}

// One group's products for a warp: NKS k-steps of 16 (query, head) pairs.
// dk / dv hold the warp's 4 m-tiles (dims 16 mt .. 16 mt + 15): the record
// selection of a lane's key is done once for all 64 dims.
//
// B: the records of the (query, head) pairs k = 2 tig, 2 tig + 1 (+8) that
// reach the lane's key j.  Within a query the k order of the heads is 0, 2,
// 1, 3, so the pair of lane tig is record half tig & 1 (heads tig & 1 and
// (tig & 1) + 2), and k-step ks, half hb reads query offset
// ql = 4 ks + 2 hb + (tig >> 1) from qw.  Which slot of that query reaches
// key j depends only on ql - (j - qw): bit m = ql - (tig >> 1) of `mask` says
// whether it is a slot of this group at all (and inside the sequence), and
// its record half sits at word rec + m * STEP of the staged records.
//
// FOLD (G > 4): records carry hi + lo words; corr points at delta - psi of
// the group's 4 query heads ([4][T], written by the query side), and each dS
// coefficient becomes wt dS + (wt P)(delta - psi) = wt P (dP - psi): the dS of
// the exact delta = sum_j P_ij dP_ij instead of dO . O from the bf16-rounded
// O, whose error the key side would otherwise sum over G heads.  The
// correction is folded into the lo word.
//
// ONEHOT (a rung group): the lane's two query offsets that reach its key are
// consecutive, so at most one of the (k-step, half) entries it reads (query
// offsets of one parity) is set: one record load (and with FOLD one pair of
// corrections), then selects.
//
// PASS 0 runs both products; PASS 1 (a split window chunk's q~ slab) runs the
// dK products and keeps the lane's dV coefficients in bsave; PASS 2 (its dO
// slab, in dst) runs the dV products from bsave.
template <int NKS, int STEP, bool FOLD, bool ONEHOT = false, int PASS = 0>
__device__ __forceinline__ void kv_group(uint32_t qst, uint32_t dst, const uint32_t* csm, int rec,
                                         uint32_t mask, int qw, int kq, int qoff, int T,
                                         const float* corr, float (*dk)[4], float (*dv)[4],
                                         uint32_t (*bsave)[2] = nullptr) {
  const int lane = threadIdx.x & 31, tig = lane & 3, mi = lane >> 3;
  using Fmt = CoefFmt<FOLD>;
  // ONEHOT: the lane's one entry m1 (-1: none) as the four B words dS, dS lo,
  // P, P lo (the lo words stay 0 without FOLD); with FOLD the correction of
  // that entry alone is loaded
  int m1 = -1;
  uint4 one = make_uint4(0u, 0u, 0u, 0u);
  if (ONEHOT) {
    const uint32_t me = mask & (0x55555555u >> (32 - 2 * 2 * NKS));  // the even bits read below
    if (me) {
      m1 = __ffs(me) - 1;
      if (FOLD) {  // words dS hi, dS lo, P hi, P lo
        const uint4 r4 = *reinterpret_cast<const uint4*>(csm + rec + m1 * STEP);
        const int qi = qw + m1 + (tig >> 1);
        const float c0 = __ldg(corr + (int64_t)(tig & 1) * T + qi);
        const float c1 = __ldg(corr + (int64_t)((tig & 1) + 2) * T + qi);
        const float2 lo = unpack_bf16(r4.y), pw = unpack_bf16(r4.z);
        one = make_uint4(r4.x, pack_bf16(fmaf(pw.x, c0, lo.x), fmaf(pw.y, c1, lo.y)), r4.z, r4.w);
      } else {  // words dS, P
        const uint2 r2 = *reinterpret_cast<const uint2*>(csm + rec + m1 * STEP);
        one = make_uint4(r2.x, 0u, r2.y, 0u);
      }
    }
  }
  // FOLD: the delta - psi values of every (k-step, half) this lane reads, loaded
  // before the products so their latency overlaps (heads tig & 1 and
  // (tig & 1) + 2 of query qw + m + (tig >> 1); 0 where the lane reads nothing)
  float cf[FOLD && !ONEHOT ? NKS : 1][2][2];
  if (FOLD && !ONEHOT) {
#pragma unroll
    for (int ks = 0; ks < NKS; ++ks)
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int m = 4 * ks + 2 * hb;
        const bool on = (mask >> m) & 1u;
        const int qi = on ? qw + m + (tig >> 1) : 0;
        cf[ks][hb][0] = on ? __ldg(corr + (int64_t)(tig & 1) * T + qi) : 0.0f;
        cf[ks][hb][1] = on ? __ldg(corr + (int64_t)((tig & 1) + 2) * T + qi) : 0.0f;
      }
  }
#pragma unroll
  for (int ks = 0; ks < NKS; ++ks) {
    uint32_t bk[2], bvv[2], bkl[2], bvl[2];
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int m = 4 * ks + 2 * hb;
      bk[hb] = bkl[hb] = bvv[hb] = bvl[hb] = 0u;
      if (PASS == 2) {
        bvv[hb] = bsave[ks][hb];
      } else if (ONEHOT) {
        bk[hb] = m1 == m ? one.x : 0u;
        bvv[hb] = m1 == m ? one.z : 0u;
        if (FOLD) {
          bkl[hb] = m1 == m ? one.y : 0u;
          bvl[hb] = m1 == m ? one.w : 0u;
        }
      } else if ((mask >> m) & 1u) {
        const uint32_t* half = csm + rec + m * STEP;
        if (FOLD) {  // words dS hi, dS lo, P hi, P lo
          const uint4 r4 = *reinterpret_cast<const uint4*>(half);
          const float c0 = cf[FOLD && !ONEHOT ? ks : 0][hb][0];
          const float c1 = cf[FOLD && !ONEHOT ? ks : 0][hb][1];
          const float2 lo = unpack_bf16(r4.y), pw = unpack_bf16(r4.z);
          bk[hb] = r4.x;
          bkl[hb] = pack_bf16(fmaf(pw.x, c0, lo.x), fmaf(pw.y, c1, lo.y));
          bvv[hb] = r4.z;
          bvl[hb] = r4.w;
        } else {  // words dS, P
          const uint2 r2 = *reinterpret_cast<const uint2*>(half);
          bk[hb] = r2.x;
          bvv[hb] = r2.y;
        }
      }
    }
    // A: q~^T and dO^T [16 dims x 16 (query, head)] by transposed ldmatrix;
    // k index kx = 4 (query offset) + hs (head slot; head 2 (hs & 1) + (hs >> 1)
    // by the order 0, 2, 1, 3) lives in slab row head * kq + query
    if (PASS == 1) {
      bsave[ks][0] = bvv[0];
      bsave[ks][1] = bvv[1];
    }
    const int kx = 8 * (mi >> 1) + (lane & 7);
    const int arow = (((kx & 1) << 1) | ((kx >> 1) & 1)) * kq + qoff + 4 * ks + (kx >> 2);
#pragma unroll
    for (int mt = 0; mt < kKvMT; ++mt) {
      uint32_t aq[4], ad[4];
      const uint32_t off = swz(arow, 2 * mt + (mi & 1));
      if (PASS != 2) {
        ldsm_x4_t(qst + off, aq[0], aq[1], aq[2], aq[3]);
        mma_bf16(dk[mt], aq, bk[0], bk[1]);
        if (FOLD) mma_bf16(dk[mt], aq, bkl[0], bkl[1]);
      }
      if (PASS != 1) {
        ldsm_x4_t(dst + off, ad[0], ad[1], ad[2], ad[3]);
        mma_bf16(dv[mt], ad, bvv[0], bvv[1]);
        if (FOLD) mma_bf16(dv[mt], ad, bvl[0], bvl[1]);
      }
    }
  }
}

// MULTI: G > 4, the key side loops over the G / 4 query-head groups of its KV head
template <bool INTERP, bool MULTI>
__global__ void __launch_bounds__(kKvThreads, KvLayout<MULTI>::MinBlocks)
    bwd_kv_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap md, const __grid_constant__ CUtensorMap mqr,
                     const __grid_constant__ CUtensorMap mdr, const __grid_constant__ CUtensorMap mcw,
                     const __grid_constant__ CUtensorMap mcr, const __grid_constant__ Plan P) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bars[kKvStages];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int kw = warp;  // key group: rows 8 kw .. 8 kw + 7 of the tile
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int T = a.T;
  const int j0 = blockIdx.x * kKvTK, j0w = j0 + 8 * kw;
  const int j = j0w + gid;  // key row of B column gid
  // the m = G / 4 groups of 4 query heads that read this KV head, one after
  // the other: group s has query heads 4 (g m + s) .. + 3 and record plane
  // b (Hq / 4) + g m + s
  const int msub = MULTI ? 1 << (a.lgG - 2) : 1;
  auto hplane_of = [&](int sg) { return b * a.Hq + (g * msub + sg) * 4; };
  auto rplane_of = [&](int sg) { return b * (a.Hq >> 2) + g * msub + sg; };

  float dk[kKvMT][4], dv[kKvMT][4];
#pragma unroll
  for (int x = 0; x < kKvMT; ++x) dk[x][0] = dk[x][1] = dk[x][2] = dk[x][3] = dv[x][0] = dv[x][1] =
      dv[x][2] = dv[x][3] = 0.0f;

  const int wmax = min(P.W, T - 1 - j0);
  using L = KvLayout<MULTI>;
  const int nwc = wmax >= 0 ? wmax / L::WC + 1 : 0;
  const int nwg = L::SPLIT ? 2 * nwc : nwc;  // window groups (SPLIT: q~ pass, then dO pass)
  const int nr = rungs_upto(P, T - j0);
  const int NG = nwg + nr;       // groups per query-head group
  const int NGt = MULTI ? NG * msub : NG;  // all groups: query-head group gt / NG, group gt % NG
  // window group -> its chunk; group -> first staged query: window chunk
  // s_lo = WC chunk, or rung grp - nwg
  auto chunk_of = [&](int grp) { return L::SPLIT ? grp >> 1 : grp; };
  auto qb_of = [&](int grp) { return grp < nwg ? j0 + L::WC * chunk_of(grp) : j0 + P.c[grp - nwg] - 1; };
  auto issue = [&](int gt, uint32_t st, uint32_t bar) {
    const int sg = MULTI ? gt / NG : 0, grp = MULTI ? gt - sg * NG : gt;
    const int hplane = hplane_of(sg), rp = rplane_of(sg);
    const int qb = qb_of(grp);
    if (grp < nwg) {
      const int ch = chunk_of(grp);
      if (!L::SPLIT) {
        mbar_expect_tx(bar, 2 * L::PlaneB + L::WRecB);
        tma_load_3d(st, &mq, 0, qb, hplane, bar);
        tma_load_3d(st + L::PlaneB, &md, 0, qb, hplane, bar);
        tma_load_4d(st + 2 * L::PlaneB, &mcw, 0, L::WC * ch, qb, rp, bar);
      } else if ((grp & 1) == 0) {  // q~ slab and records
        mbar_expect_tx(bar, L::PlaneB + L::WRecB);
        tma_load_3d(st, &mq, 0, qb, hplane, bar);
        tma_load_4d(st + L::PlaneB, &mcw, 0, L::WC * ch, qb, rp, bar);
      } else {  // dO slab
        mbar_expect_tx(bar, L::PlaneB);
        tma_load_3d(st, &md, 0, qb, hplane, bar);
      }
    } else {
      mbar_expect_tx(bar, 2 * kKvQR * 4 * 128 + kKvQR * 2 * CoefFmt<MULTI>::kRecBytes);
      tma_load_3d(st, &mqr, 0, qb, hplane, bar);
      tma_load_3d(st + L::RDoff, &mdr, 0, qb, hplane, bar);
      tma_load_4d(st + 2 * L::RDoff, &mcr, 0, P.W + 1 + 2 * (grp - nwg), qb, rp, bar);
    }
  };

  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kKvStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();  // the query side's q~, records and partials are complete from here on
  if (tid == 0)
    for (int s = 0; s < kKvStages && s < NGt; ++s) issue(s, sbase + s * L::StageB, smem_u32(&bars[s]));
  // the RoPE pairs of the dK epilogue (keys 2 tig (+1) of the warp's group,
  // pairs 16 h2 + gid (+8) for h2 = 0, 1), loaded now so their latency hides
  // under the loop
  const float2* rope = static_cast<const float2*>(a.rope);
  float2 kcs[2][2][2];
  if (rope)
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int jj = min(j0w + 2 * tig + e, T - 1);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          kcs[h2][e][hh] = __ldg(rope + (int64_t)jj * 32 + 16 * h2 + gid + 8 * hh);
      }
  uint32_t wsave[L::WKS][2];  // SPLIT: a window chunk's dV coefficients between its two groups
  int grpm = 0;  // with MULTI: gt mod NG, kept by a counter (no division per group)
  for (int gt = 0; gt < NGt; ++gt) {
    const int grp = MULTI ? grpm : gt;
    const int st = gt % kKvStages;
    const bool okw = mbar_wait_bounded(smem_u32(&bars[st]), (gt / kKvStages) & 1, a.wait_cycles);
    if (__syncthreads_or(!okw)) {
      if (tid == 0) {
        record_status(a.status, SFA_ERR_TIMEOUT);
        for (int g2 = gt; g2 < NGt && g2 < gt + kKvStages; ++g2)
          mbar_wait_bounded(smem_u32(&bars[g2 % kKvStages]), (g2 / kKvStages) & 1, a.wait_cycles);
      }
      return;
    }
    const uint32_t qst = sbase + st * L::StageB;
    const unsigned char* stg = sgen + st * L::StageB;
    // MULTI: query-head group gt / NG; its delta - psi rows for the correction
    const float* corr = MULTI ? a.dcorr + (int64_t)hplane_of(gt / NG) * T : nullptr;
    constexpr int RW = CoefFmt<MULTI>::kRecWords, HW = CoefFmt<MULTI>::kHalfWords;
    const int t1 = tig >> 1;
    if (grp < nwg) {
      // window chunk: query qw + ql reaches key j through slot s = ql + rel of
      // the chunk (s in 0 .. s_hi - s_lo), record (qoff + ql) * WC + s
      const int s_lo = L::WC * chunk_of(grp), qoff = min(8 * kw, L::Q - 4 * L::WKS);
      const int qw = qb_of(grp) + qoff;
      if (L::SPLIT && (grp & 1)) {  // the chunk's dO slab: dV from the kept coefficients
        kv_group<L::WKS, (L::WC + 1) * RW, MULTI, false, 2>(qst, qst, nullptr, 0, 0u, qw, L::Q, qoff,
                                                           T, corr, dk, dv, wsave);
      } else {
        const int rel = qw - j - s_lo;
        const uint32_t mask =
            j < T ? ql_mask(max(-rel, 0), min(min(P.W, s_lo + L::WC - 1) - s_lo - rel, T - 1 - qw), t1) : 0u;
        const int rec = (qoff * L::WC + rel) * RW + HW * (tig & 1) + t1 * (L::WC + 1) * RW;
        const uint32_t* csm =
            reinterpret_cast<const uint32_t*>(stg + (L::SPLIT ? 1 : 2) * L::PlaneB);
        if (L::SPLIT)  // the chunk's q~ slab and records: dK, and the dV coefficients kept
          kv_group<L::WKS, (L::WC + 1) * RW, MULTI, false, 1>(qst, qst, csm, rec, mask, qw, L::Q, qoff,
                                                             T, corr, dk, dv, wsave);
        else
          kv_group<L::WKS, (L::WC + 1) * RW, MULTI>(qst, qst + L::PlaneB, csm, rec, mask, qw, L::Q,
                                                    qoff, T, corr, dk, dv);
      }
    } else {
      // rung: query qw + ql reaches key j as role 1 (key i - c + 1) when
      // ql + rel = 0 and as role 0 (key i - c) when ql + rel = 1, and only if
      // it reads the rung at all (qw + ql >= c); record (qoff + ql) * 2 + role.
      // An integer rung (w = 0) has no role 1: a warp's 8 keys then read 8
      // queries, 8 kw + 1 .. 8 kw + 8 of the slab, two k-steps instead of three
      constexpr int RKS = INTERP ? 3 : 2;
      const int c = P.c[grp - nwg];
      const int qoff = INTERP ? min(8 * kw, kKvQR - 12) : 8 * kw + 1, qw = qb_of(grp) + qoff;
      const int rel = qw - j - c + 1;
      const uint32_t mask =
          j < T ? ql_mask(max(INTERP ? -rel : 1 - rel, c - qw), min(1 - rel, T - 1 - qw), t1) : 0u;
      const int rec = (2 * qoff + 1 - rel) * RW + HW * (tig & 1) + t1 * RW;
      const uint32_t* csm = reinterpret_cast<const uint32_t*>(stg + 2 * L::RDoff);
      kv_group<RKS, RW, MULTI, true>(qst, qst + L::RDoff, csm, rec, mask, qw, kKvQR, qoff, T,
                                     corr, dk, dv);
    }
    __syncthreads();
    if (tid == 0 && gt + kKvStages < NGt) issue(gt + kKvStages, qst, smem_u32(&bars[st]));
    if (MULTI && ++grpm == NG) grpm = 0;
  }

  // dK = R(-phi) dk' at key positions; transpose through shared memory for
  // row-contiguous stores.  Lane holds dims 16 mt + gid (+8) for mt = 0..3,
  // keys 2 tig (+1) of its key group.
  if (rope) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // m-tiles h2 and h2 + 2 hold dims d and d + 32
          const float2 cs = kcs[h2][e][hh];
          const float lo = dk[h2][2 * hh + e], hi = dk[h2 + 2][2 * hh + e];
          dk[h2][2 * hh + e] = lo * cs.x + hi * cs.y;
          dk[h2 + 2][2 * hh + e] = hi * cs.x - lo * cs.y;
        }
      }
  }
  bf16* tk = reinterpret_cast<bf16*>(sgen);  // [32 keys][72] for dK, then dV
  bf16* tv = tk + kKvTK * 72;
#pragma unroll
  for (int x = 0; x < kKvMT; ++x)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int d = 16 * x + gid + 8 * hh, n = 8 * kw + 2 * tig + e;
        tk[n * 72 + d] = __float2bfloat16_rn(dk[x][2 * hh + e]);
        tv[n * 72 + d] = __float2bfloat16_rn(dv[x][2 * hh + e]);
      }
  __syncthreads();
  for (int it = tid; it < kKvTK * 8; it += kKvThreads) {
    const int n = it >> 3, ch = it & 7;  // key row n of the tile, 8 dims per thread
    const int jr = j0 + n;
    if (jr < T) {
      const int64_t row = ((int64_t)bg * T + jr) * kD + 8 * ch;
      *reinterpret_cast<uint4*>(static_cast<bf16*>(a.dk) + row) = *reinterpret_cast<const uint4*>(tk + n * 72 + 8 * ch);
      *reinterpret_cast<uint4*>(static_cast<bf16*>(a.dv) + row) = *reinterpret_cast<const uint4*>(tv + n * 72 + 8 * ch);
    }
  }
  if (INTERP && a.dalpha_out && blockIdx.x == 0 && blockIdx.y == 0) {
    // dL/dalpha = the query side's per-CTA partials summed in a fixed order
    // (strided per thread, then the warp tree, then the warps in order), and
    // dL/dtheta = dL/dalpha (alpha - 0.5)(1.5 - alpha)
    __shared__ double red[kKvThreads / 32];
    const int nblk = ((T + kTcTQ - 1) / kTcTQ) * a.B * (a.Hq >> 2);
    double sum = 0.0;
    for (int x = tid; x < nblk; x += kKvThreads) sum += a.dalpha_part[x];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_down_sync(0xffffffffu, sum, off);
    if (lane == 0) red[warp] = sum;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int x = 0; x < kKvThreads / 32; ++x) t += red[x];
      a.dalpha_out[0] = t;
      a.dalpha_out[1] = t * (a.alpha - 0.5) * (1.5 - a.alpha);
    }
  }
}

size_t backward_tc_workspace_bytes(const sfa_desc* d, const Plan& p, size_t* off_kr, size_t* off_qt,
                                   size_t* off_coef, size_t* off_corr) {
  const size_t nparts = (size_t)((d->T + kTcTQ - 1) / kTcTQ) * d->B * (d->Hq / 4);
  size_t o = align256(nparts * sizeof(double));  // per-CTA dL/dalpha partials
  *off_corr = 0;
  if (d->Hq / d->Hkv > 4) {  // delta - psi per query row, for the key side's correction
    *off_corr = o;
    o += align256((size_t)d->B * d->Hq * d->T * sizeof(float));
  }
  *off_kr = o;
  o += kr_bytes(d);
  *off_qt = o;
  o += align256((size_t)d->B * d->Hq * d->T * kD * 2);
  *off_coef = o;
  const size_t NS = (size_t)p.W + 1 + 2 * p.n;  // records per query: window slots, 2 per rung
  const size_t rec_bytes = d->Hq / d->Hkv > 4 ? CoefFmt<true>::kRecBytes : CoefFmt<false>::kRecBytes;
  o += align256((size_t)d->B * (d->Hq / 4) * d->T * NS * rec_bytes);  // one plane per group of 4 heads
  return o;
}

int launch_backward_tc(const AttnArgs& a, const Plan& p, const void* kr, void* qt, void* coef,
                       void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  const int NS = p.W + 1 + 2 * p.n;
  const int64_t kvplanes = (int64_t)a.B * a.Hkv, qplanes = (int64_t)a.B * a.Hq;
  // query side: Q / dO / O tile loads (20-row boxes), q~ and dQ tile stores
  // (16-row boxes); key side: q~ and dO slabs (34 rows; 42 for a window chunk
  // at G > 4) and the record boxes
  const bool multi = a.lgG > 2;
  const int rec_words = multi ? CoefFmt<true>::kRecWords : CoefFmt<false>::kRecWords;
  const int wq = multi ? KvLayout<true>::Q : KvLayout<false>::Q;
  const int wc = multi ? KvLayout<true>::WC : KvLayout<false>::WC;
  const size_t kv_smem = multi ? KvLayout<true>::Smem : KvLayout<false>::Smem;
  CUtensorMap mk, mv, mq, md, mqr, mdr, mcw, mcr, tq, tdo, to, sqt, sdq;
  if (make_rows_map(&mk, kr, kvplanes, a.T, kTcBoxRows, 1) != SFA_OK ||
      make_rows_map(&mv, a.v, kvplanes, a.T, kTcBoxRows, 1) != SFA_OK ||
      make_rows_map(&tq, a.q, qplanes, a.T, kTcQRows, 4) != SFA_OK ||
      make_rows_map(&tdo, a.dO, qplanes, a.T, kTcQRows, 4) != SFA_OK ||
      make_rows_map(&to, a.o, qplanes, a.T, kTcQRows, 4) != SFA_OK ||
      make_rows_map(&sqt, qt, qplanes, a.T, kTcORows, 4) != SFA_OK ||
      make_rows_map(&sdq, a.dq, qplanes, a.T, kTcORows, 4) != SFA_OK ||
      make_rows_map(&mq, qt, qplanes, a.T, wq, 4) != SFA_OK ||
      make_rows_map(&md, a.dO, qplanes, a.T, wq, 4) != SFA_OK ||
      make_rows_map(&mqr, qt, qplanes, a.T, kKvQR, 4) != SFA_OK ||
      make_rows_map(&mdr, a.dO, qplanes, a.T, kKvQR, 4) != SFA_OK ||
      make_coef_map(&mcw, coef, qplanes / 4, a.T, NS, rec_words, wc, wq) != SFA_OK ||
      make_coef_map(&mcr, coef, qplanes / 4, a.T, NS, rec_words, 2, kKvQR) != SFA_OK)
    return SFA_ERR_CUDA;
  const bool psi = a.dcorr != nullptr;
  auto kq = p.interp ? (psi ? bwd_q_tc_kernel<true, true> : bwd_q_tc_kernel<true, false>)
                     : (psi ? bwd_q_tc_kernel<false, true> : bwd_q_tc_kernel<false, false>);
  auto kkv = p.interp ? (multi ? bwd_kv_tc_kernel<true, true> : bwd_kv_tc_kernel<true, false>)
                      : (multi ? bwd_kv_tc_kernel<false, true> : bwd_kv_tc_kernel<false, false>);
  if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBwdQTcSmem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kv_smem) !=
          cudaSuccess)
    return SFA_ERR_CUDA;
  dim3 gq((unsigned)((a.T + kTcTQ - 1) / kTcTQ), (unsigned)(a.B * (a.Hq / 4)));
  {
    LaunchTimer tm(SFA_KERNEL_BWD_Q, stream);
    if (launch_pdl(kq, gq, dim3(kTcThreads), kBwdQTcSmem, s, a, mk, mv, tq, tdo, to, sqt, sdq,
                   static_cast<uint32_t*>(coef), NS, p) != cudaSuccess)
      return SFA_ERR_CUDA;
  }
  dim3 gkv((unsigned)((a.T + kKvTK - 1) / kKvTK), (unsigned)(a.B * a.Hkv));
  {
    LaunchTimer tm(SFA_KERNEL_BWD_KV, stream);
    if (launch_pdl(kkv, gkv, dim3(kKvThreads), kv_smem, s, a, mq, md, mqr, mdr, mcw, mcr, p) !=
        cudaSuccess)
      return SFA_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

}  // namespace sfa
