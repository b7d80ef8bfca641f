// Tensor-core forward (bf16 I/O, G = 4, 8 or 16 query heads per KV head, taken
// in groups of 4).
//
// Same result as the SIMT forward ("Depth-Staggered Fibonacci Spacing for
// Sparse Attention", method section: window 0..W plus rungs read by two-row
// interpolation after RoPE), organised for mma.sync m16n8k16 (bf16 in, fp32
// accumulate):
//
//  * A warp owns 4 consecutive query positions x the 4 heads of one KV
//    group = 16 rows (row r = 4 h + p).  Its q~ = q'/8 (rotated, scaled)
//    stays in registers as bf16 A fragments; logits take log2(e) in fp32.
//  * Keys are the raw rotated rows K' (bf16, written by the prep kernel) and
//    raw V rows, staged per CTA as contiguous shifted slabs by TMA (rows
//    outside the sequence are zero-filled by the copy engine).
//  * Window: the 16 keys i0w + 3 - s_lo - 15 .. i0w + 3 - s_lo of a chunk of
//    12 distances form two n-tiles; the band is masked per row.
//  * Rung: the 8 B-columns are (floor row, floor-plus-one row) of each of the
//    4 positions, so the lane holding position p (tig = p) has both raw
//    logits and applies the interpolation on the logit:
//    s = (1 - w) q'.K'[i - c] + w q'.K'[i - c + 1].  The probability is split
//    the same way over the two V rows in the P.V product, so no interpolated
//    row is ever materialised.  Two rungs share one k16 step of P.V.
//  * Online softmax in base 2 across window chunks and rung pairs.
#include <math.h>

#include "sfa_tc.cuh"

namespace sfa {

// K' = RoPE(K) as bf16 rows (the operand of every key-side product).  A
// thread owns one position and one 8-pair chunk of the rotation: it loads
// that chunk of the cos/sin table once and rotates the position's rows in
// kPrepPlanes consecutive (batch, KV head) planes per grid row (loads issued
// before the arithmetic).  One plane per grid row spreads a config-2 layer
// (64 planes of 1024 rows) over 1024 CTAs, which hides the loads' latency
// best.

constexpr int kPrepPlanes = 1;

__global__ void __launch_bounds__(256) rope_prep_kernel(const bf16* __restrict__ k,
                                                        const float2* __restrict__ rope,
                                                        bf16* __restrict__ kr, int64_t planes, int T) {
  pdl_launch_dependents();
  pdl_wait();  // K may be the previous kernel's output
  const int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (it >= (int64_t)T * 4) return;
  const int pos = (int)(it >> 2), pc = (int)(it & 3);
  float cs[8], sn[8];
  load_rope8(rope, pos, 8 * pc, cs, sn);
  for (int64_t p0 = (int64_t)blockIdx.y * kPrepPlanes; p0 < planes;
       p0 += (int64_t)gridDim.y * kPrepPlanes) {
    float lo[kPrepPlanes][8], hi[kPrepPlanes][8];
#pragma unroll
    for (int x = 0; x < kPrepPlanes; ++x) {  // all loads first
      const int64_t row = (p0 + x < planes ? p0 + x : p0) * T + pos;
      load8(k + row * kD + 8 * pc, lo[x]);
      load8(k + row * kD + 32 + 8 * pc, hi[x]);
    }
#pragma unroll
    for (int x = 0; x < kPrepPlanes; ++x) {
      if (p0 + x >= planes) break;
      const int64_t row = (p0 + x) * T + pos;
      rotate8(lo[x], hi[x], cs, sn);
      store8(kr + row * kD + 8 * pc, lo[x]);
      store8(kr + row * kD + 32 + 8 * pc, hi[x]);
    }
  }
}

int launch_rope_prep(const void* k, const void* rope, void* kr, int64_t rows, int T, void* stream) {
  const int64_t planes = rows / T;
  dim3 grid((unsigned)(((int64_t)T * 4 + 255) / 256), (unsigned)((planes + kPrepPlanes - 1) / kPrepPlanes < 65535 ? (planes + kPrepPlanes - 1) / kPrepPlanes : 65535));
  return launch_pdl(rope_prep_kernel, grid, dim3(256), 0, (cudaStream_t)stream,
                    static_cast<const bf16*>(k), static_cast<const float2*>(rope),
                    static_cast<bf16*>(kr), planes, T) == cudaSuccess
             ? SFA_OK
             : SFA_ERR_CUDA;
}

template <bool INTERP>
__global__ void __launch_bounds__(kTcThreads, 5)
    fwd_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mq,
                  const __grid_constant__ CUtensorMap mo, const __grid_constant__ Plan P) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bars[kTcStages + 1];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  // blockIdx.y = (batch, group g of 4 query heads); with G = 4m query heads per
  // KV head the group reads KV head g / m
  const int ng4 = a.Hq >> 2, b = blockIdx.y / ng4, g = blockIdx.y - b * ng4;
  const int bg = b * a.Hkv + (g >> (a.lgG - 2));
  const int T = a.T;
  const int i0 = blockIdx.x * kTcTQ, i0w = i0 + 4 * warp;
  const int p = gid & 3, i = i0w + p;  // position of rows gid and gid + 8
  const int imax = min(T - 1, i0 + kTcTQ - 1);
  const int hA = g * 4 + (gid >> 2), hB = hA + 2;  // heads of rows gid, gid + 8
  const float2* rope = static_cast<const float2*>(a.rope);

  const int wmax = min(P.W, imax);
  const int nwc = wmax >= 0 ? wmax / kTcWC + 1 : 0;
  const int nr = rungs_upto(P, imax);
  const int NG = nwc + (nr + 1) / 2;
  const uint32_t qtile = sbase, stages = sbase + kTcQTileB;
  const int qplane = b * a.Hq + g * 4;
  const int skip_grp = (blockIdx.x | blockIdx.y) == 0 ? a.debug_skip : -1;  // test injection
  const CUtensorMap* qmaps[1] = {&mq};
  tc_start(&mk, &mv, qmaps, 1, qtile, qplane, P, bg, i0, nwc, nr, NG, stages, bars, skip_grp);
  float4 rp[4];
  if (rope) load_frag_rope(rope, min(i, T - 1), rp);  // while the Q tile is in flight
  if (!tc_wait_qtiles(bars, a)) return;
  uint32_t qa[4][4];
  // q~ = q'/8 rounded exactly as the query-side backward rounds it, log2(e)
  // applied to the fp32 logits: the backward's P = exp(S - LSE) recomputes
  // this kernel's logits bit for bit and stays normalised
  tile_frags(qtile, warp, rope ? rp : nullptr, 0.125f, true, qa);
  float o[8][4];
#pragma unroll
  for (int nd = 0; nd < 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.0f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};

  // online-softmax step for this lane's logits of rows gid (r = 0) and gid + 8
  // (r = 1); s holds N values per row (invalid = -inf), returns P in place.
  // The running maximum m (base 2) is refreshed only when some logit of the
  // warp exceeds it by more than kMargin: between refreshes p = 2^(s - m) stays
  // below 2^kMargin, and O = sum p v / sum p and LSE = m + log2 l are exact for
  // any m.  m stays uniform over a row's quad (it changes only through the quad
  // reduction).
  constexpr float kMargin = 8.0f;
  auto softmax_step = [&](float (*s)[4], auto Nc) {
    constexpr int N = decltype(Nc)::value;
    float mx[2];
    bool need = false;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = s[r][0];
#pragma unroll
      for (int e = 1; e < N; ++e) mx[r] = fmaxf(mx[r], s[r][e]);
      need |= mx[r] > m[r] + kMargin;  // m = -inf: any valid logit
    }
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        if (mx[r] > m[r]) {
          const float corr = ex2(m[r] - mx[r]);  // 0 while the row had no key
          m[r] = mx[r];
          l[r] *= corr;
#pragma unroll
          for (int nd = 0; nd < 8; ++nd) {
            o[nd][2 * r] *= corr;
            o[nd][2 * r + 1] *= corr;
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float mm = m[r] == -INFINITY ? 0.0f : m[r];
#pragma unroll
      for (int e = 0; e < N; ++e) {
        const float pe = ex2(s[r][e] - mm);  // ex2(-inf) = 0
        s[r][e] = pe;
        l[r] += pe;
      }
    }
  };

  const int colrow = 4 * warp + ((lane & 7) >> 1) + (lane & 1);

  const bool ok = tc_run(&mk, &mv, P, bg, i0, nwc, nr, NG, stages, bars, a, skip_grp,
                              [&](int grp, uint32_t kst, uint32_t vst) {
    uint32_t pa[4];
    if (grp < nwc) {
      // window chunk: key column n = 0..15 <-> key i0w + 3 - s_lo - 15 + n = row 4w + n
      const int s_lo = kTcWC * grp, s_hi = min(s_lo + kTcWC - 1, P.W);
      float acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
      qk_tile(qa, kst, 4 * warp + (lane & 7), acc[0]);
      qk_tile(qa, kst, 4 * warp + 8 + (lane & 7), acc[1]);
      // distance of column n for this lane's rows: p + 12 + s_lo - n
      float s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int dist = p + 12 + s_lo - (8 * nt + 2 * tig + (e & 1));
          const bool v = dist >= s_lo && dist <= s_hi && dist <= i;
          s[e >> 1][2 * nt + (e & 1)] = v ? acc[nt][e] * kLog2e : -INFINITY;
        }
      softmax_step(s, std::integral_constant<int, 4>());
      pa[0] = pack_bf16(s[0][0], s[0][1]);
      pa[1] = pack_bf16(s[1][0], s[1][1]);
      pa[2] = pack_bf16(s[0][2], s[0][3]);
      pa[3] = pack_bf16(s[1][2], s[1][3]);
      pv_tile(pa, vst, 4 * warp + (lane & 7), 4 * warp + 8 + (lane & 7), o);
    } else if (!INTERP) {
      // integer rung pair: one tile, column (rung x, position p') = raw row
      // 4w + p' of box x; the lane of this row's position p holds rung
      // x = tig >> 1 at column e = p & 1 when tig & 1 == p >> 1
      const int r0 = 2 * (grp - nwc), rg = r0 + (tig >> 1), e = p & 1;
      float acc[4] = {0, 0, 0, 0};
      qk_tile(qa, kst, int_pair_row(warp), acc);
      const bool v = (tig & 1) == (p >> 1) && rg < nr && i >= P.c[min(rg, P.n - 1)];
      float s[2][4];
      s[0][0] = v ? (e ? acc[1] : acc[0]) * kLog2e : -INFINITY;
      s[1][0] = v ? (e ? acc[3] : acc[2]) * kLog2e : -INFINITY;
      softmax_step(s, std::integral_constant<int, 1>());
      const uint32_t pk8[2] = {pack_bf16(e ? 0.0f : s[0][0], e ? s[0][0] : 0.0f),
                               pack_bf16(e ? 0.0f : s[1][0], e ? s[1][0] : 0.0f)};
      pv_tile_k8(pk8, vst, int_pair_row(warp), o);
    } else {
      // rung pair: box x, B column n = 2 p' + e' is row 4w + p' + e'
      const int r0 = 2 * (grp - nwc);
      float s[2][4];
      float wgt[2];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int rg = r0 + x;
        float acc[4] = {0, 0, 0, 0};
        qk_tile(qa, kst, x * kTcBoxRows + colrow, acc);
        const bool v = rg < nr && p == tig && i >= P.c[rg];
        const float w = (INTERP && rg < nr) ? P.w[rg] : 0.0f;
        wgt[x] = w;
        s[0][x] = v ? fmaf(w, acc[1], (1.0f - w) * acc[0]) * kLog2e : -INFINITY;
        s[1][x] = v ? fmaf(w, acc[3], (1.0f - w) * acc[2]) * kLog2e : -INFINITY;
      }
      softmax_step(s, std::integral_constant<int, 2>());
      pa[0] = pack_bf16(s[0][0] * (1.0f - wgt[0]), s[0][0] * wgt[0]);
      pa[1] = pack_bf16(s[1][0] * (1.0f - wgt[0]), s[1][0] * wgt[0]);
      pa[2] = pack_bf16(s[0][1] * (1.0f - wgt[1]), s[0][1] * wgt[1]);
      pa[3] = pack_bf16(s[1][1] * (1.0f - wgt[1]), s[1][1] * wgt[1]);
      pv_tile(pa, vst, colrow, kTcBoxRows + colrow, o);
    }
  });
  if (!ok) return;

#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  // O = acc / l through an output tile (the Q tile's space) and one TMA store
  uint32_t pk[8][2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float inv = 1.0f / l[r];
#pragma unroll
    for (int nd = 0; nd < 8; ++nd) pk[nd][r] = pack_bf16(o[nd][2 * r] * inv, o[nd][2 * r + 1] * inv);
    if (tig == 0 && i < T)
      a.out_lse[(int64_t)(b * a.Hq + (r ? hB : hA)) * T + i] = (m[r] + log2f(l[r])) * kLn2;
  }
  store_otile(qtile, warp, pk);
  fence_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    tc_store_tile(&mo, qtile, i0, qplane);
    bulk_wait_read();
  }
}

int launch_forward_tc(const AttnArgs& a, const Plan& p, const void* kr, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  CUtensorMap mk, mv, mq, mo;
  const int64_t planes = (int64_t)a.B * a.Hkv, qplanes = (int64_t)a.B * a.Hq;
  if (make_rows_map(&mk, kr, planes, a.T, kTcBoxRows, 1) != SFA_OK ||
      make_rows_map(&mv, a.v, planes, a.T, kTcBoxRows, 1) != SFA_OK ||
      make_rows_map(&mq, a.q, qplanes, a.T, kTcQRows, 4) != SFA_OK ||
      make_rows_map(&mo, a.out_o, qplanes, a.T, kTcORows, 4) != SFA_OK)
    return SFA_ERR_CUDA;
  auto kern = p.interp ? fwd_tc_kernel<true> : fwd_tc_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFwdTcSmem) !=
      cudaSuccess)
    return SFA_ERR_CUDA;
  dim3 grid((unsigned)((a.T + kTcTQ - 1) / kTcTQ), (unsigned)(a.B * (a.Hq / 4)));
  LaunchTimer tm(SFA_KERNEL_FWD, stream);
  return launch_pdl(kern, grid, dim3(kTcThreads), kFwdTcSmem, s, a, mk, mv, mq, mo, p) == cudaSuccess
             ? SFA_OK
             : SFA_ERR_CUDA;
}

}  // namespace sfa
