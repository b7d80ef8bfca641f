// Incremental decode on the integer path: one query per sequence against a
// key/value cache ("Depth-Staggered Fibonacci Spacing for Sparse Attention",
// method section: integer offsets as an exact gather; its efficiency case is
// inference).
//
// One warp per query head, four heads per CTA (heads of a KV group share the
// CTA, so their key rows meet in L1).  The query row is rotated at pos[b] and
// scaled by 1/8 in registers.  Keys are taken 32 at a time, one per lane:
// the lane loads its raw key row, rotates it at the key's own position and
// forms the logit, and copies its value row into the warp's slice of shared
// memory (all rows of a chunk in flight at once); the warp then runs one
// online-softmax step over the chunk and accumulates O from the staged rows
// (two dims per lane, the probabilities broadcast by shuffles).  fp32
// throughout.
#include <math.h>

#include "sfa_device.cuh"
#include "sfa_launch.cuh"
#include "sfa_tma.cuh"

namespace sfa {

constexpr int kDecHeadsPerCta = 1;

template <typename TIO>
__global__ void __launch_bounds__(32 * kDecHeadsPerCta)
    decode_int_kernel(const AttnArgs a, const __grid_constant__ Plan P) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's outputs (this layer's q, the cache) are complete
  const int lane = threadIdx.x & 31;
  const int64_t gh = (int64_t)blockIdx.x * kDecHeadsPerCta + (threadIdx.x >> 5);  // b * Hq + h
  if (gh >= (int64_t)a.B * a.Hq) return;
  const int b = (int)(gh / a.Hq), h = (int)(gh - (int64_t)b * a.Hq);
  const int kvh = h >> a.lgG;
  const int T = a.T;
  const int t = a.pos[b];
  if (t < 0 || t >= T) {
    if (lane == 0) record_status(a.status, SFA_ERR_DEVICE_BOUNDS);
    return;
  }
  const float2* rope = static_cast<const float2*>(a.rope);
  const TIO* qrow = static_cast<const TIO*>(a.q) + gh * kD;
  const TIO* kbase = static_cast<const TIO*>(a.k) + ((int64_t)b * a.Hkv + kvh) * T * kD;
  const TIO* vbase = static_cast<const TIO*>(a.v) + ((int64_t)b * a.Hkv + kvh) * T * kD;

  // q' = R(t) q / 8, all 64 dims in every lane
  float qv[kD];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float lo[8], hi[8];
    load8(qrow + 8 * c, lo);
    load8(qrow + 32 + 8 * c, hi);
    if (rope) {
      float cs[8], sn[8];
      load_rope8(rope, t, 8 * c, cs, sn);
      rotate8(lo, hi, cs, sn);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      qv[8 * c + e] = lo[e] * 0.125f;
      qv[32 + 8 * c + e] = hi[e] * 0.125f;
    }
  }

  __shared__ float vs[kDecHeadsPerCta][32][kD + 2];  // + 2: lanes' rows on distinct banks
  float(*vrows)[kD + 2] = vs[threadIdx.x >> 5];
  const int Wt = min(P.W, t);
  int nr = 0;
  while (nr < P.n && P.c[nr] <= t) ++nr;
  const int nk = Wt + 1 + nr;
  float m = -INFINITY, l = 0.0f, o0 = 0.0f, o1 = 0.0f;
  for (int j0 = 0; j0 < nk; j0 += 32) {
    const int j = j0 + lane;
    float s = -INFINITY;
    int kp = 0;
    if (j < nk) {
      kp = t - (j <= Wt ? j : P.c[j - Wt - 1]);
      const TIO* krow = kbase + (int64_t)kp * kD;
      float acc = 0.0f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float lo[8], hi[8];
        load8(krow + 8 * c, lo);
        load8(krow + 32 + 8 * c, hi);
        if (rope) {
          float cs[8], sn[8];
          load_rope8(rope, kp, 8 * c, cs, sn);
          rotate8(lo, hi, cs, sn);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(qv[8 * c + e], lo[e], fmaf(qv[32 + 8 * c + e], hi[e], acc));
      }
      s = acc;
      const TIO* vrow = vbase + (int64_t)kp * kD;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float x[8];
        load8(vrow + 8 * c, x);
#pragma unroll
        for (int e = 0; e < 8; e += 2) *reinterpret_cast<float2*>(&vrows[lane][8 * c + e]) = make_float2(x[e], x[e + 1]);
      }
    }
    __syncwarp();
    float mx = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float mn = fmaxf(m, mx);  // finite: every chunk holds at least one key
    const float corr = expf(m - mn);  // 0 on the first chunk
    const float p = expf(s - mn);     // 0 for lanes past the key count
    float ps = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * corr + ps;
    o0 *= corr;
    o1 *= corr;
    m = mn;
    const int nc = min(32, nk - j0);
    for (int jj = 0; jj < nc; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const float2 v2 = *reinterpret_cast<const float2*>(&vrows[jj][2 * lane]);
      o0 = fmaf(pj, v2.x, o0);
      o1 = fmaf(pj, v2.y, o1);
    }
    __syncwarp();  // the slice is refilled by the next chunk
  }
  const float inv = 1.0f / l;
  store2(static_cast<TIO*>(a.out_o) + gh * kD + 2 * lane, o0 * inv, o1 * inv);
  if (a.out_lse && lane == 0) a.out_lse[gh] = m + logf(l);
}

int launch_decode_int(const AttnArgs& a, const Plan& p, int dtype, void* stream) {
  const int64_t heads = (int64_t)a.B * a.Hq;
  const unsigned grid = (unsigned)((heads + kDecHeadsPerCta - 1) / kDecHeadsPerCta);
  if (grid == 0) return SFA_OK;
  LaunchTimer tm(SFA_KERNEL_DECODE, stream);
  if (dtype == SFA_BF16)
    return launch_pdl(decode_int_kernel<bf16>, grid, dim3(32 * kDecHeadsPerCta), 0,
                      (cudaStream_t)stream, a, p) == cudaSuccess
               ? SFA_OK
               : SFA_ERR_CUDA;
  else
    return launch_pdl(decode_int_kernel<float>, grid, dim3(32 * kDecHeadsPerCta), 0,
                      (cudaStream_t)stream, a, p) == cudaSuccess
               ? SFA_OK
               : SFA_ERR_CUDA;
}

}  // namespace sfa
