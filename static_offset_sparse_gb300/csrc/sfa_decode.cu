// Incremental decode on the integer path: one query per sequence against a
// key/value cache ("Depth-Staggered Fibonacci Spacing for Sparse Attention",
// method section: integer offsets as an exact gather; its efficiency case is
// inference).
//
// One warp per query head, one head per CTA (a decode step has few heads, so
// they spread over as many SMs as possible).  The query row is rotated at
// pos[b] and scaled by 1/8 in registers.  Keys are taken 32 at a time, one
// per lane: the lane loads its raw key row, rotates it at the key's own
// position and forms the logit, and copies its value row into the warp's
// slice of shared memory (all rows of a chunk in flight at once); the warp
// then runs one online-softmax step over the chunk and accumulates O from the
// staged rows (two dims per lane, the probabilities broadcast by shuffles).
// fp32 throughout.  Steps of at most kDecStagedMaxHeads heads run a variant
// that starts the key-side copies before the query rotation (below).
#include <math.h>

#include "sfa_device.cuh"
#include "sfa_launch.cuh"
#include "sfa_tma.cuh"

namespace sfa {

constexpr int kDecHeadsPerCta = 1;
constexpr int64_t kDecStagedMaxHeads = 1024;

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

// 16-byte asynchronous global -> shared copy through L2 (cp.async.cg).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Eight consecutive elements of a shared-memory row -> fp32 (p 16-byte aligned).
__device__ __forceinline__ void lds8(const float* p, float* x) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void lds8(const bf16* p, float* x) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}

// Latency-lean variant for steps of few heads (one wave): the key, value and
// RoPE rows of a chunk are copied into shared memory with cp.async as soon as
// the position is known, so they travel while the query row is rotated.
template <typename TIO>
__global__ void __launch_bounds__(32 * kDecHeadsPerCta)
    decode_staged_kernel(const AttnArgs a, const __grid_constant__ Plan P) {
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

  // the warp's staging: 32 keys' raw rows (padded by 16 bytes so the lanes'
  // rows start on different banks) and their RoPE (cos, sin) rows
  constexpr int kRowE = kD + 16 / (int)sizeof(TIO);
  __shared__ __align__(16) TIO ks[kDecHeadsPerCta][32][kRowE];
  __shared__ __align__(16) TIO vs[kDecHeadsPerCta][32][kRowE];
  __shared__ __align__(16) float2 rs[kDecHeadsPerCta][32][34];
  TIO(*krows)[kRowE] = ks[threadIdx.x >> 5];
  TIO(*vrows)[kRowE] = vs[threadIdx.x >> 5];
  float2(*rrows)[34] = rs[threadIdx.x >> 5];
  const int Wt = min(P.W, t);
  int nr = 0;
  while (nr < P.n && P.c[nr] <= t) ++nr;
  const int nk = Wt + 1 + nr;
  auto stage = [&](int j0) {  // copies of key j0 + lane (one commit group per chunk)
    const int j = j0 + lane;
    if (j < nk) {
      const int kp = t - (j <= Wt ? j : P.c[j - Wt - 1]);
      const char* kg = reinterpret_cast<const char*>(kbase + (int64_t)kp * kD);
      const char* vg = reinterpret_cast<const char*>(vbase + (int64_t)kp * kD);
      char* kd = reinterpret_cast<char*>(krows[lane]);
      char* vd = reinterpret_cast<char*>(vrows[lane]);
#pragma unroll
      for (int c = 0; c < kD * (int)sizeof(TIO) / 16; ++c) {
        cp_async16(kd + 16 * c, kg + 16 * c);
        cp_async16(vd + 16 * c, vg + 16 * c);
      }
      if (rope)
#pragma unroll
        for (int c = 0; c < 16; ++c) cp_async16(&rrows[lane][2 * c], rope + (int64_t)kp * 32 + 2 * c);
    }
    cp_async_commit();
  };
  stage(0);  // the first chunk's rows travel while the query row is rotated

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

  float m = -INFINITY, l = 0.0f, o0 = 0.0f, o1 = 0.0f;
  for (int j0 = 0; j0 < nk; j0 += 32) {
    if (j0 > 0) stage(j0);
    cp_async_wait_all();
    __syncwarp();
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j < nk) {
      float acc = 0.0f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float lo[8], hi[8];
        lds8(&krows[lane][8 * c], lo);
        lds8(&krows[lane][32 + 8 * c], hi);
        if (rope) {
          float cs[8], sn[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 r2 = rrows[lane][8 * c + e];
            cs[e] = r2.x;
            sn[e] = r2.y;
          }
          rotate8(lo, hi, cs, sn);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(qv[8 * c + e], lo[e], fmaf(qv[32 + 8 * c + e], hi[e], acc));
      }
      s = acc;
    }
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
      float v2[2];
      load2(&vrows[jj][2 * lane], v2);
      o0 = fmaf(pj, v2[0], o0);
      o1 = fmaf(pj, v2[1], o1);
    }
    __syncwarp();  // the slices are refilled by the next chunk
  }
  const float inv = 1.0f / l;
  store2(static_cast<TIO*>(a.out_o) + gh * kD + 2 * lane, o0 * inv, o1 * inv);
  if (a.out_lse && lane == 0) a.out_lse[gh] = m + logf(l);
}

int launch_decode_int(const AttnArgs& a, const Plan& p, int dtype, void* stream) {
  const int64_t heads = (int64_t)a.B * a.Hq;
  const unsigned grid = (unsigned)((heads + kDecHeadsPerCta - 1) / kDecHeadsPerCta);
  if (grid == 0) return SFA_OK;
  // up to about one wave of staged CTAs (18-26 KB of shared memory each) the
  // staged kernel's shorter load chain wins; past that its occupancy loses
  const bool staged = heads <= kDecStagedMaxHeads;
  cudaStream_t s = (cudaStream_t)stream;
  const dim3 block(32 * kDecHeadsPerCta);
  LaunchTimer tm(SFA_KERNEL_DECODE, stream);
  cudaError_t e;
  if (dtype == SFA_BF16)
    e = staged ? launch_pdl(decode_staged_kernel<bf16>, dim3(grid), block, 0, s, a, p)
               : launch_pdl(decode_int_kernel<bf16>, dim3(grid), block, 0, s, a, p);
  else
    e = staged ? launch_pdl(decode_staged_kernel<float>, dim3(grid), block, 0, s, a, p)
               : launch_pdl(decode_int_kernel<float>, dim3(grid), block, 0, s, a, p);
  return e == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

}  // namespace sfa
