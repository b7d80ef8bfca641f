// Backward kernels of causal shared-offset sparse attention.
//
// Gradients of L = sum(O * dO) for the key set of "Depth-Staggered Fibonacci
// Spacing for Sparse Attention" (method section): window distances 0..W plus
// rungs read by two-row interpolation after RoPE.  With P the softmax
// weights, delta_i = dO_i . O_i, dP = dO . v~ and dS = P (dP - delta):
//   dq'_i = sum_slots dS k~ / 8,             dQ = R(-phi) dq'
//   window key j: dk'_j += dS q'_i / 8, dv_j += P dO_i   for i = j .. j + W
//   rung (c, w): the gradient of the interpolated row splits (1 - w) to row
//   i - c and w to row i - c + 1, so key row j collects it from queries
//   j + c (weight 1 - w) and j + c - 1 (weight w): an offset-transposed
//   gather, written by exactly one CTA per key row (no atomics).
//   dL/dd_k = sum dS q'.(k'[i-c] - k'[i-c+1]) / 8 + P dO.(v[i-c] - v[i-c+1])
//   (w = c - d with c fixed), dL/dalpha = sum_k f_k dL/dd_k and
//   dL/dtheta = dL/dalpha (alpha - 0.5)(1.5 - alpha).
//
// Three launches: bwd_q (per query tile: delta, dQ), bwd_kv (per key tile:
// dK, dV and per-CTA partials of dL/dalpha), dalpha_reduce (one CTA, fixed
// order fp64 sum).
#include <math.h>

#include "sfa_stage.cuh"

namespace sfa {

constexpr size_t kBwdQSmem = (size_t)(2 * kSlab * kRowPad) * sizeof(float);

// Full dot product of two 64-vectors held as 32-float halves by lanes t, t^1.
__device__ __forceinline__ float pair_dot(const float* r, const float* s) {
  const float part = dot32(r, s);
  return part + __shfl_xor_sync(0xffffffffu, part, 1);
}

template <typename TIO, bool INTERP>
__global__ void __launch_bounds__(kThreads, 2) bwd_q_kernel(const AttnArgs a,
                                                            const __grid_constant__ Plan P) {
  extern __shared__ float4 smem4[];
  float* sK = reinterpret_cast<float*>(smem4);
  float* sV = sK + kSlab * kRowPad;

  const int G = 1 << a.lgG, TQ = 128 >> a.lgG;
  const int t = threadIdx.x, half = t & 1, qh = t >> 1;
  const int pl = qh >> a.lgG, hl = qh & (G - 1);
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int i0 = blockIdx.x * TQ, i = i0 + pl, h = g * G + hl;
  const bool active = i < a.T && dbg_in((int64_t)(b * a.Hq + h) * a.T + i, (int64_t)a.B * a.Hq * a.T, a.status);
  const int ic = active ? i : 0;
  const int imax = min(a.T - 1, i0 + TQ - 1);
  const int64_t rowidx = (int64_t)(b * a.Hq + h) * a.T + ic;
  const int64_t qrow = rowidx * kD;
  const TIO* Kb = static_cast<const TIO*>(a.k) + (int64_t)bg * a.T * kD;
  const TIO* Vb = static_cast<const TIO*>(a.v) + (int64_t)bg * a.T * kD;
  const float2* rope = static_cast<const float2*>(a.rope);

  // q~ = q'/8 (my half), dO (my half), delta = dO . O
  float qr[32], dor[32], dq[32];
  float delta;
  {
    const TIO* qp = static_cast<const TIO*>(a.q) + qrow;
    const TIO* dp = static_cast<const TIO*>(a.dO) + qrow + half * 32;
    const TIO* op = static_cast<const TIO*>(a.o) + qrow + half * 32;
    float part = 0.0f;
#pragma unroll
    for (int pc = 0; pc < 4; ++pc) {
      float lo[8], hi[8], ov[8];
      load_pair_chunk(qp, pc, rope, ic, lo, hi);
#pragma unroll
      for (int e = 0; e < 8; ++e) qr[8 * pc + e] = (half ? hi[e] : lo[e]) * 0.125f;
      load8(dp + 8 * pc, dor + 8 * pc);
      load8(op + 8 * pc, ov);
#pragma unroll
      for (int e = 0; e < 8; ++e) part = fmaf(dor[8 * pc + e], ov[e], part);
    }
    delta = part + __shfl_xor_sync(0xffffffffu, part, 1);
  }
#pragma unroll
  for (int e = 0; e < 32; ++e) dq[e] = 0.0f;
  const float lse2 = active ? a.lse[rowidx] * kLog2e : 0.0f;
  if (active && half == 0) a.delta[rowidx] = delta;

  // One slot: P, dS and the dq update.  `ok` is uniform across the lane pair.
  auto slot_update = [&](bool ok, int row) {
    ok = ok && dbg_in(row, kSlab, a.status);
    const int r = ok ? row : 0;
    const float s = pair_dot(qr, sK + r * kRowPad + half * 32);
    const float dp = pair_dot(dor, sV + r * kRowPad + half * 32);
    if (!ok) return;
    const float p = exp2f(fmaf(s, kLog2e, -lse2));
    const float ds = p * (dp - delta);
    axpy32(dq, ds, sK + r * kRowPad + half * 32);
  };

  const int wmax = min(P.W, imax);
  for (int s_lo = 0; s_lo <= wmax; s_lo += kWinChunk) {
    const int s_hi = min(wmax, s_lo + kWinChunk - 1);
    const int pos_lo = i0 - s_hi;
    __syncthreads();
    stage_rows<TIO>(Kb, Vb, rope, pos_lo, imax - s_lo - pos_lo + 1, sK, sV, a.T, a.status);
    __syncthreads();
    for (int s = s_lo; s <= s_hi; ++s) slot_update(active && i >= s, pl + (s_hi - s));
  }
  int nr = 0;
  while (nr < P.n && P.c[nr] <= imax) ++nr;
  const int RB = min(kMaxBatch, kSlab / TQ);
  for (int r0 = 0; r0 < nr; r0 += RB) {
    const int nb = min(RB, nr - r0);
    __syncthreads();
    stage_rungs<TIO, INTERP>(Kb, Vb, rope, P, r0, nb, i0, TQ, a.T, sK, sV, a.status);
    __syncthreads();
    for (int x = 0; x < nb; ++x)
      slot_update(active && i >= P.c[r0 + x] && i - P.c[r0 + x] < a.T, x * TQ + pl);
  }

  // dq' = sum dS k~ / 8 (the logit is q'.k~/8); dQ = R(-phi) dq'.  The
  // rotation pairs dim j (lane half 0) with dim j + 32 (lane half 1).
  float other[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    dq[e] *= 0.125f;
    other[e] = __shfl_xor_sync(0xffffffffu, dq[e], 1);
  }
  if (!active) return;
  float out[32];
  if (rope) {
#pragma unroll
    for (int pc = 0; pc < 4; ++pc) {
      float cs[8], sn[8];
      load_rope8(rope, ic, 8 * pc, cs, sn);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = 8 * pc + e;
        // half 0 owns dim j (partner holds j + 32); half 1 owns j + 32.
        out[j] = half ? (dq[j] * cs[e] - other[j] * sn[e]) : (dq[j] * cs[e] + other[j] * sn[e]);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) out[e] = dq[e];
  }
  TIO* dqp = static_cast<TIO*>(a.dq) + qrow + half * 32;
#pragma unroll
  for (int c8 = 0; c8 < 4; ++c8) store8(dqp + 8 * c8, out + 8 * c8);
}


constexpr int kKvChunk = 8;  // window distances per key-side batch

__host__ __device__ constexpr int kv_rows(int lgG) { return (128 >> lgG) + kKvChunk - 1; }
__host__ __device__ constexpr size_t kv_smem_floats(int lgG) {
  return (size_t)2 * ((128 >> lgG) + 2) * kRowPad +
         (size_t)kv_rows(lgG) * (1 << lgG) * (2 * kRowPad + 2);
}

// Dot of two 64-vectors stored in shared memory, split over the lane pair.
__device__ __forceinline__ float pair_dot_ss(const float* x, const float* y) {
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 u = *reinterpret_cast<const float4*>(x + e);
    const float4 v = *reinterpret_cast<const float4*>(y + e);
    acc0 = fmaf(u.x, v.x, acc0);
    acc1 = fmaf(u.y, v.y, acc1);
    acc0 = fmaf(u.z, v.z, acc0);
    acc1 = fmaf(u.w, v.w, acc1);
  }
  const float part = acc0 + acc1;
  return part + __shfl_xor_sync(0xffffffffu, part, 1);
}

// Stage the query-side rows of positions [pos_lo, pos_lo + nrows) for all G
// heads of the group: q~ = R(phi) q / 8, dO, LSE * log2(e) and delta.
template <typename TIO>
__device__ __forceinline__ void stage_queries(const AttnArgs& a, int b, int g, int G, int pos_lo,
                                              int nrows, float* sQ, float* sD, float* sLse,
                                              float* sDel, int rows_cap) {
  const float2* rope = static_cast<const float2*>(a.rope);
  for (int it = threadIdx.x; it < nrows * G * 4; it += kThreads) {
    const int pc = it & 3, rh = it >> 2;
    const int r = rh / G, hh = rh - r * G;
    const int pos = pos_lo + r;
    if (pos < 0 || pos >= a.T) continue;
    const int64_t ridx = (int64_t)(b * a.Hq + g * G + hh) * a.T + pos;
    if (!dbg_in(r * G + hh, (int64_t)rows_cap * G, a.status) ||
        !dbg_in(ridx, (int64_t)a.B * a.Hq * a.T, a.status))
      continue;
    float lo[8], hi[8];
    load_pair_chunk(static_cast<const TIO*>(a.q) + ridx * kD, pc, rope, pos, lo, hi);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      lo[e] *= 0.125f;
      hi[e] *= 0.125f;
    }
    float* q = sQ + (r * G + hh) * kRowPad;
    st_smem8(q + 8 * pc, lo);
    st_smem8(q + 32 + 8 * pc, hi);
    load_pair_chunk<TIO>(static_cast<const TIO*>(a.dO) + ridx * kD, pc, nullptr, pos, lo, hi);
    float* d = sD + (r * G + hh) * kRowPad;
    st_smem8(d + 8 * pc, lo);
    st_smem8(d + 32 + 8 * pc, hi);
    if (pc == 0) {
      sLse[r * G + hh] = a.lse[ridx] * kLog2e;
      sDel[r * G + hh] = a.delta[ridx];
    }
  }
}

template <typename TIO, bool INTERP>
__global__ void __launch_bounds__(kThreads, 1) bwd_kv_kernel(const AttnArgs a,
                                                             const __grid_constant__ Plan P) {
  extern __shared__ float4 smem4[];
  const int G = 1 << a.lgG, TK = 128 >> a.lgG, QR = kv_rows(a.lgG);
  float* sKt = reinterpret_cast<float*>(smem4);  // rows j0-1 .. j0+TK
  float* sVt = sKt + (TK + 2) * kRowPad;
  float* sQ = sVt + (TK + 2) * kRowPad;           // [QR][G][kRowPad]
  float* sD = sQ + QR * G * kRowPad;
  float* sLse = sD + QR * G * kRowPad;            // [QR][G]
  float* sDel = sLse + QR * G;

  const int t = threadIdx.x, half = t & 1, kh = t >> 1;
  const int jl = kh >> a.lgG, hl = kh & (G - 1);
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int j0 = blockIdx.x * TK, j = j0 + jl;
  const bool active = j < a.T;
  const int jmax = min(a.T - 1, j0 + TK - 1);
  const TIO* Kb = static_cast<const TIO*>(a.k) + (int64_t)bg * a.T * kD;
  const TIO* Vb = static_cast<const TIO*>(a.v) + (int64_t)bg * a.T * kD;
  const float2* rope = static_cast<const float2*>(a.rope);

  // key tile with one halo row on each side; rows outside [0, T) are zero
  for (int it = t; it < (TK + 2) * 4; it += kThreads) {
    const int r = it >> 2, pc = it & 3, pos = j0 - 1 + r;
    float lo[8] = {0}, hi[8] = {0}, vl[8] = {0}, vh[8] = {0};
    if (pos >= 0 && pos < a.T) {
      load_pair_chunk(Kb + (int64_t)pos * kD, pc, rope, pos, lo, hi);
      load_pair_chunk<TIO>(Vb + (int64_t)pos * kD, pc, nullptr, pos, vl, vh);
    }
    st_smem8(sKt + r * kRowPad + 8 * pc, lo);
    st_smem8(sKt + r * kRowPad + 32 + 8 * pc, hi);
    st_smem8(sVt + r * kRowPad + 8 * pc, vl);
    st_smem8(sVt + r * kRowPad + 32 + 8 * pc, vh);
  }

  float dk[32], dv[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) dk[e] = dv[e] = 0.0f;
  double dacc = 0.0;
  const int hoff = half * 32;
  const float* kj = sKt + (jl + 1) * kRowPad + hoff;
  const float* vj = sVt + (jl + 1) * kRowPad + hoff;

  // window: queries i = j + s, s = 0..W
  const int wmax = min(P.W, a.T - 1 - j0);
  for (int s_lo = 0; s_lo <= wmax; s_lo += kKvChunk) {
    const int s_hi = min(wmax, s_lo + kKvChunk - 1);
    const int pos_lo = j0 + s_lo;
    __syncthreads();
    stage_queries<TIO>(a, b, g, G, pos_lo, min(a.T - 1, jmax + s_hi) - pos_lo + 1, sQ, sD, sLse,
                       sDel, QR);
    __syncthreads();
    for (int s = s_lo; s <= s_hi; ++s) {
      const bool ok = active && j + s < a.T && dbg_in((jl + s - s_lo) * G + hl, (int64_t)QR * G, a.status);
      const int r = ok ? (jl + s - s_lo) * G + hl : hl;
      const float* q = sQ + r * kRowPad + hoff;
      const float* d = sD + r * kRowPad + hoff;
      const float sc = pair_dot_ss(q, kj);
      const float dp = pair_dot_ss(d, vj);
      if (!ok) continue;
      const float p = exp2f(fmaf(sc, kLog2e, -sLse[r]));
      const float ds = p * (dp - sDel[r]);
      axpy32(dk, ds, q);
      axpy32(dv, p, d);
    }
  }

  // rungs: key row j gets query j + c (as the floor row, weight 1 - w) and
  // query j + c - 1 (as the floor-plus-one row, weight w).
  int nr = 0;
  while (nr < P.n && P.c[nr] <= a.T - j0) ++nr;
  for (int rg = 0; rg < nr; ++rg) {
    const int c = P.c[rg];
    const float w = INTERP ? P.w[rg] : 0.0f;
    const float u = 1.0f - w;
    const int pos_lo = j0 + c - 1;
    __syncthreads();
    stage_queries<TIO>(a, b, g, G, pos_lo, min(a.T - 1, jmax + c) - pos_lo + 1, sQ, sD, sLse,
                       sDel, QR);
    __syncthreads();
    // query j + c: interpolates rows j (weight u) and j + 1 (weight w)
    {
      const bool ok = active && j + c >= 0 && j + c < a.T && dbg_in((jl + 1) * G + hl, (int64_t)QR * G, a.status);
      const int r = (ok ? jl + 1 : 0) * G + hl;
      const float* q = sQ + r * kRowPad + hoff;
      const float* d = sD + r * kRowPad + hoff;
      const float sa = pair_dot_ss(q, kj), da = pair_dot_ss(d, vj);
      float sb = 0.0f, db = 0.0f;
      if (INTERP) {
        sb = pair_dot_ss(q, kj + kRowPad);
        db = pair_dot_ss(d, vj + kRowPad);
      }
      if (ok) {
        const float sc = INTERP ? fmaf(w, sb, u * sa) : sa;
        const float dp = INTERP ? fmaf(w, db, u * da) : da;
        const float p = exp2f(fmaf(sc, kLog2e, -sLse[r]));
        const float ds = p * (dp - sDel[r]);
        axpy32(dk, u * ds, q);
        axpy32(dv, u * p, d);
        if (INTERP && half == 0)  // dL/dd_k of this (query, rung), times f_k
          dacc += (double)P.f[rg] * (double)(ds * (sa - sb) + p * (da - db));
      }
    }
    // query j + c - 1: interpolates rows j - 1 (weight u) and j (weight w)
    if (INTERP && w != 0.0f) {
      const bool ok = active && j >= 1 && j + c - 1 < a.T && dbg_in(jl * G + hl, (int64_t)QR * G, a.status);
      const int r = (ok ? jl : 0) * G + hl;
      const float* q = sQ + r * kRowPad + hoff;
      const float* d = sD + r * kRowPad + hoff;
      const float sa = pair_dot_ss(q, kj - kRowPad), da = pair_dot_ss(d, vj - kRowPad);
      const float sb = pair_dot_ss(q, kj), db = pair_dot_ss(d, vj);
      if (ok) {
        const float p = exp2f(fmaf(fmaf(w, sb, u * sa), kLog2e, -sLse[r]));
        const float ds = p * (fmaf(w, db, u * da) - sDel[r]);
        axpy32(dk, w * ds, q);
        axpy32(dv, w * p, d);
      }
    }
  }

  // sum over the G heads of the group (fixed order), then dK = R(-phi) dk'
  __syncthreads();
  float* rk = sQ;  // [TK][G][kRowPad]
  float* rv = sD;
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    *reinterpret_cast<float4*>(rk + kh * kRowPad + hoff + e) =
        make_float4(dk[e], dk[e + 1], dk[e + 2], dk[e + 3]);
    *reinterpret_cast<float4*>(rv + kh * kRowPad + hoff + e) =
        make_float4(dv[e], dv[e + 1], dv[e + 2], dv[e + 3]);
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    float sk = 0.0f, sv = 0.0f;
    for (int hh = 0; hh < G; ++hh) {
      sk += rk[(jl * G + hh) * kRowPad + hoff + e];
      sv += rv[(jl * G + hh) * kRowPad + hoff + e];
    }
    dk[e] = sk;
    dv[e] = sv;
  }
  float other[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) other[e] = __shfl_xor_sync(0xffffffffu, dk[e], 1);
  if (active && hl == 0 && dbg_in((int64_t)bg * a.T + j, (int64_t)a.B * a.Hkv * a.T, a.status)) {
    const int64_t krow = ((int64_t)bg * a.T + j) * kD + hoff;
    float out[32];
    if (rope) {
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        float cs[8], sn[8];
        load_rope8(rope, j, 8 * pc, cs, sn);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int x = 8 * pc + e;
          out[x] = half ? (dk[x] * cs[e] - other[x] * sn[e]) : (dk[x] * cs[e] + other[x] * sn[e]);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) out[e] = dk[e];
    }
    TIO* kp = static_cast<TIO*>(a.dk) + krow;
    TIO* vp = static_cast<TIO*>(a.dv) + krow;
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
      store8(kp + 8 * c8, out + 8 * c8);
      store8(vp + 8 * c8, dv + 8 * c8);
    }
  }

  if (INTERP) {  // per-CTA partial of dL/dalpha, fixed-order reduction
    __shared__ double wsum[kThreads / 32];
    for (int off = 16; off > 0; off >>= 1) dacc += __shfl_down_sync(0xffffffffu, dacc, off);
    if ((t & 31) == 0) wsum[t >> 5] = dacc;
    __syncthreads();
    if (t == 0) {
      double s = 0.0;
      for (int x = 0; x < kThreads / 32; ++x) s += wsum[x];
      a.dalpha_part[(int64_t)blockIdx.y * gridDim.x + blockIdx.x] = s;
    }
  }
}

__global__ void dalpha_reduce_kernel(const double* part, int64_t n, double alpha, double* out) {
  __shared__ double sh[256];
  double s = 0.0;
  for (int64_t x = threadIdx.x; x < n; x += 256) s += part[x];
  sh[threadIdx.x] = s;
  __syncthreads();
  for (int off = 128; off > 0; off >>= 1) {
    if ((int)threadIdx.x < off) sh[threadIdx.x] += sh[threadIdx.x + off];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    out[0] = sh[0];
    out[1] = sh[0] * (alpha - 0.5) * (1.5 - alpha);
  }
}

static int kv_grid_x(int T, int lgG) { return (T + (128 >> lgG) - 1) / (128 >> lgG); }

size_t backward_workspace_bytes(const sfa_desc* d, const Plan& p) {
  (void)p;
  const int lgG = __builtin_ctz((unsigned)(d->Hq / d->Hkv));
  const size_t nparts = (size_t)kv_grid_x(d->T, lgG) * d->B * d->Hkv;
  return align256(nparts * sizeof(double)) + (size_t)d->B * d->Hq * d->T * sizeof(float);
}

template <typename TIO, bool INTERP>
static int launch_bwd_t(const AttnArgs& a, const Plan& p, cudaStream_t s) {
  const int TQ = 128 >> a.lgG;
  auto kq = bwd_q_kernel<TIO, INTERP>;
  auto kkv = bwd_kv_kernel<TIO, INTERP>;
  const size_t kvs = kv_smem_floats(a.lgG) * sizeof(float);
  if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBwdQSmem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kvs) !=
          cudaSuccess)
    return SFA_ERR_CUDA;
  dim3 gq((unsigned)((a.T + TQ - 1) / TQ), (unsigned)(a.B * a.Hkv));
  {
    LaunchTimer tm(SFA_KERNEL_BWD_Q, s);
    kq<<<gq, kThreads, kBwdQSmem, s>>>(a, p);
  }
  dim3 gkv((unsigned)kv_grid_x(a.T, a.lgG), (unsigned)(a.B * a.Hkv));
  {
    LaunchTimer tm(SFA_KERNEL_BWD_KV, s);
    kkv<<<gkv, kThreads, kvs, s>>>(a, p);
  }
  if (INTERP && a.dalpha_out) {
    LaunchTimer tm(SFA_KERNEL_DALPHA, s);
    dalpha_reduce_kernel<<<1, 256, 0, s>>>(a.dalpha_part, (int64_t)gkv.x * gkv.y, a.alpha,
                                           a.dalpha_out);
  }
  return cudaGetLastError() == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

int launch_backward(const AttnArgs& a, const Plan& p, int dtype, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == SFA_BF16)
    return p.interp ? launch_bwd_t<bf16, true>(a, p, s) : launch_bwd_t<bf16, false>(a, p, s);
  return p.interp ? launch_bwd_t<float, true>(a, p, s) : launch_bwd_t<float, false>(a, p, s);
}

}  // namespace sfa
