// Forward kernel of causal shared-offset sparse attention, and the RoPE table.
//
// "Depth-Staggered Fibonacci Spacing for Sparse Attention", method section:
// query i attends window distances 0..W and rungs d_k = alpha f_k, a rung row
// being the interpolation (1 - w) row[i - c] + w row[i - c + 1] with
// c = ceil(d_k), w = c - d_k, after RoPE at each row's own position.
//
// Layout of the work: one CTA per (query tile, batch b, KV head g).  The tile
// holds TQ = 128 / G query positions and all G query heads of the group, so
// every staged key/value row is read by G heads.  Two threads share one
// (position, head): each holds half of the 64 dims (q and the output
// accumulator), and a single shuffle completes each dot product.
//
// Offsets are shared by all queries, so for each rung the rows the tile needs
// form one contiguous, shifted slab: the CTA stages it (RoPE and the two-row
// interpolation applied on the way in) into shared memory in fp32, then every
// thread reads the one row that belongs to its position.  The window is staged
// as one slab per chunk of distances.  Softmax is online across batches of
// slots, in base 2, with fp32 accumulation.
#include <math.h>

#include "sfa_stage.cuh"

namespace sfa {

constexpr size_t kFwdSmem = (size_t)(2 * kSlab * kRowPad + kMaxBatch * kThreads) * sizeof(float);

// Online-softmax update over one batch of ns slots.  slot(a, row) returns
// whether slot a is a key of this thread's query and sets the staged row.
// Logits are in log2 units (q was pre-scaled by log2(e) / sqrt(D)).
template <typename SlotFn>
__device__ __forceinline__ void softmax_batch(int ns, SlotFn slot, const float* qr,
                                              const float* sK, const float* sV, float* sL,
                                              float& m, float& l, float* acc) {
  const int t = threadIdx.x, half = t & 1;
  float mloc = -INFINITY;
  for (int a = 0; a < ns; ++a) {
    int row;
    const bool ok = slot(a, row);
    const float part = dot32(qr, sK + (ok ? row : 0) * kRowPad + half * 32);
    const float sv = part + __shfl_xor_sync(0xffffffffu, part, 1);
    const float s = ok ? sv : -INFINITY;
    sL[a * kThreads + t] = s;
    mloc = fmaxf(mloc, s);
  }
  if (mloc == -INFINITY) return;  // no key of this query in the batch
  const float mnew = fmaxf(m, mloc);
  const float corr = exp2f(m - mnew);
  l *= corr;
#pragma unroll
  for (int e = 0; e < 32; ++e) acc[e] *= corr;
  for (int a = 0; a < ns; ++a) {
    const float s = sL[a * kThreads + t];
    if (s == -INFINITY) continue;
    int row;
    slot(a, row);
    const float p = exp2f(s - mnew);
    l += p;
    axpy32(acc, p, sV + row * kRowPad + half * 32);
  }
  m = mnew;
}

template <typename TIO, bool INTERP>
__global__ void __launch_bounds__(kThreads, 2) fwd_kernel(const AttnArgs a,
                                                          const __grid_constant__ Plan P) {
  extern __shared__ float4 smem4[];
  float* sK = reinterpret_cast<float*>(smem4);
  float* sV = sK + kSlab * kRowPad;
  float* sL = sV + kSlab * kRowPad;

  const int G = 1 << a.lgG, TQ = 128 >> a.lgG;
  const int t = threadIdx.x, half = t & 1, qh = t >> 1;
  const int pl = qh >> a.lgG, hl = qh & (G - 1);
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int i0 = blockIdx.x * TQ, i = i0 + pl, h = g * G + hl;
  const bool active = i < a.T;
  const int imax = min(a.T - 1, i0 + TQ - 1);
  const int64_t qrow = ((int64_t)(b * a.Hq + h) * a.T + (active ? i : 0)) * kD;
  const TIO* Kb = static_cast<const TIO*>(a.k) + (int64_t)bg * a.T * kD;
  const TIO* Vb = static_cast<const TIO*>(a.v) + (int64_t)bg * a.T * kD;
  const float2* rope = static_cast<const float2*>(a.rope);

  // q' (rotated at position i), pre-scaled by log2(e)/sqrt(64); my half only.
  float qr[32];
  {
    const TIO* qp = static_cast<const TIO*>(a.q) + qrow;
    const float sc = 0.125f * kLog2e;
#pragma unroll
    for (int pc = 0; pc < 4; ++pc) {
      float lo[8], hi[8];
      load_pair_chunk(qp, pc, rope, active ? i : 0, lo, hi);
#pragma unroll
      for (int e = 0; e < 8; ++e) qr[8 * pc + e] = (half ? hi[e] : lo[e]) * sc;
    }
  }
  float m = -INFINITY, l = 0.0f, acc[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) acc[e] = 0.0f;

  // window: distances 0..W in chunks; slab rows are positions pos_lo .. imax - s_lo
  const int wmax = min(P.W, imax);
  for (int s_lo = 0; s_lo <= wmax; s_lo += kWinChunk) {
    const int s_hi = min(wmax, s_lo + kWinChunk - 1);
    const int pos_lo = i0 - s_hi;
    __syncthreads();
    stage_rows<TIO>(Kb, Vb, rope, pos_lo, imax - s_lo - pos_lo + 1, sK, sV, a.T, a.status);
    __syncthreads();
    softmax_batch(
        s_hi - s_lo + 1,
        [&](int x, int& row) {
          const int s = s_lo + x;
          row = pl + (s_hi - s);
          return active && i >= s && dbg_in(row, kSlab, a.status);
        },
        qr, sK, sV, sL, m, l, acc);
  }

  // rungs (sorted by c): only those reaching some query of the tile
  int nr = 0;
  while (nr < P.n && P.c[nr] <= imax) ++nr;
  const int RB = min(kMaxBatch, kSlab / TQ);
  for (int r0 = 0; r0 < nr; r0 += RB) {
    const int nb = min(RB, nr - r0);
    __syncthreads();
    stage_rungs<TIO, INTERP>(Kb, Vb, rope, P, r0, nb, i0, TQ, a.T, sK, sV, a.status);
    __syncthreads();
    softmax_batch(
        nb,
        [&](int x, int& row) {
          row = x * TQ + pl;
          return active && i >= P.c[r0 + x] && i - P.c[r0 + x] < a.T && dbg_in(row, kSlab, a.status);
        },
        qr, sK, sV, sL, m, l, acc);
  }

  if (active && dbg_in((int64_t)(b * a.Hq + h) * a.T + i, (int64_t)a.B * a.Hq * a.T, a.status)) {
    const float inv = 1.0f / l;
    TIO* op = static_cast<TIO*>(a.out_o) + qrow + half * 32;
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = acc[8 * c8 + e] * inv;
      store8(op + 8 * c8, x);
    }
    if (half == 0) a.out_lse[(int64_t)(b * a.Hq + h) * a.T + i] = (m + log2f(l)) * kLn2;
  }
}

__global__ void rope_table_kernel(int T, double theta, float2* tab) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)T * 32) return;
  const int t = (int)(idx >> 5), j = (int)(idx & 31);
  const double inv = pow(theta, -(2.0 * j) / 64.0);
  double s, c;
  sincos((double)t * inv, &s, &c);
  tab[idx] = make_float2((float)c, (float)s);
}

int launch_rope_table(int T, double theta, float* table, void* stream) {
  const int64_t n = (int64_t)T * 32;
  LaunchTimer tm(SFA_KERNEL_ROPE, stream);
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
      T, theta, reinterpret_cast<float2*>(table));
  return cudaGetLastError() == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

template <typename TIO, bool INTERP>
static int launch_fwd_t(const AttnArgs& a, const Plan& p, cudaStream_t s) {
  auto kern = fwd_kernel<TIO, INTERP>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFwdSmem) !=
      cudaSuccess)
    return SFA_ERR_CUDA;
  const int TQ = 128 >> a.lgG;
  dim3 grid((unsigned)((a.T + TQ - 1) / TQ), (unsigned)(a.B * a.Hkv));
  {
    LaunchTimer tm(SFA_KERNEL_FWD, s);
    kern<<<grid, kThreads, kFwdSmem, s>>>(a, p);
  }
  return cudaGetLastError() == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
}

int launch_forward(const AttnArgs& a, const Plan& p, int dtype, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == SFA_BF16)
    return p.interp ? launch_fwd_t<bf16, true>(a, p, s) : launch_fwd_t<bf16, false>(a, p, s);
  return p.interp ? launch_fwd_t<float, true>(a, p, s) : launch_fwd_t<float, false>(a, p, s);
}

}  // namespace sfa
