// Device helpers shared by the libsfa kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sfa_internal.h"

namespace sfa {

constexpr int kThreads = 256;   // threads per CTA of the attention kernels
constexpr int kRowPad = 68;     // floats per staged smem row (64 + 4: conflict-free float4 rows)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

using bf16 = __nv_bfloat16;

// Bounds checks of the SIMT kernels' indices, compiled in by SFA_DEBUG_BOUNDS
// (the bounds-checked build, libsfa_debug.so): an index outside [0, n) is
// recorded as SFA_ERR_DEVICE_BOUNDS in the status word and the access it
// guards is skipped; nothing traps.  In the release build the check is
// constant true and compiles away.
#ifdef SFA_DEBUG_BOUNDS
__device__ __forceinline__ bool dbg_in(int64_t i, int64_t n, int* status) {
  if (i >= 0 && i < n) return true;
  if (status) atomicCAS(status, 0, SFA_ERR_DEVICE_BOUNDS);
  return false;
}
#else
__device__ __forceinline__ bool dbg_in(int64_t, int64_t, int*) { return true; }
#endif

// Eight consecutive elements -> fp32.  p must be 16-byte aligned.
__device__ __forceinline__ void load8(const float* p, float* x) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void load8(const bf16* p, float* x) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}

__device__ __forceinline__ void load2(const float* p, float* x) {
  const float2 v = *reinterpret_cast<const float2*>(p);
  x[0] = v.x;
  x[1] = v.y;
}
__device__ __forceinline__ void load2(const bf16* p, float* x) {
  const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(p);
  x[0] = __bfloat162float(v.x);
  x[1] = __bfloat162float(v.y);
}
__device__ __forceinline__ void store2(float* p, float a, float b) {
  *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
__device__ __forceinline__ void store2(bf16* p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}
__device__ __forceinline__ void store8(float* p, const float* x) {
  reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

__device__ __forceinline__ void store8(bf16* p, const float* x) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}

// cos/sin of the 8 rotation pairs j0 .. j0+7 at position pos; table is
// [T][32] float2 (cos, sin).
__device__ __forceinline__ void load_rope8(const float2* tab, int64_t pos, int j0, float* cs,
                                           float* sn) {
  const float4* p = reinterpret_cast<const float4*>(tab + pos * 32 + j0);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float4 v = __ldg(p + e);
    cs[2 * e] = v.x;
    sn[2 * e] = v.y;
    cs[2 * e + 1] = v.z;
    sn[2 * e + 1] = v.w;
  }
}

// Rotate pairs (lo[e], hi[e]) = (x[j], x[j+32]) by +phi in place.
__device__ __forceinline__ void rotate8(float* lo, float* hi, const float* cs, const float* sn) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float a = lo[e], b = hi[e];
    lo[e] = a * cs[e] - b * sn[e];
    hi[e] = a * sn[e] + b * cs[e];
  }
}

// Load the pair chunk (dims 8pc..8pc+7 and 32+8pc..32+8pc+7) of row `row`,
// rotated by RoPE at position `pos` when tab != nullptr.
template <typename TIO>
__device__ __forceinline__ void load_pair_chunk(const TIO* row, int pc, const float2* tab,
                                                int64_t pos, float* lo, float* hi) {
  load8(row + 8 * pc, lo);
  load8(row + 32 + 8 * pc, hi);
  if (tab) {
    float cs[8], sn[8];
    load_rope8(tab, pos, 8 * pc, cs, sn);
    rotate8(lo, hi, cs, sn);
  }
}

__device__ __forceinline__ void st_smem8(float* p, const float* x) {
  reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

// Dot of a 32-float register half with the same half of a staged smem row.
__device__ __forceinline__ float dot32(const float* r, const float* s) {
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int e = 0; e < 32; e += 8) {
    const float4 a = *reinterpret_cast<const float4*>(s + e);
    const float4 b = *reinterpret_cast<const float4*>(s + e + 4);
    acc0 = fmaf(r[e], a.x, acc0);
    acc1 = fmaf(r[e + 1], a.y, acc1);
    acc0 = fmaf(r[e + 2], a.z, acc0);
    acc1 = fmaf(r[e + 3], a.w, acc1);
    acc0 = fmaf(r[e + 4], b.x, acc0);
    acc1 = fmaf(r[e + 5], b.y, acc1);
    acc0 = fmaf(r[e + 6], b.z, acc0);
    acc1 = fmaf(r[e + 7], b.w, acc1);
  }
  return acc0 + acc1;
}

// acc[0..32) += p * s[0..32)
__device__ __forceinline__ void axpy32(float* acc, float p, const float* s) {
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 a = *reinterpret_cast<const float4*>(s + e);
    acc[e] = fmaf(p, a.x, acc[e]);
    acc[e + 1] = fmaf(p, a.y, acc[e + 1]);
    acc[e + 2] = fmaf(p, a.z, acc[e + 2]);
    acc[e + 3] = fmaf(p, a.w, acc[e + 3]);
  }
}

}  // namespace sfa
