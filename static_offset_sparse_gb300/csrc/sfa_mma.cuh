// Warp-level tensor-core helpers (inline PTX, sm_103a).
//
// mma.sync m16n8k16 bf16 -> fp32 fragment layouts used throughout (lane =
// 4 * gid + tig, gid = lane >> 2, tig = lane & 3):
//   A (16x16, row-major): a0 (row gid,   k 2tig..2tig+1)  a1 (row gid+8, same k)
//                         a2 (row gid,   k 2tig+8..+9)    a3 (row gid+8, same k)
//   B (16x8, k-major):    b0 (k 2tig..2tig+1, n gid)      b1 (k 2tig+8..+9, n gid)
//   C (16x8, fp32):       c0,c1 (row gid, n 2tig..+1)     c2,c3 (row gid+8, same n)
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>

namespace sfa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ldmatrix: four 8x8 b16 tiles from shared memory (lanes 8t..8t+7 give tile t's row addresses).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// d += a * b  (bf16 inputs, fp32 accumulate)
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d += a * b for k = 8 (m16n8k8): a0 (row gid, k 2tig..2tig+1), a1 (row
// gid+8, same k), b0 (k 2tig..2tig+1, n gid).
__device__ __forceinline__ void mma_bf16_k8(float* d, const uint32_t* a, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(b0));
}

// 2^x with the hardware approximation (ex2.approx.ftz; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Two floats -> packed bf16x2 (round to nearest even); x in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(h);
}

}  // namespace sfa
