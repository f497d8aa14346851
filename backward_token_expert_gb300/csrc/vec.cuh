// 128-bit global memory helpers and bf16 packing used by the streaming
// kernels (score, compaction).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace lrm {

// Read-only streaming load: bypass L1, ask L2 to fetch the whole 256-byte
// neighbourhood (rows are read front to back).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_v4(uint4* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Adds the squares of the 8 bf16 values of v into 8 separate fp32 chains
// (the product of two bf16 values is exact in fp32).
__device__ __forceinline__ void acc_sq8(const uint4& v, float (&a)[8]) {
  a[0] = fmaf(bf16_lo(v.x), bf16_lo(v.x), a[0]);
  a[1] = fmaf(bf16_hi(v.x), bf16_hi(v.x), a[1]);
  a[2] = fmaf(bf16_lo(v.y), bf16_lo(v.y), a[2]);
  a[3] = fmaf(bf16_hi(v.y), bf16_hi(v.y), a[3]);
  a[4] = fmaf(bf16_lo(v.z), bf16_lo(v.z), a[4]);
  a[5] = fmaf(bf16_hi(v.z), bf16_hi(v.z), a[5]);
  a[6] = fmaf(bf16_lo(v.w), bf16_lo(v.w), a[6]);
  a[7] = fmaf(bf16_hi(v.w), bf16_hi(v.w), a[7]);
}

// Adds the magnitudes of the 8 bf16 values of v into 8 fp32 chains (the sign
// bit cleared).
__device__ __forceinline__ void acc_abs8(const uint4& v, float (&a)[8]) {
  a[0] += bf16_lo(v.x & 0x7FFF7FFFu);
  a[1] += bf16_hi(v.x & 0x7FFF7FFFu);
  a[2] += bf16_lo(v.y & 0x7FFF7FFFu);
  a[3] += bf16_hi(v.y & 0x7FFF7FFFu);
  a[4] += bf16_lo(v.z & 0x7FFF7FFFu);
  a[5] += bf16_hi(v.z & 0x7FFF7FFFu);
  a[6] += bf16_lo(v.w & 0x7FFF7FFFu);
  a[7] += bf16_hi(v.w & 0x7FFF7FFFu);
}

// bf16 pair (low, high) scaled by a: one fp32 multiply each, then
// round-to-nearest-even to bf16.
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t w, float a) {
  const __nv_bfloat162 r = __floats2bfloat162_rn(__fmul_rn(a, bf16_lo(w)), __fmul_rn(a, bf16_hi(w)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint4 scale_bf16x8(const uint4& v, float a) {
  return make_uint4(scale_bf16x2(v.x, a), scale_bf16x2(v.y, a), scale_bf16x2(v.z, a), scale_bf16x2(v.w, a));
}

}  // namespace lrm
