// i8_common.cuh -- int8 -> fp16 conversion into the tcgen05 operand layout,
// shared by the INT8 kernels (i8tc.cu, fwd_i8x.cu). Every int8 value is
// exact in fp16, so an fp16 kind::f16 MMA with fp32 accumulation returns the
// exact integer dot for the dimensions these kernels accept.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace msim {
namespace {

// Four int8 (as biased bytes u = x + 128 in `xb`) -> two fp16x2 words holding
// x exactly: PRMT puts each byte under the fp16 exponent byte 0x64 (value
// 1024 + u), then one packed subtract of 1152. This is the standard
// exponent-bias ("magic number") integer-to-float conversion: fp16 numbers in
// [1024, 2048) have a spacing of exactly 1, so their low 10 mantissa bits are
// an unsigned integer u < 1024 added to 1024; 0x6400 is 1024.0 and 0x6480 is
// 1152.0 = 1024 + 128, so the subtract removes both the exponent bias and the
// +128 byte bias with no rounding (every operand and result is an integer of
// magnitude < 2048).
__device__ __forceinline__ uint32_t h2_of(uint32_t xb, uint32_t sel) {
  uint32_t r, o;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(xb), "r"(0x64646464u), "r"(sel));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o) : "r"(r), "r"(0x64806480u));
  return o;
}

__device__ __forceinline__ uint4 lds_u4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_u4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// 16 int8 of row r, dims 16 ci .. 16 ci + 15, into the fp16 K-major SW128
// layout at `dst` (atoms of 64 dims x `rows_per_atom` rows; 16-byte chunk c
// of row r stored at chunk c ^ (r & 7)).
__device__ __forceinline__ void cvt16(uint4 w, uint32_t dst, int r, int ci, uint32_t atom_bytes) {
  const uint32_t x0 = w.x ^ 0x80808080u, x1 = w.y ^ 0x80808080u, x2 = w.z ^ 0x80808080u, x3 = w.w ^ 0x80808080u;
  const int a = ci >> 2, c0 = (ci & 3) * 2;
  const uint32_t row = dst + a * atom_bytes + static_cast<uint32_t>(r) * 128;
  sts_u4(row + ((c0 ^ (r & 7)) << 4), h2_of(x0, 0x4140), h2_of(x0, 0x4342), h2_of(x1, 0x4140), h2_of(x1, 0x4342));
  sts_u4(row + (((c0 + 1) ^ (r & 7)) << 4), h2_of(x2, 0x4140), h2_of(x2, 0x4342), h2_of(x3, 0x4140),
         h2_of(x3, 0x4342));
}

}  // namespace
}  // namespace msim
