// Device helpers of the kernels that read the compressed pool with tensor
// cores: shared-memory addresses, cp.async, predicated stores, the code ->
// fp16 conversions and mma.sync m16n8k16 (fp16 in, fp32 accumulate).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace kvc {
namespace codes {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}
// A 16-byte cp.async done only when `pred` (no branch).
__device__ __forceinline__ void cp_async16_if(bool pred, uint32_t dst, const void* src) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n"
      " @q cp.async.cg.shared.global [%1], [%2], 16;\n}\n" ::"r"((uint32_t)pred),
      "r"(dst), "l"(src));
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Two floats to global memory only when `pred`, kept in L2 by `policy`.
__device__ __forceinline__ void st2_if_hint(bool pred, float* dst, float a, float b, uint64_t policy) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n"
      " @q st.global.L2::cache_hint.v2.f32 [%1], {%2, %3}, %4;\n}\n" ::"r"((uint32_t)pred),
      "l"(dst), "f"(a), "f"(b), "l"(policy)
      : "memory");
}
// Two floats to global memory only when `pred` (no branch).
__device__ __forceinline__ void st2_if(bool pred, float* dst, float a, float b) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n"
      " @q st.global.v2.f32 [%1], {%2, %3};\n}\n" ::"r"((uint32_t)pred),
      "l"(dst), "f"(a), "f"(b)
      : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_half2(uint32_t u) {
  return __half22float2(*reinterpret_cast<__half2*>(&u));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// x (two fp32 values) as a bf16 pair plus the bf16 pair of its remainder:
// together 16 significant bits (x - hi is exact in fp32)
__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x - __low2float(h), y - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
// bf16 pair times 16 (exact: a power of two)
__device__ __forceinline__ uint32_t bf16x2_times16(uint32_t v) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&v);
  x = __hmul2(x, __floats2bfloat162_rn(16.0f, 16.0f));
  return *reinterpret_cast<uint32_t*>(&x);
}

// Integer codes enter the MMA as fp16 subnormals: a field of u < 1024 in the
// low mantissa bits of an fp16 (exponent bits zero) is exactly u * 2^-24.
// The codes are offset to unsigned first (INT8: c + 128, INT4: c + 8, by
// flipping the field's top bit), so every product and partial sum is exact
// or rounded as an fp16 x fp16 -> fp32 MMA rounds it; the offsets come back
// out once per dot product (K) or once per output (V), see the kernel.
// INT8: bytes 0 and 2 of w -> (b0 + 128, b2 + 128) * 2^-24.
// One logic instruction each: (w & mask) ^ flip, written as lop3 so that the
// mask and the flip are not split into two.
__device__ __forceinline__ uint32_t and_xor(uint32_t w, uint32_t mask, uint32_t flip) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(w), "r"(mask), "r"(flip));
  return d;
}
__device__ __forceinline__ uint32_t u8_even(uint32_t w) { return and_xor(w, 0x00FF00FFu, 0x00800080u); }
// INT4: the low nibble of each 16-bit half -> (n + 8) * 2^-24.
__device__ __forceinline__ uint32_t u4_lo(uint32_t w) { return and_xor(w, 0x000F000Fu, 0x00080008u); }
// INT4: bits 4..7 of each 16-bit half -> 16 (n + 8) * 2^-24.
__device__ __forceinline__ uint32_t u4_hi(uint32_t w) { return and_xor(w, 0x00F000F0u, 0x00800080u); }

// FP8 E4M3 codes -> fp16 (every E4M3 value is exact in fp16), by the
// conversion instruction: 4 codes (bytes b0..b3 of w) -> (b0, b1) and (b2, b3).
__device__ __forceinline__ void e4m3x4_to_h2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l, h;\n"
      " mov.b32 {l, h}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l;\n"
      " cvt.rn.f16x2.e4m3x2 %1, h;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// Byte k of x and byte k of y (E4M3 codes) -> fp16x2 (x_k, y_k).
__device__ __forceinline__ uint32_t e4m3_pair_to_h2(uint32_t x, uint32_t y, int k) {
  const uint32_t pr = prmt(x, y, (uint32_t)k | ((uint32_t)(4 + k) << 4));
  uint32_t d;
  asm("{\n .reg .b16 l, h;\n"
      " mov.b32 {l, h}, %1;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l;\n}"
      : "=r"(d)
      : "r"(pr));
  return d;
}

// 2^e as a float, for -126 <= e <= 127 (exact).
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

// Unbiased exponent of a positive normal float (floor(log2 x)).
__device__ __forceinline__ int exponent_of(float x) {
  return (int)((__float_as_uint(x) >> 23) & 0xFF) - 127;
}

}  // namespace codes
}  // namespace kvc
