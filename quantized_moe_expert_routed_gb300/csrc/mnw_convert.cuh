// mnw_convert.cuh -- register-level conversions of the quantised codes into
// tensor-core operands, and 128-byte-swizzle shared-memory helpers.  Shared
// by the tcgen05 kernel (mnw_gemm.cu) and the warp-MMA kernel
// (mnw_gemm_warp.cu).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mnw_ptx.cuh"

namespace mnw {

// ---------------------------------------------------------------------------
// conversions (register level)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t f16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two FP32 lanes in one 64-bit register: d = a * b and d = a * b + c, each
// lane rounded to nearest exactly as the scalar operation (sm_100 family).
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_pack(uint32_t lo, uint32_t hi) {
  return static_cast<uint64_t>(lo) | (static_cast<uint64_t>(hi) << 32);
}

// 32 signed INT4 codes (one 16-byte chunk, element 2c in the low nibble of
// byte c) -> 16 words of (even, odd) pairs holding the integers q exactly, as
// BF16 (kBf16) or FP16.  The group scale is applied later, in FP32.
template <bool kBf16>
__device__ __forceinline__ void cvt_int4x32(const uint4 v, uint32_t (&o)[16]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t hi = w[i] >> 4;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t x = prmt(w[i], hi, 0x0400u + 0x0101u * b);  // byte b: low nibble -> half 0, high -> half 1
      if (kBf16) {
        // 0x4308 ^ n is BF16 128 + (n_signed + 8); subtracting 136 is exact.
        o[i * 4 + b] = bf16x2_sub(and_xor(x, 0x000F000Fu, 0x43084308u), 0x43084308u);
      } else {
        // FP16 1024 + (n_signed + 8) minus 1032.
        o[i * 4 + b] = f16x2_sub(and_xor(x, 0x000F000Fu, 0x64086408u), 0x64086408u);
      }
    }
  }
}

// 32 signed INT8 codes (two 16-byte chunks) -> 16 words holding the integers
// q exactly, as BF16 (kBf16) or FP16.
template <bool kBf16>
__device__ __forceinline__ void cvt_int8x32(const uint4 v0, const uint4 v1, uint32_t (&o)[16]) {
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t u = w[i] ^ 0x80808080u;  // q + 128 per byte
    if (kBf16) {
      float f[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        // 0x4B0000uu is FP32 2^23 + u; minus (2^23 + 128) gives q exactly.
        f[b] = __fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7540u + b)), 8388736.0f);
      }
      o[2 * i] = pack_bf16x2(f[0], f[1]);
      o[2 * i + 1] = pack_bf16x2(f[2], f[3]);
    } else {
      // 0x64uu is FP16 1024 + u; minus 1152 gives q exactly.
      o[2 * i] = f16x2_sub(prmt(u, 0x64646464u, 0x4140u), 0x64806480u);
      o[2 * i + 1] = f16x2_sub(prmt(u, 0x64646464u, 0x4342u), 0x64806480u);
    }
  }
}

// 32 E2M1 codes (one 16-byte chunk) with the E4M3 scales of its two 16-blocks
// -> 16 words of exact FP16 products.
__device__ __forceinline__ void cvt_fp4x32(const uint4 v, uint32_t sf0, uint32_t sf1, uint32_t (&o)[16]) {
  uint32_t s0, s1;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s0) : "h"(static_cast<uint16_t>(sf0 | (sf0 << 8))));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s1) : "h"(static_cast<uint16_t>(sf1 | (sf1 << 8))));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h0, h1, h2, h3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w[i]));
    const uint32_t s = i < 2 ? s0 : s1;
    o[4 * i + 0] = f16x2_mul(h0, s);
    o[4 * i + 1] = f16x2_mul(h1, s);
    o[4 * i + 2] = f16x2_mul(h2, s);
    o[4 * i + 3] = f16x2_mul(h3, s);
  }
}

// Address of 16-byte chunk c of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(uint32_t base, int r, int c) {
  return base + r * 128 + ((c ^ (r & 7)) << 4);
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void stg128(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}


}  // namespace mnw
