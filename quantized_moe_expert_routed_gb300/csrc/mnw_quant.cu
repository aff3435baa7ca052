// mnw_quant.cu -- dynamic activation quantisers (bit-exact by construction:
// every step is one IEEE binary32 operation with round-to-nearest-even, and
// the FP8/FP4 roundings use the hardware's rn.satfinite conversions).
//
//  INT8 per 128 ("LLaDA2.2-flash-minnow" model card, W8A8/W4A8 paragraph):
//    scale = amax / 127, code = clamp(rne(x / scale), -127, 127); amax 0 gives
//    scale 0 and codes 0.
//  NVFP4 (model card, NVFP4 row, activation column): outer = amax_row / 2688,
//    sb = e4m3(amax_16 / outer / 6), code = e2m1(x / (sb * outer)).
// Rows of up to 1024 values: one warp per row, the whole row loaded first
// with 16-byte loads (lane l holds 16-byte words l, l + 32, ...), so a warp
// has its row's bytes in flight at once; the group or block maxima are warp
// reductions over the lanes that hold the group.  Longer INT8 rows: chunks of
// up to 512 values, one warp each; longer NVFP4 rows: a two-pass warp per row
// (four or eight warps per row meeting in shared memory for the row's maximum
// measured no faster on the 2048-value rows of the prefill batch).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mnw_internal.h"
#include "mnw_ptx.cuh"

namespace mnw {

__device__ __forceinline__ int source_row(int r, const int32_t* row_index, int index_div) {
  if (!row_index) return r;
  const int a = __ldg(row_index + r);
  return a < 0 ? -1 : a / index_div;
}

// kScatter = false: output row r is the quantised source row source_row(r)
// (R output rows).  kScatter = true: source row r (R source rows, r = token)
// is quantised once and written to output rows assign_pos[r * k + j], j < k,
// that are >= 0 (row_index = assign_pos, index_div = k).
template <bool kScatter>
__global__ void __launch_bounds__(256) quant_int8_g128_kernel(const __nv_bfloat16* __restrict__ x, int R, int K,
                                                              const int32_t* __restrict__ row_index,
                                                              int index_div, int8_t* __restrict__ codes,
                                                              float* __restrict__ scales) {
  pdl_launch_dependents();
  pdl_wait();
  const int G = K / 128;
  const long long total = static_cast<long long>(R) * G;
  const int lane = threadIdx.x & 31;
  for (long long wg = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5); wg < total;
       wg += static_cast<long long>(gridDim.x) * 8) {
    const int r = static_cast<int>(wg / G), g = static_cast<int>(wg % G);
    const int src = kScatter ? r : source_row(r, row_index, index_div);
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (src >= 0) {
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(x + static_cast<size_t>(src) * K + g * 128) + lane);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
      v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    }
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    uint32_t packed = 0;
    float scale = 0.f;
    if (amax > 0.f) {
      scale = __fdiv_rn(amax, 127.0f);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        int q = __float2int_rn(__fdiv_rn(v[i], scale));
        q = max(-127, min(127, q));
        packed |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * i);
      }
    }
    if constexpr (kScatter) {
      for (int j = 0; j < index_div; ++j) {
        const int d = __ldg(row_index + static_cast<size_t>(r) * index_div + j);
        if (d < 0) continue;
        reinterpret_cast<uint32_t*>(codes + static_cast<size_t>(d) * K + g * 128)[lane] = packed;
        if (lane == 0) scales[static_cast<size_t>(d) * G + g] = scale;
      }
    } else {
      reinterpret_cast<uint32_t*>(codes + static_cast<size_t>(r) * K + g * 128)[lane] = packed;
      if (lane == 0) scales[static_cast<size_t>(r) * G + g] = scale;
    }
  }
}

__device__ __forceinline__ uint8_t e4m3_rn_satfinite(float s) {
  uint16_t pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(s));
  return static_cast<uint8_t>(pair & 0xFF);
}
__device__ __forceinline__ float e4m3_to_float(uint8_t b) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(b);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFF)));
}
// Two values to one byte of E2M1 codes: lo in the low nibble, hi in the high one.
__device__ __forceinline__ uint32_t e2m1x2_rn_satfinite(float lo, float hi) {
  uint32_t out;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(out)
      : "f"(hi), "f"(lo));
  return out;
}

// kScatter as for quant_int8_g128_kernel.
template <bool kScatter>
__global__ void __launch_bounds__(256) quant_nvfp4_g16_kernel(const __nv_bfloat16* __restrict__ x, int R, int K,
                                                              const int32_t* __restrict__ row_index,
                                                              int index_div, uint8_t* __restrict__ codes,
                                                              uint8_t* __restrict__ sf, float* __restrict__ outer) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int nb = K / 16;
  for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < R; r += gridDim.x * 8) {
    const int src = kScatter ? r : source_row(r, row_index, index_div);
    const int ndst = kScatter ? index_div : 1;  // output rows this source row goes to
    const __nv_bfloat16* xr = src >= 0 ? x + static_cast<size_t>(src) * K : nullptr;
    // row amax
    float amax = 0.f;
    if (xr) {
      for (int b = lane; b < nb; b += 32) {
        const uint4* p = reinterpret_cast<const uint4*>(xr + b * 16);
        const uint4 q0 = __ldg(p), q1 = __ldg(p + 1);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
          amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    const float o = __fdiv_rn(amax, 2688.0f);
    if (lane == 0) {
      for (int j = 0; j < ndst; ++j) {
        const int d = kScatter ? __ldg(row_index + static_cast<size_t>(r) * index_div + j) : r;
        if (d >= 0) outer[d] = o;
      }
    }
    for (int b = lane; b < nb; b += 32) {
      uint2 packed = make_uint2(0, 0);
      uint8_t sbyte = 0;
      if (xr && o != 0.f) {
        const uint4* p = reinterpret_cast<const uint4*>(xr + b * 16);
        const uint4 q0 = __ldg(p), q1 = __ldg(p + 1);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        float v[16];
        float ab = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
          v[2 * i] = f.x;
          v[2 * i + 1] = f.y;
          ab = fmaxf(ab, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
        sbyte = e4m3_rn_satfinite(__fdiv_rn(__fdiv_rn(ab, o), 6.0f));
        const float d = __fmul_rn(e4m3_to_float(sbyte), o);
        if (d != 0.f) {
          uint32_t lo = 0, hi = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            lo |= e2m1x2_rn_satfinite(__fdiv_rn(v[2 * i], d), __fdiv_rn(v[2 * i + 1], d)) << (8 * i);
            hi |= e2m1x2_rn_satfinite(__fdiv_rn(v[8 + 2 * i], d), __fdiv_rn(v[8 + 2 * i + 1], d)) << (8 * i);
          }
          packed = make_uint2(lo, hi);
        }
      }
      for (int j = 0; j < ndst; ++j) {
        const int d = kScatter ? __ldg(row_index + static_cast<size_t>(r) * index_div + j) : r;
        if (d < 0) continue;
        reinterpret_cast<uint2*>(codes + static_cast<size_t>(d) * (K / 2))[b] = packed;
        sf[static_cast<size_t>(d) * nb + b] = sbyte;
      }
    }
  }
}

// ---- rows of up to 32 * 8 * kU values, one warp per row, held in registers ----

// The destination rows of source row r: lane j < index_div holds
// row_index[r * index_div + j] (kScatter), else only r itself.
template <bool kScatter>
__device__ __forceinline__ int dest_of_lane(int r, const int32_t* row_index, int index_div, int lane) {
  if (!kScatter) return lane == 0 ? r : -1;
  return lane < index_div ? __ldg(row_index + static_cast<size_t>(r) * index_div + lane) : -1;
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& q, float (&v)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// INT8 per 128: a warp takes one chunk of nch per row (Kc = K / nch values, a
// multiple of 128); word i of the chunk (8 values) belongs to the chunk's
// group i / 16, so the lanes of a half-warp hold one group per word slot.
// index_div <= 32 when kScatter.
template <bool kScatter, int kU>
__global__ void __launch_bounds__(256) quant_int8_rows_kernel(const __nv_bfloat16* __restrict__ x, int R, int K,
                                                              int nch, const int32_t* __restrict__ row_index,
                                                              int index_div, int8_t* __restrict__ codes,
                                                              float* __restrict__ scales) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int Kc = K / nch, K8 = Kc / 8, G = K / 128;
  const int items = R * nch;  // (< 2^31: checked by the launcher)
  for (int wi = blockIdx.x * 8 + (threadIdx.x >> 5); wi < items; wi += gridDim.x * 8) {
    const int r = nch == 1 ? wi : wi / nch;
    const int c0 = (wi - r * nch) * Kc;  // the chunk's first value
    const int src = kScatter ? r : source_row(r, row_index, index_div);
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(src < 0 ? 0 : src) * K + c0);
    uint4 raw[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = u * 32 + lane;
      raw[u] = (src >= 0 && i < K8) ? __ldg(xr + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    const int my_dst = dest_of_lane<kScatter>(r, row_index, index_div, lane);
    const int ndst = kScatter ? index_div : 1;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (u * 32 >= K8) break;  // (uniform)
      const int i = u * 32 + lane;
      float v[8];
      bf16x8_to_float(raw[u], v);
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
      for (int d = 8; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
      uint2 packed = make_uint2(0u, 0u);
      float scale = 0.f;
      if (amax > 0.f) {
        scale = __fdiv_rn(amax, 127.0f);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q0 = max(-127, min(127, __float2int_rn(__fdiv_rn(v[e], scale))));
          const int q1 = max(-127, min(127, __float2int_rn(__fdiv_rn(v[4 + e], scale))));
          lo |= (static_cast<uint32_t>(q0) & 0xFFu) << (8 * e);
          hi |= (static_cast<uint32_t>(q1) & 0xFFu) << (8 * e);
        }
        packed = make_uint2(lo, hi);
      }
      const int g = c0 / 128 + (i >> 4);
      for (int j = 0; j < ndst; ++j) {
        const int d = __shfl_sync(0xffffffffu, my_dst, j);
        if (d < 0 || i >= K8) continue;
        reinterpret_cast<uint2*>(codes + static_cast<size_t>(d) * K + c0)[i] = packed;
        if ((lane & 15) == 0) scales[static_cast<size_t>(d) * G + g] = scale;
      }
    }
  }
}

// NVFP4: 16-block b of the row is words 2b, 2b + 1; lane l holds blocks
// l, l + 32, ... (two consecutive words each).  index_div <= 32 when kScatter.
template <bool kScatter, int kU>
__global__ void __launch_bounds__(256) quant_nvfp4_rows_kernel(const __nv_bfloat16* __restrict__ x, int R, int K,
                                                               const int32_t* __restrict__ row_index,
                                                               int index_div, uint8_t* __restrict__ codes,
                                                               uint8_t* __restrict__ sf, float* __restrict__ outer) {
  static_assert(kU % 2 == 0, "two words per block");
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int K8 = K / 8, nb = K / 16;
  for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < R; r += gridDim.x * 8) {
    const int src = kScatter ? r : source_row(r, row_index, index_div);
    const uint4* xr = reinterpret_cast<const uint4*>(x) + static_cast<size_t>(src < 0 ? 0 : src) * K8;
    uint4 raw[kU];
#pragma unroll
    for (int u = 0; u < kU / 2; ++u) {
      const int b = u * 32 + lane;
      const bool ok = src >= 0 && b < nb;
      raw[2 * u] = ok ? __ldg(xr + 2 * b) : make_uint4(0u, 0u, 0u, 0u);
      raw[2 * u + 1] = ok ? __ldg(xr + 2 * b + 1) : make_uint4(0u, 0u, 0u, 0u);
    }
    const int my_dst = dest_of_lane<kScatter>(r, row_index, index_div, lane);
    const int ndst = kScatter ? index_div : 1;
    float bmax[kU / 2];
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < kU / 2; ++u) {
      float v[8], w[8];
      bf16x8_to_float(raw[2 * u], v);
      bf16x8_to_float(raw[2 * u + 1], w);
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fmaxf(fabsf(v[e]), fabsf(w[e])));
      bmax[u] = m;
      amax = fmaxf(amax, m);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    const float o = __fdiv_rn(amax, 2688.0f);
    for (int j = 0; j < ndst; ++j) {
      const int d = __shfl_sync(0xffffffffu, my_dst, j);
      if (d >= 0 && lane == 0) outer[d] = o;
    }
#pragma unroll
    for (int u = 0; u < kU / 2; ++u) {
      if (u * 32 >= nb) break;  // (uniform)
      const int b = u * 32 + lane;
      uint2 packed = make_uint2(0u, 0u);
      uint8_t sbyte = 0;
      if (o != 0.f) {
        float v[16];
        {
          float lo8[8], hi8[8];
          bf16x8_to_float(raw[2 * u], lo8);
          bf16x8_to_float(raw[2 * u + 1], hi8);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            v[e] = lo8[e];
            v[8 + e] = hi8[e];
          }
        }
        sbyte = e4m3_rn_satfinite(__fdiv_rn(__fdiv_rn(bmax[u], o), 6.0f));
        const float dd = __fmul_rn(e4m3_to_float(sbyte), o);
        if (dd != 0.f) {
          uint32_t lo = 0, hi = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            lo |= e2m1x2_rn_satfinite(__fdiv_rn(v[2 * e], dd), __fdiv_rn(v[2 * e + 1], dd)) << (8 * e);
            hi |= e2m1x2_rn_satfinite(__fdiv_rn(v[8 + 2 * e], dd), __fdiv_rn(v[8 + 2 * e + 1], dd)) << (8 * e);
          }
          packed = make_uint2(lo, hi);
        }
      }
      for (int j = 0; j < ndst; ++j) {
        const int d = __shfl_sync(0xffffffffu, my_dst, j);
        if (d < 0 || b >= nb) continue;
        reinterpret_cast<uint2*>(codes + static_cast<size_t>(d) * (K / 2))[b] = packed;
        sf[static_cast<size_t>(d) * nb + b] = sbyte;
      }
    }
  }
}

// 16-byte words per lane for a row of K values (0: the row kernels do not take
// it).  Measured on GB300 (NVFP4, 8192-token prefill): rows of 512 values
// 30.5 -> 27 us with the row kernel; rows of 2048 (8 words a lane, ~90
// registers, 16 warps per SM) 23 -> 29 us, the divisions then wanting more
// warps than the registers leave, so longer rows keep the other kernels.
static int rows_words_per_lane(int K, int index_div, bool scatter) {
  if (scatter && index_div > 32) return 0;
  const int w = (K / 8 + 31) / 32;
  if (w <= 2) return 2;
  if (w <= 4) return 4;
  return 0;
}

// INT8 rows of more than 1024 values are cut into chunks of 512 (or 256, or
// 128) values, one warp each: the groups are independent.
static int int8_chunks(int K) {
  if (K <= 1024) return 1;
  if (K % 512 == 0) return K / 512;
  if (K % 256 == 0) return K / 256;
  return K / 128;
}

// The chunked INT8 kernel counts its (row, chunk) items in 32 bits.
static bool int8_items_fit(int R, int K) { return static_cast<long long>(R) * int8_chunks(K) < (1LL << 31); }

template <bool kScatter>
static cudaError_t launch_quant_rows(int act, int kU, const void* x, int R, int K, const int32_t* row_index,
                                     int index_div, void* codes, void* scales, float* row_outer, cudaStream_t st) {
  const int sms = current_sm_count();
  const int nch = act == MNW_ACT_INT8_G128 ? int8_chunks(K) : 1;
  long long blocks = (static_cast<long long>(R) * nch + 7) / 8;
  if (blocks > static_cast<long long>(sms) * 16) blocks = static_cast<long long>(sms) * 16;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<int>(blocks)), block(256);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  if (act == MNW_ACT_INT8_G128) {
    auto* c = static_cast<int8_t*>(codes);
    auto* sc = static_cast<float*>(scales);
    switch (K / nch <= 512 ? 2 : 4) {  // 16-byte words per lane for a chunk
      case 2: return launch_pdl(quant_int8_rows_kernel<kScatter, 2>, grid, block, 0, st, xb, R, K, nch, row_index, index_div, c, sc);
      default: return launch_pdl(quant_int8_rows_kernel<kScatter, 4>, grid, block, 0, st, xb, R, K, nch, row_index, index_div, c, sc);
    }
  }
  auto* c = static_cast<uint8_t*>(codes);
  auto* sfp = static_cast<uint8_t*>(scales);
  switch (kU) {
    case 2: return launch_pdl(quant_nvfp4_rows_kernel<kScatter, 2>, grid, block, 0, st, xb, R, K, row_index, index_div, c, sfp, row_outer);
    default: return launch_pdl(quant_nvfp4_rows_kernel<kScatter, 4>, grid, block, 0, st, xb, R, K, row_index, index_div, c, sfp, row_outer);
  }
}

cudaError_t launch_quantize(int act, const void* x, int R, int K, const int32_t* row_index, int index_div,
                            void* codes, void* scales, float* row_outer, cudaStream_t st) {
  if (act == MNW_ACT_INT8_G128 && int8_items_fit(R, K))  // (the chunk decides the words per lane)
    return launch_quant_rows<false>(act, 0, x, R, K, row_index, index_div, codes, scales, row_outer, st);
  if (const int kU = rows_words_per_lane(K, index_div, false))
    return launch_quant_rows<false>(act, kU, x, R, K, row_index, index_div, codes, scales, row_outer, st);
  const int sms = current_sm_count();
  if (act == MNW_ACT_INT8_G128) {
    const long long warps = static_cast<long long>(R) * (K / 128);
    long long blocks = (warps + 7) / 8;
    if (blocks > static_cast<long long>(sms) * 16) blocks = static_cast<long long>(sms) * 16;
    if (blocks < 1) blocks = 1;
    return launch_pdl(quant_int8_g128_kernel<false>, dim3(static_cast<int>(blocks)), dim3(256), 0, st,
                      static_cast<const __nv_bfloat16*>(x), R, K, row_index, index_div, static_cast<int8_t*>(codes),
                      static_cast<float*>(scales));
  } else {
    long long blocks = (static_cast<long long>(R) + 7) / 8;
    if (blocks > static_cast<long long>(sms) * 16) blocks = static_cast<long long>(sms) * 16;
    if (blocks < 1) blocks = 1;
    return launch_pdl(quant_nvfp4_g16_kernel<false>, dim3(static_cast<int>(blocks)), dim3(256), 0, st,
                      static_cast<const __nv_bfloat16*>(x), R, K, row_index, index_div, static_cast<uint8_t*>(codes),
                      static_cast<uint8_t*>(scales), row_outer);
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize_scatter(int act, const void* x, int R, int K, const int32_t* row_index, int index_div,
                            void* codes, void* scales, float* row_outer, cudaStream_t st) {
  if (act == MNW_ACT_INT8_G128 && index_div <= 32 && int8_items_fit(R, K))
    return launch_quant_rows<true>(act, 0, x, R, K, row_index, index_div, codes, scales, row_outer, st);
  if (const int kU = rows_words_per_lane(K, index_div, true))
    return launch_quant_rows<true>(act, kU, x, R, K, row_index, index_div, codes, scales, row_outer, st);
  const int sms = current_sm_count();
  if (act == MNW_ACT_INT8_G128) {
    const long long warps = static_cast<long long>(R) * (K / 128);
    long long blocks = (warps + 7) / 8;
    if (blocks > static_cast<long long>(sms) * 16) blocks = static_cast<long long>(sms) * 16;
    if (blocks < 1) blocks = 1;
    return launch_pdl(quant_int8_g128_kernel<true>, dim3(static_cast<int>(blocks)), dim3(256), 0, st,
                      static_cast<const __nv_bfloat16*>(x), R, K, row_index, index_div, static_cast<int8_t*>(codes),
                      static_cast<float*>(scales));
  } else {
    long long blocks = (static_cast<long long>(R) + 7) / 8;
    if (blocks > static_cast<long long>(sms) * 16) blocks = static_cast<long long>(sms) * 16;
    if (blocks < 1) blocks = 1;
    return launch_pdl(quant_nvfp4_g16_kernel<true>, dim3(static_cast<int>(blocks)), dim3(256), 0, st,
                      static_cast<const __nv_bfloat16*>(x), R, K, row_index, index_div, static_cast<uint8_t*>(codes),
                      static_cast<uint8_t*>(scales), row_outer);
  }
  return cudaGetLastError();
}

}  // namespace mnw
