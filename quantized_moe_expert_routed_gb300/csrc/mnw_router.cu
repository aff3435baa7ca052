// mnw_router.cu -- GPU routing of the decode path, fused with the permutation.
//
// The "coder543/minnow" README, section "Quantization", routes the tokens of
// the 32-token decode blocks on the GPU, and the "LLaDA2.2-flash-minnow" model
// card ("Checkpoints and precision") keeps the router in its source floating
// point (BF16).  The pages give no formula; this library's reading:
//   logits[t, e] = x[t] . wr[e]                   (BF16 inputs, FP32 accumulation)
//   ids[t, 0..k) = the k largest logits, largest first; on equal logits the
//                  lower expert index first
//   w[t, j]      = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k chosen
// followed by the same stable permutation as mnw_moe_permute.
//
// One launch, three phases, no CTA ever waits for another:
//   1. CTA (token tile of 16, expert tile of 32): 8 warps, each one eighth of
//      H, m16n8k16 BF16 MMAs; the eight partial tiles are summed in shared
//      memory in warp order (a fixed order: the logits are reproducible).
//   2. The last CTA of a token tile to finish (a per-tile arrival counter)
//      takes the top-k of its 16 tokens (one warp per two tokens) and the
//      softmax weights.
//   3. The last token tile to finish (a global arrival counter) permutes all
//      T*k ids in place with the one-CTA permutation, when they fit one CTA
//      (T*k <= 4096); larger batches get the permutation kernels after this
//      launch.
// Every counter is left at zero by its last arrival.  Writes before an arrival
// are fenced (__threadfence) and the last arrival reads them through L2.
#include <cuda_bf16.h>

#include <atomic>
#include <cfloat>
#include <climits>
#include <cmath>

#include "mnw_internal.h"
#include "mnw_permute.cuh"
#include "mnw_ptx.cuh"

namespace mnw {

constexpr int kRtTok = 16;                 // tokens per CTA (the MMA's M)
constexpr int kRtExp = 32;                 // experts per CTA (four n8 tiles)
constexpr int kRtWarps = 8;                // K slices per CTA
constexpr int kRtThreads = kRtWarps * 32;
constexpr int kRtPermB = 16;               // permutation batches per warp in the last CTA
constexpr int kRtPermMax = kRtWarps * kRtPermB * 32;  // 4096 assignments
constexpr int kRtMaxE = 1024;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kRtThreads) route_kernel(const uint32_t* __restrict__ x, const uint32_t* __restrict__ wr,
                                                          int T, int H, int E, int k, float* logits, int32_t* ids,
                                                          float* w, int32_t* offsets, int32_t* sorted_assign,
                                                          int32_t* assign_pos, uint32_t* counters, uint32_t* err,
                                                          int fuse_permute, int logits_only) {
  extern __shared__ __align__(16) int32_t rt_smem[];
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t total_valid;
  __shared__ int last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int t0 = blockIdx.x * kRtTok, e0 = blockIdx.y * kRtExp;
  const int H2 = H / 2;  // 32-bit words (BF16 pairs) per row
  pdl_launch_dependents();
  pdl_wait();

  // ---- 1. logits of 16 tokens x 32 experts, K slice `warp` ----
  float acc[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;
  {
    const int kw = H / kRtWarps;  // a multiple of 16
    const int kb = warp * kw;
    const bool r0 = t0 + g < T, r1 = t0 + g + 8 < T;
    const uint32_t* xa = x + static_cast<size_t>(min(t0 + g, T - 1)) * H2;
    const uint32_t* xb = x + static_cast<size_t>(min(t0 + g + 8, T - 1)) * H2;
    const uint32_t* wb[4];
    bool ev[4];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const int e = e0 + n * 8 + g;
      ev[n] = e < E;
      wb[n] = wr + static_cast<size_t>(min(e, E - 1)) * H2;
    }
#pragma unroll 4
    for (int kk = kb; kk < kb + kw; kk += 16) {
      const int w0 = kk / 2 + c, w1 = w0 + 4;
      uint32_t a[4];
      a[0] = r0 ? __ldg(xa + w0) : 0u;
      a[1] = r1 ? __ldg(xb + w0) : 0u;
      a[2] = r0 ? __ldg(xa + w1) : 0u;
      a[3] = r1 ? __ldg(xb + w1) : 0u;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const uint32_t b0 = ev[n] ? __ldg(wb[n] + w0) : 0u;
        const uint32_t b1 = ev[n] ? __ldg(wb[n] + w1) : 0u;
        mma_bf16_16816(acc[n], a, b0, b1);
      }
    }
  }
  // partial tiles -> shared memory [warp][16][32], then a sum in warp order
  float* red = reinterpret_cast<float*>(rt_smem);
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    float* p = red + warp * (kRtTok * kRtExp);
    p[g * kRtExp + n * 8 + 2 * c] = acc[n][0];
    p[g * kRtExp + n * 8 + 2 * c + 1] = acc[n][1];
    p[(g + 8) * kRtExp + n * 8 + 2 * c] = acc[n][2];
    p[(g + 8) * kRtExp + n * 8 + 2 * c + 1] = acc[n][3];
  }
  __syncthreads();
  for (int i = tid; i < kRtTok * kRtExp; i += kRtThreads) {
    float s = red[i];
#pragma unroll
    for (int q = 1; q < kRtWarps; ++q) s += red[q * (kRtTok * kRtExp) + i];
    const int t = t0 + i / kRtExp, e = e0 + i % kRtExp;
    if (t < T && e < E) logits[static_cast<size_t>(t) * E + e] = s;
  }

  if (logits_only) return;  // host routing: the host picks the experts

  // ---- 2. the last expert tile of this token tile picks the top-k ----
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(counters + 1 + blockIdx.x, 1u) == gridDim.y - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (tid == 0) counters[1 + blockIdx.x] = 0;
  for (int tl = warp; tl < kRtTok; tl += kRtWarps) {
    const int t = t0 + tl;
    if (t >= T) break;
    const float* lrow = logits + static_cast<size_t>(t) * E;
    float v[kRtMaxE / 32];
    uint32_t taken = 0;  // bit i: expert lane + 32 i already chosen
#pragma unroll
    for (int i = 0; i < kRtMaxE / 32; ++i) {
      const int e = lane + 32 * i;
      float f = e < E ? __ldcg(lrow + e) : -INFINITY;
      v[i] = f != f ? -INFINITY : f;  // a NaN logit ranks last
    }
    float l0 = 0.f, den = 0.f, my_p = 0.f;  // lane j keeps choice j
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = INT_MAX;
#pragma unroll
      for (int i = 0; i < kRtMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
        const int oe = __shfl_xor_sync(0xffffffffu, be, d);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (j == 0) l0 = bv;
      const float p = bv == l0 ? 1.f : expf(bv - l0);  // (equal infinite logits: equal weights)
      den += p;
      if (lane == j) {
        my_id = be;
        my_p = p;
      }
    }
    if (lane < k) {
      ids[static_cast<size_t>(t) * k + lane] = my_id;
      w[static_cast<size_t>(t) * k + lane] = my_p / den;
    }
  }

  // ---- 3. the last token tile permutes all T*k assignments ----
  if (!fuse_permute) return;
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(counters, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (tid == 0) counters[0] = 0;
  permute_block<kRtWarps, kRtPermB>(ids, T * k, E, offsets, sorted_assign, assign_pos, err, rt_smem, warp_tot,
                                    &total_valid);
}

static_assert(kRtTok == 16, "route_counter_bytes assumes 16-token tiles");

size_t route_scratch_bytes(int T, int E) { return route_counter_bytes(T) + static_cast<size_t>(T) * E * 4; }

bool route_shape_ok(int T, int H, int E, int k) {
  return T >= 0 && H > 0 && H % 128 == 0 && E >= 1 && E <= kRtMaxE && k >= 1 && k <= 32 && k <= E &&
         static_cast<long long>(T) * k <= (1LL << 24);
}

cudaError_t launch_route(const void* x, const void* wr, int T, int H, int E, int k, int32_t* ids, float* w,
                         int32_t* offsets, int32_t* sorted_assign, int32_t* assign_pos, void* scratch, uint32_t* err,
                         cudaStream_t st) {
  const int tiles = (T + kRtTok - 1) / kRtTok;
  uint32_t* counters = static_cast<uint32_t*>(scratch);
  float* logits = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + route_counter_bytes(T));
  const bool fuse = T * k <= kRtPermMax;
  const size_t red_bytes = static_cast<size_t>(kRtWarps) * kRtTok * kRtExp * 4;
  const size_t perm_bytes = fuse ? static_cast<size_t>(kRtWarps + 1) * E * 4 : 0;
  const size_t smem = red_bytes > perm_bytes ? red_bytes : perm_bytes;
  static std::atomic<uint64_t> attr{0};
  uint64_t bit;
  if (attrs_needed(attr, &bit)) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>((kRtWarps + 1) * kRtMaxE * 4));
    if (e != cudaSuccess) return e;
    attrs_done(attr, bit);
  }
  const dim3 grid(tiles, (E + kRtExp - 1) / kRtExp);
  cudaError_t e = launch_pdl(route_kernel, grid, dim3(kRtThreads), smem, st, static_cast<const uint32_t*>(x),
                             static_cast<const uint32_t*>(wr), T, H, E, k, logits, ids, w, offsets, sorted_assign,
                             assign_pos, counters, err, fuse ? 1 : 0, 0);
  if (e != cudaSuccess || fuse) return e;
  return launch_permute(ids, T, k, E, offsets, sorted_assign, assign_pos, nullptr, 0, nullptr, err, st);
}

cudaError_t launch_route_logits(const void* x, const void* wr, int T, int H, int E, float* logits, cudaStream_t st) {
  const int tiles = (T + kRtTok - 1) / kRtTok;
  const size_t smem = static_cast<size_t>(kRtWarps) * kRtTok * kRtExp * 4;
  return launch_pdl(route_kernel, dim3(tiles, (E + kRtExp - 1) / kRtExp), dim3(kRtThreads), smem, st,
                    static_cast<const uint32_t*>(x), static_cast<const uint32_t*>(wr), T, H, E, 1, logits,
                    static_cast<int32_t*>(nullptr), static_cast<float*>(nullptr), static_cast<int32_t*>(nullptr),
                    static_cast<int32_t*>(nullptr), static_cast<int32_t*>(nullptr), static_cast<uint32_t*>(nullptr),
                    static_cast<uint32_t*>(nullptr), 0, 1);
}

void route_topk_host(const float* logits, int T, int E, int k, int32_t* ids, float* w) {
  for (int t = 0; t < T; ++t) {
    const float* l = logits + static_cast<size_t>(t) * E;
    uint64_t taken[kRtMaxE / 64] = {};
    float l0 = 0.f, den = 0.f;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = -1;
      for (int e = 0; e < E; ++e) {
        if ((taken[e >> 6] >> (e & 63)) & 1u) continue;
        const float v = l[e] != l[e] ? -INFINITY : l[e];  // a NaN logit ranks last
        if (be < 0 || v > bv) {
          bv = v;
          be = e;
        }
      }
      taken[be >> 6] |= 1ull << (be & 63);
      if (j == 0) l0 = bv;
      const float p = bv == l0 ? 1.f : std::exp(bv - l0);
      den += p;
      ids[static_cast<size_t>(t) * k + j] = be;
      w[static_cast<size_t>(t) * k + j] = p;
    }
    for (int j = 0; j < k; ++j) w[static_cast<size_t>(t) * k + j] /= den;
  }
}

}  // namespace mnw
