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
//   1. CTA (token tile of 16 * kMT, expert tile of 32): 16 warps, each the
//      32-element K chunks c with c % 16 == warp, m16n8k16 BF16 MMAs fed by
//      16-byte loads.  A chunk's K order inside the MMAs is permuted (lane
//      quarter q holds elements 8q..8q+7 of the chunk; the first MMA takes
//      8q..8q+3, the second 8q+4..8q+7), the same permutation on both
//      operands, so each product still pairs x[h] with w[h].  The sixteen
//      partial tiles are summed in shared memory in warp order (a fixed
//      order: the logits are reproducible).
//   2. The last CTA of a token tile to finish (a per-tile arrival counter)
//      takes the top-k of its tokens (one warp per token) and the softmax
//      weights.  Each lane keeps kNE logits (experts lane + 32 i) as
//      order-preserving unsigned keys; one choice is a warp max of the lanes'
//      best keys (redux) and a warp min of the expert indices that hold it.
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

constexpr int kRtTok = 16;                 // tokens per MMA tile (the MMA's M)
constexpr int kRtExp = 32;                 // experts per CTA (four n8 tiles)
constexpr int kRtWarps = 16;               // K chunk phases per CTA
constexpr int kRtThreads = kRtWarps * 32;
constexpr int kRtRow = kRtExp + 4;         // padded row of a partial tile in shared memory (floats)
constexpr int kRtPermB = 8;                // permutation batches per warp in the last CTA
constexpr int kRtPermMax = kRtWarps * kRtPermB * 32;  // 4096 assignments
constexpr int kRtMaxE = 1024;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// An unsigned key with the order of the float (NaN as -inf, -0 as +0); every
// finite or infinite logit maps above 0, the key of "no expert".
__device__ __forceinline__ uint32_t logit_key(float f) {
  if (f != f) f = -INFINITY;
  if (f == 0.f) f = 0.f;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ uint4 ldg_or_zero(const uint4* p, bool ok) {
  return ok ? __ldg(p) : make_uint4(0u, 0u, 0u, 0u);
}

// kMT: 16-token MMA tiles per CTA; kNE: logits per lane in the top-k (E <= 32 kNE).
template <int kMT, int kNE>
__global__ void __launch_bounds__(kRtThreads) route_kernel(const uint4* __restrict__ x, const uint4* __restrict__ wr,
                                                          int T, int H, int E, int k, float* logits, int32_t* ids,
                                                          float* w, int32_t* offsets, int32_t* sorted_assign,
                                                          int32_t* assign_pos, uint32_t* counters, uint32_t* err,
                                                          int fuse_permute, int logits_only) {
  constexpr int kTok = kRtTok * kMT;
  extern __shared__ __align__(16) int32_t rt_smem[];
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t total_valid;
  __shared__ int last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int t0 = blockIdx.x * kTok, e0 = blockIdx.y * kRtExp;
  const int H8 = H / 8;  // 16-byte words per row
  pdl_launch_dependents();
  pdl_wait();

  // ---- 1. logits of kTok tokens x 32 experts, chunks warp, warp + 16, ... ----
  float acc[kMT][4][4];
#pragma unroll
  for (int m = 0; m < kMT; ++m)
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][n][i] = 0.f;
  {
    // (a row past T or an expert past E is never loaded: its pointer is not dereferenced)
    const uint4* xg = x + static_cast<size_t>(t0 + g) * H8 + c;
    const uint4* wg = wr + static_cast<size_t>(e0 + g) * H8 + c;
    bool rv[kMT][2];
#pragma unroll
    for (int m = 0; m < kMT; ++m)
#pragma unroll
      for (int h = 0; h < 2; ++h) rv[m][h] = t0 + m * kRtTok + g + 8 * h < T;
    bool ev[4];
#pragma unroll
    for (int n = 0; n < 4; ++n) ev[n] = e0 + n * 8 + g < E;
    const int nch = H / 32;
    // kMT == 1: two chunks in flight per warp; kMT == 2: one (the registers)
    constexpr int kIn = kMT == 1 ? 2 : 1;
    for (int ch = warp; ch < nch; ch += kRtWarps * kIn) {
      uint4 a[kIn][kMT][2], b[kIn][4];
#pragma unroll
      for (int u = 0; u < kIn; ++u) {
        const int cu = ch + u * kRtWarps;
        const bool ok = cu < nch;
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
          for (int h = 0; h < 2; ++h) a[u][m][h] = ldg_or_zero(xg + (m * kRtTok + 8 * h) * H8 + cu * 4, ok && rv[m][h]);
#pragma unroll
        for (int n = 0; n < 4; ++n) b[u][n] = ldg_or_zero(wg + n * 8 * H8 + cu * 4, ok && ev[n]);
      }
#pragma unroll
      for (int u = 0; u < kIn; ++u) {
        if (ch + u * kRtWarps >= nch) break;
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            mma_bf16_16816(acc[m][n], a[u][m][0].x, a[u][m][1].x, a[u][m][0].y, a[u][m][1].y, b[u][n].x, b[u][n].y);
            mma_bf16_16816(acc[m][n], a[u][m][0].z, a[u][m][1].z, a[u][m][0].w, a[u][m][1].w, b[u][n].z, b[u][n].w);
          }
      }
    }
  }
  // partial tiles -> shared memory [warp][kTok][kRtRow], then a sum in warp order
  float* red = reinterpret_cast<float*>(rt_smem);
  {
    float* p = red + warp * (kTok * kRtRow);
#pragma unroll
    for (int m = 0; m < kMT; ++m)
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int r = m * kRtTok + g, col = n * 8 + 2 * c;
        *reinterpret_cast<float2*>(p + r * kRtRow + col) = make_float2(acc[m][n][0], acc[m][n][1]);
        *reinterpret_cast<float2*>(p + (r + 8) * kRtRow + col) = make_float2(acc[m][n][2], acc[m][n][3]);
      }
  }
  __syncthreads();
  for (int i = tid; i < kTok * kRtExp; i += kRtThreads) {
    const int r = i / kRtExp, col = i % kRtExp;
    float s = red[r * kRtRow + col];
#pragma unroll
    for (int q = 1; q < kRtWarps; ++q) s += red[q * (kTok * kRtRow) + r * kRtRow + col];
    const int t = t0 + r, e = e0 + col;
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
  for (int tl = warp; tl < kTok; tl += kRtWarps) {
    const int t = t0 + tl;
    if (t >= T) break;
    const float* lrow = logits + static_cast<size_t>(t) * E;
    uint32_t key[kNE];
#pragma unroll
    for (int i = 0; i < kNE; ++i) {
      const int e = lane + 32 * i;
      key[i] = e < E ? logit_key(__ldcg(lrow + e)) : 0u;
    }
    uint32_t taken = 0;  // bit i: expert lane + 32 i already chosen
    float l0 = 0.f, den = 0.f, my_p = 0.f;  // lane j keeps choice j
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
      uint32_t bk = 0u;  // this lane's best untaken key, its lowest index on ties
      int bi = 0;
#pragma unroll
      for (int i = 0; i < kNE; ++i) {
        if (!((taken >> i) & 1u) && key[i] > bk) {
          bk = key[i];
          bi = i;
        }
      }
      const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
      const int be = static_cast<int>(__reduce_min_sync(0xffffffffu, bk == mk ? static_cast<uint32_t>(lane + 32 * bi)
                                                                              : 0xffffffffu));
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      const float bv = key_logit(mk);
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

static_assert(kRtTok == 16, "route_counter_bytes assumes at least 16-token tiles");

// Token tiles of 32 from 1024 tokens up: fewer CTAs, each reading a 32 x H
// tile of x against the same 32 x H router rows.
static int route_mt(int T) { return T >= 1024 ? 2 : 1; }

template <int kMT, int kNE>
static cudaError_t launch_route_t(const void* x, const void* wr, int T, int H, int E, int k, float* logits,
                                  int32_t* ids, float* w, int32_t* offsets, int32_t* sorted_assign,
                                  int32_t* assign_pos, uint32_t* counters, uint32_t* err, bool fuse, bool logits_only,
                                  cudaStream_t st) {
  constexpr size_t kRed = static_cast<size_t>(kRtWarps) * kRtTok * kMT * kRtRow * 4;
  constexpr size_t kPermMax = static_cast<size_t>(permute_block_smem_ints(kRtWarps, kRtPermB, kRtMaxE)) * 4;
  const size_t perm_bytes = fuse ? static_cast<size_t>(permute_block_smem_ints(kRtWarps, kRtPermB, E)) * 4 : 0;
  const size_t smem = kRed > perm_bytes ? kRed : perm_bytes;
  static std::atomic<uint64_t> attr{0};
  uint64_t bit;
  if (attrs_needed(attr, &bit)) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel<kMT, kNE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kRed > kPermMax ? kRed : kPermMax));
    if (e != cudaSuccess) return e;
    attrs_done(attr, bit);
  }
  const dim3 grid((T + kRtTok * kMT - 1) / (kRtTok * kMT), (E + kRtExp - 1) / kRtExp);
  return launch_pdl(route_kernel<kMT, kNE>, grid, dim3(kRtThreads), smem, st, static_cast<const uint4*>(x),
                    static_cast<const uint4*>(wr), T, H, E, k, logits, ids, w, offsets, sorted_assign, assign_pos,
                    counters, err, fuse ? 1 : 0, logits_only ? 1 : 0);
}

static cudaError_t launch_route_any(const void* x, const void* wr, int T, int H, int E, int k, float* logits,
                                    int32_t* ids, float* w, int32_t* offsets, int32_t* sorted_assign,
                                    int32_t* assign_pos, uint32_t* counters, uint32_t* err, bool fuse,
                                    bool logits_only, cudaStream_t st) {
  const bool big = route_mt(T) == 2, wide = E > 256;
  if (!big && !wide)
    return launch_route_t<1, 8>(x, wr, T, H, E, k, logits, ids, w, offsets, sorted_assign, assign_pos, counters, err,
                                fuse, logits_only, st);
  if (!big)
    return launch_route_t<1, kRtMaxE / 32>(x, wr, T, H, E, k, logits, ids, w, offsets, sorted_assign, assign_pos,
                                           counters, err, fuse, logits_only, st);
  if (!wide)
    return launch_route_t<2, 8>(x, wr, T, H, E, k, logits, ids, w, offsets, sorted_assign, assign_pos, counters, err,
                                fuse, logits_only, st);
  return launch_route_t<2, kRtMaxE / 32>(x, wr, T, H, E, k, logits, ids, w, offsets, sorted_assign, assign_pos,
                                         counters, err, fuse, logits_only, st);
}

size_t route_scratch_bytes(int T, int E) { return route_counter_bytes(T) + static_cast<size_t>(T) * E * 4; }

bool route_shape_ok(int T, int H, int E, int k) {
  return T >= 0 && H > 0 && H % 128 == 0 && E >= 1 && E <= kRtMaxE && k >= 1 && k <= 32 && k <= E &&
         static_cast<long long>(T) * k <= (1LL << 24);
}

cudaError_t launch_route(const void* x, const void* wr, int T, int H, int E, int k, int32_t* ids, float* w,
                         int32_t* offsets, int32_t* sorted_assign, int32_t* assign_pos, void* scratch, uint32_t* err,
                         cudaStream_t st) {
  uint32_t* counters = static_cast<uint32_t*>(scratch);
  float* logits = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + route_counter_bytes(T));
  const bool fuse = T * k <= kRtPermMax;
  cudaError_t e = launch_route_any(x, wr, T, H, E, k, logits, ids, w, offsets, sorted_assign, assign_pos, counters,
                                   err, fuse, false, st);
  if (e != cudaSuccess || fuse) return e;
  return launch_permute(ids, T, k, E, offsets, sorted_assign, assign_pos, nullptr, 0, nullptr, err, st);
}

cudaError_t launch_route_logits(const void* x, const void* wr, int T, int H, int E, float* logits, cudaStream_t st) {
  return launch_route_any(x, wr, T, H, E, 1, logits, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                          false, true, st);
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
