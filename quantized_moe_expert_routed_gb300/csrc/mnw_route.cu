// mnw_route.cu -- token permutation into expert-sorted order, the row gather,
// and the top-k weighted combine.
//
// Permutation (the grouping by expert that the "coder543/minnow" README,
// section "Quantization", runs on the GPU for decode blocks): a single CTA
// ranks every assignment a = t*k + j
// stably within its expert, with no atomics whose order could leak into the
// result.  Each of the 32 warps owns a contiguous segment of assignments; a
// first pass counts per (warp, expert) with warp match-any groups, a scan over
// (expert, warp) turns counts into starting positions, and a second pass
// re-walks the segment in order, ranking lanes that share an expert by lane
// index.  Each warp reads its ids with 16-byte loads (four consecutive ids a
// lane) into a window of shared memory and takes them back in lane order
// (load_ids in mnw_permute.cuh); ids off a 16-byte boundary fall back to
// 4-byte loads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mnw_internal.h"
#include "mnw_permute.cuh"
#include "mnw_ptx.cuh"

namespace mnw {

constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;
constexpr int kPermBatchesInFlight = 8;  // id loads issued ahead per lane

__global__ void __launch_bounds__(kPermThreads, 1)
    permute_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ offsets,
                   int32_t* __restrict__ sorted_assign, int32_t* __restrict__ assign_pos,
                   uint32_t* __restrict__ err) {
  extern __shared__ __align__(16) int32_t sm[];
  int32_t* cnt = sm;                       // [kPermWarps][E]: counts, then next position
  int32_t* tot = sm + kPermWarps * E;      // [E]
  __shared__ int32_t warp_tot[kPermWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();

  for (int i = tid; i < kPermWarps * E; i += kPermThreads) cnt[i] = 0;
  pdl_wait();
  for (int a = tid; a < P; a += kPermThreads) sorted_assign[a] = -1;
  __syncthreads();

  // segments of a multiple of 4 assignments: each starts on a 16-byte boundary of ids
  const int seg = ((P + kPermWarps - 1) / kPermWarps + 3) & ~3;
  const int a0 = min(P, warp * seg), a1 = min(P, a0 + seg);
  int32_t* my = cnt + warp * E;
  int32_t* win = sm + ids_window_base((kPermWarps + 1) * E) + warp * 32 * kPermBatchesInFlight;

  // Pass 1: per-warp counts.
  for (int base = a0; base < a1; base += 32 * kPermBatchesInFlight) {
    int idv[kPermBatchesInFlight];
    load_ids<kPermBatchesInFlight>(ids, base, min(a1, base + 32 * kPermBatchesInFlight), win, idv);
#pragma unroll
    for (int b = 0; b < kPermBatchesInFlight; ++b) {
      const int a = base + b * 32 + lane;
      const bool active = a < a1;
      const int id = idv[b];
      const bool valid = active && id >= 0 && id < E;
      if (active && !valid && err) atomicOr(err, MNW_DEVERR_BAD_EXPERT_ID);
      const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t peers = __match_any_sync(vmask, id);
        if (lane == __ffs(peers) - 1) my[id] += __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();

  // Exclusive prefix over warps for every expert; totals per expert.
  for (int e = tid; e < E; e += kPermThreads) {
    int run = 0;
    for (int w = 0; w < kPermWarps; ++w) {
      const int c = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();

  // Exclusive scan of the totals over experts (E <= kPermThreads).
  const int v = tid < E ? tot[tid] : 0;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
    int ti = t;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, ti, d);
      if (lane >= d) ti += o;
    }
    warp_tot[lane] = ti - t;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const int excl = incl - v + warp_tot[warp];
  if (tid < E) {
    offsets[tid] = excl;
    tot[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + v;
  }
  __syncthreads();
  for (int i = tid; i < kPermWarps * E; i += kPermThreads) cnt[i] += tot[i % E];
  __syncthreads();

  // Pass 2: stable positions.
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int base = a0; base < a1; base += 32 * kPermBatchesInFlight) {
    int idv[kPermBatchesInFlight];
    load_ids<kPermBatchesInFlight>(ids, base, min(a1, base + 32 * kPermBatchesInFlight), win, idv);
#pragma unroll
    for (int b = 0; b < kPermBatchesInFlight; ++b) {
      const int a = base + b * 32 + lane;
      const bool active = a < a1;
      const int id = idv[b];
      const bool valid = active && id >= 0 && id < E;
      const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
      uint32_t peers = 0;
      if (valid) {
        peers = __match_any_sync(vmask, id);
        const int pos = my[id] + __popc(peers & lt_mask);
        assign_pos[a] = pos;
        sorted_assign[pos] = a;
      } else if (active) {
        assign_pos[a] = -1;
      }
      __syncwarp();
      if (valid && lane == __ffs(peers) - 1) my[id] += __popc(peers);
      __syncwarp();
    }
  }
}

// The same stable permutation for batches of at most kW * kB * 32
// assignments (a decode batch: 256 tokens x top-8 = 2048): see permute_block.
template <int kW, int kB>
__global__ void __launch_bounds__(kW * 32, 1)
    permute_small_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ sorted_assign, int32_t* __restrict__ assign_pos,
                         uint32_t* __restrict__ err) {
  extern __shared__ __align__(16) int32_t sm[];
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t total_valid;
  pdl_launch_dependents();
  pdl_wait();
  permute_block<kW, kB>(ids, P, E, offsets, sorted_assign, assign_pos, err, sm, warp_tot, &total_valid);
}

// ---------------------------------------------------------------------------
// Large batches: the same stable permutation over many CTAs, in three kernels.
// CTA c owns the contiguous chunk [c*kChunk, (c+1)*kChunk) of assignments.
//   count : per-expert counts of the chunk  -> assign_pos[c*kChunk + e]
//   scan  : one CTA turns them into, per (c, e), the first position of chunk
//           c's assignments to expert e (experts in order, chunks in order
//           within an expert), written back in place, plus expert_offsets
//   place : each CTA re-ranks its chunk and writes positions
// The chunk's own slice of assign_pos is the scratch for its counts and
// starts (kChunk >= E), and only that CTA overwrites it in the last pass, so
// no other memory is needed.
constexpr int kChunk = 1024;        // assignments per CTA (>= E)
constexpr int kChunkThreads = 256;  // 8 warps, 4 batches of 32 per warp

// Per-warp stable ranks of one chunk: ids in registers, counts in cnt[8][E].
struct ChunkIds {
  int id[4];
  uint32_t peers[4];
};
// win: this warp's window of 128 ints of shared memory (16-byte aligned).
__device__ __forceinline__ void chunk_count(const int32_t* ids, int a0, int a1, int E, int32_t* cnt, int32_t* win,
                                            ChunkIds& c, uint32_t* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* my = cnt + warp * E;
  const int w0 = a0 + warp * 128;  // this warp's 128 assignments
  load_ids<4>(ids, w0, max(w0, min(a1, w0 + 128)), win, c.id);
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int a = a0 + (warp * 4 + b) * 32 + lane;
    const bool active = a < a1;
    const bool valid = active && c.id[b] >= 0 && c.id[b] < E;
    if (active && !valid && err) atomicOr(err, MNW_DEVERR_BAD_EXPERT_ID);
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
    c.peers[b] = valid ? __match_any_sync(vmask, c.id[b]) : 0u;
    if (valid && lane == __ffs(c.peers[b]) - 1) my[c.id[b]] += __popc(c.peers[b]);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kChunkThreads) permute_count_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                                      int32_t* __restrict__ assign_pos,
                                                                      uint32_t* __restrict__ err) {
  extern __shared__ __align__(16) int32_t sm[];
  int32_t* cnt = sm;  // [8][E]
  pdl_launch_dependents();
  for (int i = threadIdx.x; i < 8 * E; i += kChunkThreads) cnt[i] = 0;
  pdl_wait();
  __syncthreads();
  const int a0 = blockIdx.x * kChunk, a1 = min(P, a0 + kChunk);
  ChunkIds c;
  chunk_count(ids, a0, a1, E, cnt, sm + ids_window_base(8 * E) + (threadIdx.x >> 5) * 128, c, err);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kChunkThreads) {
    int t = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += cnt[w * E + e];
    assign_pos[a0 + e] = t;
  }
}

// One CTA of 1024 threads; C * E counts fit in shared memory (checked by the launcher).
__global__ void __launch_bounds__(1024, 1) permute_scan_kernel(int C, int E, int32_t* __restrict__ assign_pos,
                                                               int32_t* __restrict__ offsets) {
  extern __shared__ __align__(16) int32_t sm[];
  int32_t* cnt = sm;          // [C][E]
  int32_t* tot = sm + C * E;  // [E]
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();
  pdl_wait();
  // the counts come from L2: eight loads in flight per thread, then the stores
  for (int i0 = tid; i0 < C * E; i0 += 8 * 1024) {
    int v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * 1024;
      const int c = i / E, e = i - c * E;
      v[u] = i < C * E ? assign_pos[c * kChunk + e] : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (i0 + u * 1024 < C * E) cnt[i0 + u * 1024] = v[u];
  }
  __syncthreads();
  for (int e = tid; e < E; e += 1024) {
    int run = 0;
    for (int c = 0; c < C; ++c) {
      const int v = cnt[c * E + e];
      cnt[c * E + e] = run;
      run += v;
    }
    tot[e] = run;
  }
  __syncthreads();
  // exclusive scan of the totals (E <= 1024: one expert per thread)
  const int v = tid < E ? tot[tid] : 0;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int t = warp_tot[lane];
    int ti = t;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, ti, d);
      if (lane >= d) ti += o;
    }
    warp_tot[lane] = ti - t;
  }
  __syncthreads();
  const int excl = incl - v + warp_tot[warp];
  if (tid < E) {
    offsets[tid] = excl;
    tot[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + v;
  }
  __syncthreads();
  for (int i = tid; i < C * E; i += 1024) {
    const int c = i / E, e = i - c * E;
    assign_pos[c * kChunk + e] = tot[e] + cnt[i];
  }
}

__global__ void __launch_bounds__(kChunkThreads) permute_place_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                                      const int32_t* __restrict__ offsets,
                                                                      int32_t* __restrict__ sorted_assign,
                                                                      int32_t* __restrict__ assign_pos) {
  extern __shared__ __align__(16) int32_t sm[];
  int32_t* cnt = sm;          // [8][E]: counts, then start of each warp's run
  int32_t* base = sm + 8 * E;  // [E]: first position of this chunk's assignments per expert
  pdl_launch_dependents();
  for (int i = threadIdx.x; i < 8 * E; i += kChunkThreads) cnt[i] = 0;
  pdl_wait();
  const int a0 = blockIdx.x * kChunk, a1 = min(P, a0 + kChunk);
  for (int e = threadIdx.x; e < E; e += kChunkThreads) base[e] = assign_pos[a0 + e];
  __syncthreads();  // starts read before this chunk's positions overwrite them
  ChunkIds c;
  chunk_count(ids, a0, a1, E, cnt, sm + ids_window_base(9 * E) + (threadIdx.x >> 5) * 128, c, nullptr);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kChunkThreads) {
    int run = base[e];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int v = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;
  int32_t* my = cnt + warp * E;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int a = a0 + (warp * 4 + b) * 32 + lane;
    const bool active = a < a1;
    if (c.peers[b] != 0u) {
      const int pos = my[c.id[b]] + __popc(c.peers[b] & lt_mask);
      assign_pos[a] = pos;
      sorted_assign[pos] = a;
    } else if (active) {
      assign_pos[a] = -1;
    }
    __syncwarp();
    if (c.peers[b] != 0u && lane == __ffs(c.peers[b]) - 1) my[c.id[b]] += __popc(c.peers[b]);
    __syncwarp();
  }
  // the tail of dropped assignments
  const int total = __ldg(offsets + E);
  const int per = (P - total + gridDim.x - 1) / gridDim.x;
  const int t0 = total + blockIdx.x * per, t1 = min(P, t0 + per);
  for (int p = t0 + threadIdx.x; p < t1; p += kChunkThreads) sorted_assign[p] = -1;
}

// x_perm[p] = x[sorted_assign[p] / k], zeros where sorted_assign[p] < 0.  One
// warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, int H8,
                                                          const int32_t* __restrict__ sorted_assign, int P,
                                                          int k, uint4* __restrict__ x_perm) {
  pdl_launch_dependents();
  pdl_wait();
  const int warps = gridDim.x * 8;
  for (int p = blockIdx.x * 8 + (threadIdx.x >> 5); p < P; p += warps) {
    const int a = __ldg(sorted_assign + p);
    uint4* dst = x_perm + static_cast<size_t>(p) * H8;
    if (a < 0) {
      for (int c = threadIdx.x & 31; c < H8; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* src = x + static_cast<size_t>(a / k) * H8;
    for (int c = threadIdx.x & 31; c < H8; c += 32) dst[c] = __ldg(src + c);
  }
}

// FP16 rows with a power-of-two row factor, the operand form of the FP16
// gate/up GEMM: row p reads x[src] with src = row_index[p] / div (src = p
// without row_index), writes x_perm[p] = fp16_rn(x[src] * 2^-e_p) and
// factor[p] = 2^e_p, e_p = clamp(floor(log2 amax) - 14, -110, 113).  The
// largest magnitude lands in [2^14, 2^15); FP16 holds every BF16 value of the
// row no more than 2^28 below it exactly, so the GEMM sees the activations
// unchanged up to the factor its epilogue multiplies back.  A negative
// row_index gives a zero row with factor 1.  One warp per row.
__global__ void __launch_bounds__(256) gather_rows_f16_kernel(const uint4* __restrict__ x, int H8,
                                                              const int32_t* __restrict__ row_index, int P,
                                                              int div, uint4* __restrict__ x_perm,
                                                              float* __restrict__ factor) {
  pdl_launch_dependents();
  pdl_wait();
  const int warps = gridDim.x * 8, lane = threadIdx.x & 31;
  for (int p = blockIdx.x * 8 + (threadIdx.x >> 5); p < P; p += warps) {
    const int a = row_index ? __ldg(row_index + p) : p;
    uint4* dst = x_perm + static_cast<size_t>(p) * H8;
    if (a < 0) {
      for (int c = lane; c < H8; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
      if (lane == 0) factor[p] = 1.f;
      continue;
    }
    const uint4* src = x + static_cast<size_t>(a / div) * H8;
    uint32_t m = 0;  // largest |x| as BF16 bits (magnitudes order like their bit patterns)
    for (int c = lane; c < H8; c += 32) {
      const uint4 v = __ldg(src + c);
      m = max(m, max(max(v.x & 0x7FFFu, v.x >> 16 & 0x7FFFu), max(v.y & 0x7FFFu, v.y >> 16 & 0x7FFFu)));
      m = max(m, max(max(v.z & 0x7FFFu, v.z >> 16 & 0x7FFFu), max(v.w & 0x7FFFu, v.w >> 16 & 0x7FFFu)));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
    // floor(log2 amax) - 14: the row's largest magnitude lands in [2^14, 2^15),
    // away from both FP16 overflow and FP16 subnormals.  Clamped so that 2^e
    // and 2^-e are normal FP32 numbers (an all-zero row gets e = -110; the
    // largest finite BF16 needs 113).
    const int e = min(113, max(-110, static_cast<int>(m >> 7) - 141));
    const float down = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    for (int c = lane; c < H8; c += 32) {
      const uint4 v = __ldg(src + c);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = __uint_as_float(wv[q] << 16) * down, hi = __uint_as_float(wv[q] & 0xFFFF0000u) * down;
        __half2 h = __floats2half2_rn(lo, hi);
        o[q] = *reinterpret_cast<uint32_t*>(&h);
      }
      dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (lane == 0) factor[p] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
  }
}

// out[t] = bf16(sum_j w[t, j] * y[assign_pos[t*k + j]]), FP32, j ascending.
// One thread per (token, 8 columns); the k row loads of a thread are issued
// before any of them is consumed (up to 8 in flight), so the kernel runs at
// memory rate even for a 256-token decode batch.
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ y,
                                                      const int32_t* __restrict__ assign_pos,
                                                      const float* __restrict__ w, int T, int k, int H8,
                                                      uint4* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const long long total = static_cast<long long>(T) * H8;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / H8), c = static_cast<int>(i - static_cast<long long>(t) * H8);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint4 v[8];
      float wj[8];
      bool use[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = j0 + jj;
        const int p = j < k ? __ldg(assign_pos + static_cast<size_t>(t) * k + j) : -1;
        use[jj] = p >= 0;
        wj[jj] = use[jj] ? __ldg(w + static_cast<size_t>(t) * k + j) : 0.f;
        v[jj] = use[jj] ? __ldg(y + static_cast<size_t>(p) * H8 + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        if (!use[jj]) continue;
        const uint32_t vv[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vv[q]));
          acc[2 * q] = __fmaf_rn(wj[jj], f.x, acc[2 * q]);
          acc[2 * q + 1] = __fmaf_rn(wj[jj], f.y, acc[2 * q + 1]);
        }
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 bb = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      o[q] = *reinterpret_cast<uint32_t*>(&bb);
    }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// permute_kernel: count tables for E experts, then one id window per warp.
static size_t perm_kernel_smem(int E) {
  return (static_cast<size_t>(ids_window_base((kPermWarps + 1) * E)) + kPermWarps * 32 * kPermBatchesInFlight) *
         sizeof(int32_t);
}

static int grid_for(int rows_per_block, int n, int cap) {
  int g = (n + rows_per_block - 1) / rows_per_block;
  return g < 1 ? 1 : (g > cap ? cap : g);
}

cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets, int32_t* sorted_assign,
                           int32_t* assign_pos, const void* x, int H, void* x_perm, uint32_t* err,
                           cudaStream_t st) {
  const int P = T * k;
  static std::atomic<uint64_t> attr{0};
  uint64_t bit;
  if (attrs_needed(attr, &bit)) {
    // tables for up to E = 1024 experts
    cudaError_t e = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(perm_kernel_smem(1024)));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(permute_small_kernel<16, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(permute_block_smem_ints(16, 16, 1024) * sizeof(int32_t)));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(permute_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>((48 * 1024) * sizeof(int32_t)));
    if (e != cudaSuccess) return e;
    attrs_done(attr, bit);
  }
  cudaError_t e;
  if (P <= 8 * 8 * 32) {
    e = launch_pdl(permute_small_kernel<8, 8>, dim3(1), dim3(8 * 32),
                   static_cast<size_t>(permute_block_smem_ints(8, 8, E)) * sizeof(int32_t), st, ids, P, E, offsets,
                   sorted_assign, assign_pos, err);
  } else if (P <= 16 * 16 * 32) {
    e = launch_pdl(permute_small_kernel<16, 16>, dim3(1), dim3(16 * 32),
                   static_cast<size_t>(permute_block_smem_ints(16, 16, E)) * sizeof(int32_t), st, ids, P, E, offsets,
                   sorted_assign, assign_pos, err);
  } else if (static_cast<long long>((P + kChunk - 1) / kChunk) * E + E <= 48 * 1024 && E <= kChunk &&
             (P % kChunk == 0 || P % kChunk >= E)) {
    // (every chunk, the last included, has room for its E counts in its own slice)
    // many CTAs: count, scan (counts of all chunks in shared memory), place
    const int C = (P + kChunk - 1) / kChunk;
    const size_t chunk_smem = (static_cast<size_t>(ids_window_base(9 * E)) + 8 * 128) * sizeof(int32_t);
    const size_t scan_smem = (static_cast<size_t>(C) * E + E) * sizeof(int32_t);
    e = launch_pdl(permute_count_kernel, dim3(C), dim3(kChunkThreads), chunk_smem, st, ids, P, E, assign_pos, err);
    if (e == cudaSuccess)
      e = launch_pdl(permute_scan_kernel, dim3(1), dim3(1024), scan_smem, st, C, E, assign_pos, offsets);
    if (e == cudaSuccess)
      e = launch_pdl(permute_place_kernel, dim3(C), dim3(kChunkThreads), chunk_smem, st, ids, P, E,
                     static_cast<const int32_t*>(offsets), sorted_assign, assign_pos);
  } else {
    e = launch_pdl(permute_kernel, dim3(1), dim3(kPermThreads), perm_kernel_smem(E), st, ids, P, E, offsets,
                   sorted_assign, assign_pos, err);
  }
  if (e != cudaSuccess) return e;
  if (x && x_perm && P > 0) e = launch_gather_rows(x, H, sorted_assign, P, k, x_perm, st);
  return e;
}

cudaError_t launch_gather_rows(const void* x, int H, const int32_t* sorted_assign, int P, int k, void* x_perm,
                               cudaStream_t st) {
  const int sms = current_sm_count();
  return launch_pdl(gather_rows_kernel, dim3(grid_for(8, P, sms * 8)), dim3(256), 0, st, static_cast<const uint4*>(x),
                    H / 8, sorted_assign, P, k, static_cast<uint4*>(x_perm));
}

// The activation of the unfused comparison path: h = bf16(SiLU(g) * u) from
// BF16 g and u (the same FP32 expression as the fused epilogues), 8 values
// per thread.
__global__ void __launch_bounds__(256) silu_mul_kernel(const uint4* __restrict__ g, const uint4* __restrict__ u,
                                                       size_t n8, uint4* __restrict__ h) {
  pdl_launch_dependents();
  pdl_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 gv = __ldg(g + i), uv = __ldg(u + i);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float r[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float a = __uint_as_float(e ? (gw[j] & 0xFFFF0000u) : (gw[j] << 16));
        const float b = __uint_as_float(e ? (uw[j] & 0xFFFF0000u) : (uw[j] << 16));
        r[e] = __fdividef(a, 1.f + __expf(-a)) * b;
      }
      __nv_bfloat162 p = __floats2bfloat162_rn(r[0], r[1]);
      o[j] = *reinterpret_cast<uint32_t*>(&p);
    }
    h[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_silu_mul(const void* g, const void* u, size_t n, void* h, cudaStream_t st) {
  const int sms = current_sm_count();
  const size_t n8 = n / 8;
  const int blocks = static_cast<int>(std::min<size_t>((n8 + 255) / 256, static_cast<size_t>(sms) * 8));
  return launch_pdl(silu_mul_kernel, dim3(blocks < 1 ? 1 : blocks), dim3(256), 0, st, static_cast<const uint4*>(g),
                    static_cast<const uint4*>(u), n8, static_cast<uint4*>(h));
}

cudaError_t launch_combine(const void* y, const int32_t* assign_pos, const float* w, int T, int k, int H,
                           void* out, cudaStream_t st) {
  const int sms = current_sm_count();
  const long long threads = static_cast<long long>(T) * (H / 8);
  const int blocks = static_cast<int>(std::min<long long>((threads + 255) / 256, static_cast<long long>(sms) * 16));
  return launch_pdl(combine_kernel, dim3(blocks < 1 ? 1 : blocks), dim3(256), 0, st, static_cast<const uint4*>(y),
                    assign_pos, w, T, k, H / 8, static_cast<uint4*>(out));
}

cudaError_t launch_gather_f16(const void* x, int H, const int32_t* row_index, int P, int div, void* x_perm,
                              float* factor, cudaStream_t st) {
  const int sms = current_sm_count();
  return launch_pdl(gather_rows_f16_kernel, dim3(grid_for(8, P, sms * 8)), dim3(256), 0, st, static_cast<const uint4*>(x),
                    H / 8, row_index, P, div, static_cast<uint4*>(x_perm), factor);
}

}  // namespace mnw
