// mnw_permute.cuh -- the stable permutation of one batch of assignments by
// one CTA, as a device function: used by the permute kernel for decode-sized
// batches and by the fused router, whose last CTA permutes the ids the other
// CTAs of the same launch chose.
#pragma once
#include <cstdint>

#include "mnw_ptx.cuh"

namespace mnw {

// ids[a0 + 32 b + lane] -> id[b] for b < kB (INT32_MIN at or past a1), with
// a1 - a0 <= 32 kB.  When ids + a0 is 16-byte aligned the warp reads the
// range with 16-byte loads (each lane four consecutive ids) and puts it back
// in lane order through its own window of 32 kB ints of shared memory (16-byte
// aligned); otherwise with 4-byte loads.  Loads go through L2 (ld.global.cg):
// the ids may come from other CTAs of the same launch.  Called by all 32
// lanes of a warp.
template <int kB>
__device__ __forceinline__ void load_ids(const int32_t* ids, int a0, int a1, int32_t* win, int (&id)[kB]) {
  const int lane = threadIdx.x & 31;
  const int n = a1 - a0;
  if ((reinterpret_cast<uintptr_t>(ids + a0) & 15u) == 0) {
#pragma unroll
    for (int q = 0; q < kB / 4 + (kB % 4 ? 1 : 0); ++q) {
      const int i = q * 32 + lane;  // 16-byte word i holds ids a0 + 4i .. a0 + 4i + 3
      if (i < kB * 8 && 4 * i < n) {
        int4 v;
        if (4 * i + 3 < n) {
          v = __ldcg(reinterpret_cast<const int4*>(ids + a0) + i);
        } else {  // the ragged end: no load past a1
          v.x = __ldcg(ids + a0 + 4 * i);
          v.y = 4 * i + 1 < n ? __ldcg(ids + a0 + 4 * i + 1) : INT32_MIN;
          v.z = 4 * i + 2 < n ? __ldcg(ids + a0 + 4 * i + 2) : INT32_MIN;
          v.w = INT32_MIN;
        }
        reinterpret_cast<int4*>(win)[i] = v;
      }
    }
    __syncwarp();
#pragma unroll
    for (int b = 0; b < kB; ++b) id[b] = 32 * b + lane < n ? win[32 * b + lane] : INT32_MIN;
    __syncwarp();  // the window may be refilled next
  } else {
#pragma unroll
    for (int b = 0; b < kB; ++b) id[b] = 32 * b + lane < n ? __ldcg(ids + a0 + 32 * b + lane) : INT32_MIN;
  }
}

// Shared-memory ints before the id windows: n rounded up to a 16-byte boundary.
__host__ __device__ constexpr int ids_window_base(int n) { return (n + 3) & ~3; }

// The same stable permutation for batches of at most kW * kB * 32
// assignments (a decode batch: 256 tokens x top-8 = 2048): kW warps, each
// owning a contiguous segment of at most kB * 32 assignments whose ids and
// match-any groups stay in registers from the counting pass to the placing
// pass (ids are read from global memory once), and a per-warp count table of
// kW * E entries.  Only the tail [valid assignments, P) of sorted_assign is
// filled with -1.
// Called by all kW * 32 threads of a CTA (blockDim.x == kW * 32); sm holds
// permute_block_smem_ints(kW, kB, E) ints of shared memory (16-byte aligned):
// the count tables, then one id window per warp; warp_tot 32 ints,
// total_valid one.  ids are read through L2 (ld.global.cg), so they may have
// been written earlier by other CTAs of the same launch (after a fence).
template <int kW, int kB>
__device__ __forceinline__ void permute_block(const int32_t* ids, int P, int E, int32_t* __restrict__ offsets,
                                              int32_t* __restrict__ sorted_assign, int32_t* __restrict__ assign_pos,
                                              uint32_t* __restrict__ err, int32_t* sm, int32_t* warp_tot,
                                              int32_t* total_valid_p) {
  constexpr int kThreads = kW * 32;
  int32_t* cnt = sm;                // [kW][E]: counts, then exclusive prefix over warps
  int32_t* tot = sm + kW * E;       // [E]: totals, then expert start offsets
  int32_t& total_valid = *total_valid_p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < kW * E; i += kThreads) cnt[i] = 0;

  // segments of a multiple of 4 assignments, so that each starts on a 16-byte boundary of ids
  const int seg = ((P + kW - 1) / kW + 3) & ~3;
  const int a0 = min(P, warp * seg), a1 = min(P, a0 + seg);
  int id[kB];
  uint32_t peers[kB];
  load_ids<kB>(ids, a0, a1, sm + ids_window_base((kW + 1) * E) + warp * kB * 32, id);
  __syncthreads();

  // counting pass: per-warp counts, lanes sharing an expert grouped by match-any
  int32_t* my = cnt + warp * E;
#pragma unroll
  for (int b = 0; b < kB; ++b) {
    const int a = a0 + b * 32 + lane;
    const bool active = a < a1;
    const bool valid = active && id[b] >= 0 && id[b] < E;
    if (active && !valid && err) atomicOr(err, MNW_DEVERR_BAD_EXPERT_ID);
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
    peers[b] = valid ? __match_any_sync(vmask, id[b]) : 0u;
    if (valid && lane == __ffs(peers[b]) - 1) my[id[b]] += __popc(peers[b]);
    __syncwarp();
  }
  __syncthreads();

  // exclusive prefix over warps for every expert; totals per expert
  for (int e = tid; e < E; e += kThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const int c = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();

  // exclusive scan of the totals over experts: thread tid owns experts [tid*per, tid*per + per)
  const int per = (E + kThreads - 1) / kThreads;
  const int e0 = tid * per;
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (e0 + i < E) local += tot[e0 + i];
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int t = lane < kW ? warp_tot[lane] : 0;
    int ti = t;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, ti, d);
      if (lane >= d) ti += o;
    }
    if (lane < kW) warp_tot[lane] = ti - t;
  }
  __syncthreads();
  int run = incl - local + warp_tot[warp];
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E) {
      const int c = tot[e];
      offsets[e] = run;
      tot[e] = run;
      run += c;
    }
  }
  if (tid == kThreads - 1) {
    offsets[E] = run;
    total_valid = run;
  }
  __syncthreads();

  // placing pass: stable position = expert start + earlier warps + earlier lanes/batches of this warp
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int b = 0; b < kB; ++b) {
    const int a = a0 + b * 32 + lane;
    const bool active = a < a1;
    const bool valid = peers[b] != 0u;
    if (valid) {
      const int pos = tot[id[b]] + my[id[b]] + __popc(peers[b] & lt_mask);
      assign_pos[a] = pos;
      sorted_assign[pos] = a;
    } else if (active) {
      assign_pos[a] = -1;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers[b]) - 1) my[id[b]] += __popc(peers[b]);
    __syncwarp();
  }
  for (int p = total_valid + tid; p < P; p += kThreads) sorted_assign[p] = -1;
}

// Shared-memory ints permute_block needs for kW warps, kB batches and E experts.
__host__ __device__ constexpr int permute_block_smem_ints(int kW, int kB, int E) {
  return ids_window_base((kW + 1) * E) + kW * kB * 32;
}

}  // namespace mnw
