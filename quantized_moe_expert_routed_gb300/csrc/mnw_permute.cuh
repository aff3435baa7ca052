// mnw_permute.cuh -- the stable permutation of one batch of assignments by
// one CTA, as a device function: used by the permute kernel for decode-sized
// batches and by the fused router, whose last CTA permutes the ids the other
// CTAs of the same launch chose.
#pragma once
#include <cstdint>

#include "mnw_ptx.cuh"

namespace mnw {

// The same stable permutation for batches of at most kW * kB * 32
// assignments (a decode batch: 256 tokens x top-8 = 2048): kW warps, each
// owning a contiguous segment of at most kB * 32 assignments whose ids and
// match-any groups stay in registers from the counting pass to the placing
// pass (ids are read from global memory once), and a per-warp count table of
// kW * E entries.  Only the tail [valid assignments, P) of sorted_assign is
// filled with -1.
// Called by all kW * 32 threads of a CTA (blockDim.x == kW * 32); sm holds
// (kW + 1) * E ints of shared memory, warp_tot 32 ints, total_valid one.  ids
// are read through L2 (ld.global.cg), so they may have been written earlier by
// other CTAs of the same launch (after a fence).
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

  const int seg = (P + kW - 1) / kW;
  const int a0 = min(P, warp * seg), a1 = min(P, a0 + seg);
  int id[kB];
  uint32_t peers[kB];
#pragma unroll
  for (int b = 0; b < kB; ++b) {
    const int a = a0 + b * 32 + lane;
    id[b] = a < a1 ? __ldcg(ids + a) : INT32_MIN;
  }
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

}  // namespace mnw
