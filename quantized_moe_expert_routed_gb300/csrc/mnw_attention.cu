// mnw_attention.cu -- block attention for prompt prefill on tcgen05, with the
// scores kept on chip (the "coder543/minnow" README, "Quantization": Block
// FlashAttention for long-prompt prefill; its alternative materialises the
// score matrix).
//
// What it computes: for token t of sequence b and query head h (kv head
// g = h / (Hq / Hkv)), the softmax over the allowed keys j of
// scale * q[b,t,h] . k[b,j,g], applied to v[b,j,g]; key j is allowed when
// j / blk <= t / blk (block-causal: a block-diffusion model's prompt attends
// within its own 32-token block and to every earlier block).
//
// One CTA per (128-query tile, query head, sequence), heaviest query tiles
// first.  The key tiles are split between two independent softmax groups:
// group 0 takes the even tiles, group 1 the odd ones, each with its own
// score buffer, running maximum, row sums and output accumulator, and the two
// partial results are merged at the end (the usual rescaled sum of two
// softmax partitions).  While one group computes, the other's scores are in
// the tensor pipe, and the two output accumulators form independent MMA
// chains.  Roles (576 threads):
//   warp 0      TMA producer: the Q tile once, then 128-key K and V^T tiles
//               into two-slot rings
//   warp 1      MMA issuer (one thread), owns the tensor memory:
//               S_j = Q K_j^T (tcgen05.mma kind::f16, both operands in shared
//               memory) into group (j % 2)'s score buffer, and O_g += P_j V_j
//               with P_j read from tensor memory (the A operand of
//               tcgen05.mma may live there) and V_j^T from shared memory.
//               Order: S_0, S_1, then for each j: O += P_j V_j, S_{j+2}.
//   warps 2-17  softmax: group g = warps 2 + 8g .. 9 + 8g; in a group, two
//               warps per TMEM lane quarter, warp part p owning keys
//               64p..64p+63 of the group's tiles for the quarter's 32 query
//               rows, one row per lane.  Per tile: the row maximum of the
//               scaled scores (the two parts' maxima meet through shared
//               memory and an mbarrier), P = 2^(s*log2e*scale - m) rounded to
//               BF16 and written over the first half of the part's own S
//               columns (two keys per column), the part's row sum of the
//               rounded P.  The group's running maximum m moves, and its O
//               columns and row sums are rescaled, only when a tile's maximum
//               exceeds it by more than 2^8; other tiles keep the old m, whose
//               P values stay below 2^8.  A tile's scores being complete means
//               the group's previous product into O is complete too (same
//               issuing thread, in order), so a rescale needs no extra wait.
// Tensor memory (512 columns): S_0 | S_1 | O_0 | O_1.
// V is transposed into the workspace first (keys contiguous per head
// dimension) so that both products read K-major operands.
#include <cuda_bf16.h>

#include <atomic>

#include "mnw_convert.cuh"
#include "mnw_internal.h"
#include "mnw_ptx.cuh"

namespace mnw {
namespace attn {

constexpr int kD = 128;    // head dimension
constexpr int kBQ = 128;   // queries per tile (the MMAs' M)
constexpr int kBK = 128;   // keys per tile
constexpr int kSlots = 2;  // K and V^T ring depth
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpSm0 = 2, kSmWarps = 16;
constexpr int kThreads = (kWarpSm0 + kSmWarps) * 32;
constexpr uint32_t kBoxBytes = 128 * 128;           // 128 rows x 64 BF16 (128 bytes, 128-byte swizzle)
constexpr uint32_t kTileBytes = 2 * kBoxBytes;      // 128 rows x 128 BF16
constexpr uint32_t kOffQ = 0, kOffK = kTileBytes, kOffV = kOffK + kSlots * kTileBytes;
constexpr uint32_t kOffBars = kOffV + kSlots * kTileBytes;
constexpr int kTmemCols = 512;
constexpr uint32_t kColO = 256;  // O_g at kColO + 128 g
constexpr float kRescaleLog2 = 8.f;

struct Args {
  int B, T, Hq, Hkv, blk, n_qt;
  float scale_log2;  // softmax scale times log2(e)
  __nv_bfloat16* out;
  uint32_t* err;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kSlots], k_empty[kSlots], v_full[kSlots], v_empty[kSlots];
  uint64_t s_full[2], p_full[2], o_final, mma_drain;  // s_full, p_full: per softmax group
  uint64_t xmax[2][4][2];  // [group][quarter][tile parity]: the two parts' row maxima
  uint64_t fin[4];         // [quarter]: the four (group, part) warps' final row maxima and sums
  float pmax[2][2][4][2][32];  // [group][tile parity][quarter][part][lane]
  float fm[4][2][32], fl[4][2][2][32];  // final maxima [quarter][group][lane], sums [quarter][group][part][lane]
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = kOffBars + sizeof(Bars) + 1024;

struct RingPos {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void advance(uint32_t n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One lane waits, the warp follows (tcgen05.ld/st are warp-collective, so
// the whole warp takes the same branch).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = bounded_wait(bar, parity, abort, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

// Keys 0 .. kend-1 are allowed for query t (block-causal, clipped to T).
__device__ __forceinline__ int key_end(int t, int blk, int T) {
  const long long km = (static_cast<long long>(t / blk) + 1) * blk;
  return km > T ? T : static_cast<int>(km);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Args args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = args.T, Hq = args.Hq;

  // work item: query tiles in decreasing order (most keys first), then head, then sequence
  const int per_qt = Hq * args.B;
  const int qt = args.n_qt - 1 - static_cast<int>(blockIdx.x) / per_qt;
  const int rem = static_cast<int>(blockIdx.x) % per_qt;
  const int h = rem % Hq, b = rem / Hq;
  const int g = h / (Hq / args.Hkv);
  const int q0 = qt * kBQ;
  const int kend_tile = key_end(min(q0 + kBQ, T) - 1, args.blk, T);
  const int nt = (kend_tile + kBK - 1) / kBK;  // key tiles this query tile needs (>= 1)

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], kSmWarps / 2);
    }
    mbar_init(&bars->o_final, 1);
    mbar_init(&bars->mma_drain, 1);
    for (int i = 0; i < 4; ++i) {
      for (int gg = 0; gg < 2; ++gg) {
        mbar_init(&bars->xmax[gg][i][0], 2);
        mbar_init(&bars->xmax[gg][i][1], 2);
      }
      mbar_init(&bars->fin[i], 4);
    }
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  pdl_wait();  // q, k and the transposed v are written by earlier work on the stream
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kWarpTma) {
    // ======================= producer =======================
    if (lane == 0) {
      bool ok = true;
      uint32_t k_issued = 0, v_issued = 0;
      mbar_arrive_expect_tx(&bars->q_full, kTileBytes);
      tma_load_4d(smem + kOffQ, &tmQ, &bars->q_full, 0, h, q0, b);
      tma_load_4d(smem + kOffQ + kBoxBytes, &tmQ, &bars->q_full, 64, h, q0, b);
      RingPos kp, vp;
      for (int j = 0; ok && j < nt; ++j) {
        if (!bounded_wait(&bars->k_empty[kp.slot], kp.phase ^ 1, abort, args.err)) { ok = false; break; }
        uint8_t* kd = smem + kOffK + kp.slot * kTileBytes;
        mbar_arrive_expect_tx(&bars->k_full[kp.slot], kTileBytes);
        tma_load_4d(kd, &tmK, &bars->k_full[kp.slot], 0, g, j * kBK, b);
        tma_load_4d(kd + kBoxBytes, &tmK, &bars->k_full[kp.slot], 64, g, j * kBK, b);
        ++k_issued;
        kp.advance(kSlots);
        if (!bounded_wait(&bars->v_empty[vp.slot], vp.phase ^ 1, abort, args.err)) { ok = false; break; }
        uint8_t* vd = smem + kOffV + vp.slot * kTileBytes;
        mbar_arrive_expect_tx(&bars->v_full[vp.slot], kTileBytes);
        tma_load_4d(vd, &tmV, &bars->v_full[vp.slot], j * kBK, 0, g, b);
        tma_load_4d(vd + kBoxBytes, &tmV, &bars->v_full[vp.slot], j * kBK + 64, 0, g, b);
        ++v_issued;
        vp.advance(kSlots);
      }
      if (!ok || *abort) {
        // let every copy already issued land before the CTA exits
        drain_wait(&bars->q_full, 0);
        for (uint32_t i = k_issued > kSlots ? k_issued - kSlots : 0; i < k_issued; ++i)
          drain_wait(&bars->k_full[i % kSlots], (i / kSlots) & 1);
        for (uint32_t i = v_issued > kSlots ? v_issued - kSlots : 0; i < v_issued; ++i)
          drain_wait(&bars->v_full[i % kSlots], (i / kSlots) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kBQ, kBK, true);
      const uint32_t idesc_pv = idesc_f16(kBQ, kD, true);
      const uint32_t q_s = smem_u32(smem + kOffQ);
      bool ok = bounded_wait(&bars->q_full, 0, abort, args.err);
      bool issued = false;
      RingPos kp, vp;
      auto issue_s = [&](int j) -> bool {
        if (!bounded_wait(&bars->k_full[kp.slot], kp.phase, abort, args.err)) return false;
        tc_fence_after();
        const uint32_t k_s = smem_u32(smem + kOffK + kp.slot * kTileBytes);
        const uint32_t d = tmem + static_cast<uint32_t>(j & 1) * kBK;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ss(d, sdesc_sw128(q_s + off), sdesc_sw128(k_s + off), idesc, kk > 0);
        }
        issued = true;
        mma_commit(&bars->k_empty[kp.slot]);
        mma_commit(&bars->s_full[j & 1]);
        kp.advance(kSlots);
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        if (!bounded_wait(&bars->p_full[j & 1], (j >> 1) & 1, abort, args.err)) return false;
        if (!bounded_wait(&bars->v_full[vp.slot], vp.phase, abort, args.err)) return false;
        tc_fence_after();
        const uint32_t v_s = smem_u32(smem + kOffV + vp.slot * kTileBytes);
        // P_j: keys 64p..64p+63 in columns 64p..64p+31 of the group's S buffer, two keys each
        const uint32_t p = tmem + static_cast<uint32_t>(j & 1) * kBK;
        const uint32_t o = tmem + kColO + static_cast<uint32_t>(j & 1) * kD;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ts(o, p + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_sw128(v_s + off), idesc_pv, (j > 1 || kk > 0));
        }
        mma_commit(&bars->v_empty[vp.slot]);
        vp.advance(kSlots);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && nt > 1) ok = issue_s(1);
      for (int j = 0; ok && j < nt; ++j) {
        ok = issue_pv(j);
        if (ok && j + 2 < nt) ok = issue_s(j + 2);
      }
      if (ok) mma_commit(&bars->o_final);
      if (issued) {
        // every MMA has finished with shared and tensor memory before the CTA tears down
        mma_commit(&bars->mma_drain);
        drain_wait(&bars->mma_drain, 0);
      }
    }
  } else {
    // ======================= softmax =======================
    const int grp = (warp - kWarpSm0) >> 3;         // softmax group: key tiles grp, grp + 2, ...
    const int q = warp & 3;                         // TMEM lane quarter: query rows 32q .. 32q+31
    const int part = ((warp - kWarpSm0) >> 2) & 1;  // keys (and O columns) 64 part .. 64 part + 63
    const int r = q * 32 + lane;
    const int t = q0 + r;
    const uint32_t lane_bits = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t sbase = tmem + lane_bits + static_cast<uint32_t>(grp) * kBK + part * 64;
    const uint32_t obase = tmem + lane_bits + kColO + static_cast<uint32_t>(grp) * kD + part * 64;
    const int kend = key_end(min(t, T - 1), args.blk, T);
    const float sl2 = args.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    int k = 0;  // tiles of this group done
    for (int j = grp; j < nt; j += 2, ++k) {
      if (!warp_wait(&bars->s_full[grp], k & 1, abort, args.err)) { ok = false; break; }
      tc_fence_after();
      const int lim = kend - j * kBK - part * 64;  // keys e < lim of this part are allowed for the row
      float mx = -INFINITY;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t sv[32];
        tmem_ld32(sbase + hh * 32, sv);
        tmem_wait_ld();
        const int lh = lim - 32 * hh;
        if (lh >= 32) {
#pragma unroll
          for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(sv[e]));
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e < lh) mx = fmaxf(mx, __uint_as_float(sv[e]));
        }
      }
      // the row's maximum over the two parts
      bars->pmax[grp][k & 1][q][part][lane] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->xmax[grp][q][k & 1]);
      if (!warp_wait(&bars->xmax[grp][q][k & 1], (k >> 1) & 1, abort, args.err)) { ok = false; break; }
      mx = fmaxf(bars->pmax[grp][k & 1][q][0][lane], bars->pmax[grp][k & 1][q][1][lane]) * sl2;  // scale > 0
      if (k == 0) {
        m_used = mx;  // key 0 is allowed for every row, so the first tile's maximum is finite
      } else {
        const bool resc = mx > m_used + kRescaleLog2;
        if (__any_sync(0xffffffffu, resc)) {
          // O_grp holds this group's earlier products, all complete (see above)
          const float alpha = resc ? ex2(m_used - mx) : 1.f;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t o[32];
            tmem_ld32(obase + hh * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(obase + hh * 32, *reinterpret_cast<uint32_t(*)[16]>(&o[0]));
            tmem_st16(obase + hh * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&o[16]));
          }
          tmem_wait_st();
          if (resc) {
            l *= alpha;
            m_used = mx;
          }
        }
      }
      // P as BF16 pairs over the first 32 of this part's 64 S columns: keys 32hh .. 32hh+31
      // are read (again) before their 16 columns of P are written, below them
      // two keys per packed FP32x2 operation: the exponent argument and the row sums
      const uint64_t sl2x2 = f32x2_pack(__float_as_uint(sl2), __float_as_uint(sl2));
      const uint64_t mneg2 = f32x2_pack(__float_as_uint(-m_used), __float_as_uint(-m_used));
      uint64_t l2 = 0ull;  // even and odd keys' partial sums
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t sv[32];
        tmem_ld32(sbase + hh * 32, sv);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int key = 32 * hh + 2 * e;
          const uint64_t t2 = f32x2_fma(f32x2_pack(sv[2 * e], sv[2 * e + 1]), sl2x2, mneg2);
          const float p0 = key < lim ? ex2(__uint_as_float(static_cast<uint32_t>(t2))) : 0.f;
          const float p1 = key + 1 < lim ? ex2(__uint_as_float(static_cast<uint32_t>(t2 >> 32))) : 0.f;
          const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
          const uint32_t pw = *reinterpret_cast<const uint32_t*>(&pb);
          l2 = f32x2_add(l2, f32x2_pack(pw << 16, pw & 0xFFFF0000u));  // the rounded P, as FP32
          pk[e] = pw;
        }
        tmem_st16(sbase + hh * 16, pk);
      }
      l += __uint_as_float(static_cast<uint32_t>(l2)) + __uint_as_float(static_cast<uint32_t>(l2 >> 32));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[grp]);
    }
    // merge the two groups: out = sum_g 2^(m_g - M) O_g / sum_g 2^(m_g - M) l_g, M = max m_g
    if (ok) {
      if (part == 0) bars->fm[q][grp][lane] = m_used;
      bars->fl[q][grp][part][lane] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->fin[q]);
      ok = warp_wait(&bars->fin[q], 0, abort, args.err);
    }
    if (ok && warp_wait(&bars->o_final, 0, abort, args.err)) {
      tc_fence_after();
      const float m0 = bars->fm[q][0][lane], m1 = bars->fm[q][1][lane];
      const float l0 = bars->fl[q][0][0][lane] + bars->fl[q][0][1][lane];
      const float l1 = bars->fl[q][1][0][lane] + bars->fl[q][1][1][lane];
      const bool two = nt > 1;  // with one key tile, group 1 wrote nothing (O_1 is not read)
      const float M = two ? fmaxf(m0, m1) : m0;
      const float a0 = ex2(m0 - M), a1 = two ? ex2(m1 - M) : 0.f;
      const float inv = 1.f / (l0 * a0 + l1 * a1);
      // this warp writes O columns 32 (2 grp + part) .. +31 of its quarter's rows, 16 at a time
      const float s0 = a0 * inv, s1 = a1 * inv;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int c0 = 32 * (2 * grp + part) + 16 * hh;
        uint32_t o0[16], o1[16];
        tmem_ld16(tmem + lane_bits + kColO + c0, o0);
        if (two) tmem_ld16(tmem + lane_bits + kColO + kD + c0, o1);
        tmem_wait_ld();
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float v0 = __uint_as_float(o0[2 * e]) * s0, v1 = __uint_as_float(o0[2 * e + 1]) * s0;
          if (two) {
            v0 = fmaf(__uint_as_float(o1[2 * e]), s1, v0);
            v1 = fmaf(__uint_as_float(o1[2 * e + 1]), s1, v1);
          }
          pk[e] = pack_bf16x2(v0, v1);
        }
        if (t < T) {
          __nv_bfloat16* dst = args.out + ((static_cast<size_t>(b) * T + t) * Hq + h) * kD + c0;
          stg128(dst, pk[0], pk[1], pk[2], pk[3]);
          stg128(dst + 8, pk[4], pk[5], pk[6], pk[7]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// v [B, T, Hkv, 128] -> vt [B, Hkv, 128, Tp] (keys contiguous); 64 keys per CTA.
__global__ void __launch_bounds__(256) attn_vt_kernel(const __nv_bfloat16* __restrict__ v, int T, int Hkv, int Tp,
                                                       __nv_bfloat16* __restrict__ vt) {
  __shared__ __nv_bfloat16 tile[kD][64 + 2];
  pdl_launch_dependents();
  pdl_wait();
  const int t0 = blockIdx.x * 64, g = blockIdx.y, b = blockIdx.z;
  for (int i = threadIdx.x; i < 64 * kD; i += blockDim.x) {
    const int tt = i / kD, c = i % kD;
    const int t = t0 + tt;
    tile[c][tt] = t < T ? v[((static_cast<size_t>(b) * T + t) * Hkv + g) * kD + c] : __float2bfloat16_rn(0.f);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * kD; i += blockDim.x) {
    const int c = i / 64, tt = i % 64;
    const int t = t0 + tt;
    if (t < T) vt[((static_cast<size_t>(b) * Hkv + g) * kD + c) * Tp + t] = tile[c][tt];
  }
}

inline int padded_keys(int T) { return (T + 7) / 8 * 8; }

}  // namespace attn
}  // namespace mnw

using namespace mnw;

extern "C" {

size_t mnw_attn_workspace_size(int B, int T, int Hkv, int d) {
  if (B <= 0 || T <= 0 || Hkv <= 0 || d <= 0) return 0;
  const size_t bytes = static_cast<size_t>(B) * Hkv * d * attn::padded_keys(T) * 2;
  return (bytes + 255) / 256 * 256;
}

int mnw_attn_prefill(const void* q, const void* k, const void* v, int B, int T, int Hq, int Hkv, int d, int blk,
                     float scale, void* out, void* ws, size_t ws_bytes, uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_attn_prefill");
  using namespace attn;
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || blk < 1 || Hq % Hkv) return MNW_E_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return MNW_E_INVALID_ARG;
  if (d != kD) return MNW_E_UNSUPPORTED;
  if (B == 0 || T == 0) return MNW_OK;
  if (static_cast<long long>(B) * T * Hq > (1ll << 31) / kD) return MNW_E_UNSUPPORTED;
  if (!q || !k || !v || !out || !ws || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(ws, 256))
    return MNW_E_INVALID_ARG;
  if (ws_bytes < mnw_attn_workspace_size(B, T, Hkv, d)) return MNW_E_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int Tp = padded_keys(T);
  auto* vt = static_cast<__nv_bfloat16*>(ws);

  cudaError_t e = launch_pdl(attn_vt_kernel, dim3((T + 63) / 64, Hkv, B), dim3(256), 0, st,
                             static_cast<const __nv_bfloat16*>(v), T, Hkv, Tp, vt);
  if (e != cudaSuccess) return MNW_E_CUDA;

  CUtensorMap maps[3];
  memset(maps, 0, sizeof(maps));
  const uint32_t box_qk[4] = {64, 1, static_cast<uint32_t>(kBQ), 1};
  {
    const uint64_t dims[4] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hq), static_cast<uint64_t>(T),
                              static_cast<uint64_t>(B)};
    const uint64_t strides[3] = {static_cast<uint64_t>(kD) * 2, static_cast<uint64_t>(Hq) * kD * 2,
                                 static_cast<uint64_t>(T) * Hq * kD * 2};
    if (!encode_map(&maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, q, dims, strides, box_qk, CU_TENSOR_MAP_SWIZZLE_128B))
      return MNW_E_INVALID_ARG;
  }
  {
    const uint64_t dims[4] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hkv), static_cast<uint64_t>(T),
                              static_cast<uint64_t>(B)};
    const uint64_t strides[3] = {static_cast<uint64_t>(kD) * 2, static_cast<uint64_t>(Hkv) * kD * 2,
                                 static_cast<uint64_t>(T) * Hkv * kD * 2};
    if (!encode_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k, dims, strides, box_qk, CU_TENSOR_MAP_SWIZZLE_128B))
      return MNW_E_INVALID_ARG;
  }
  {
    // keys beyond T read as zero (the map ends at T; the rows are Tp long)
    const uint64_t dims[4] = {static_cast<uint64_t>(T), static_cast<uint64_t>(kD), static_cast<uint64_t>(Hkv),
                              static_cast<uint64_t>(B)};
    const uint64_t strides[3] = {static_cast<uint64_t>(Tp) * 2, static_cast<uint64_t>(kD) * Tp * 2,
                                 static_cast<uint64_t>(Hkv) * kD * Tp * 2};
    const uint32_t box[4] = {64, static_cast<uint32_t>(kD), 1, 1};
    if (!encode_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, vt, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MNW_E_INVALID_ARG;
  }
  Args a{};
  a.B = B;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.blk = blk;
  a.n_qt = (T + kBQ - 1) / kBQ;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.err = err;

  static std::atomic<uint64_t> attr{0};
  uint64_t bit;
  if (attrs_needed(attr, &bit)) {
    e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return MNW_E_CUDA;
    attrs_done(attr, bit);
  }
  const long long grid = static_cast<long long>(a.n_qt) * Hq * B;
  if (grid > 0x7fffffffll) return MNW_E_UNSUPPORTED;
  e = launch_pdl(attn_fwd_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes, st, maps[0], maps[1],
                 maps[2], a);
  return e == cudaSuccess ? MNW_OK : MNW_E_CUDA;
}

}  // extern "C"
