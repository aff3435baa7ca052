// mnw_gemm_rows.cu -- grouped expert GEMMs on tcgen05 with the tokens as the
// MMA's M and 256 weight rows as its N ("row tiles").
//
// Why this shape: on GB300 a tcgen05.mma of M = 128 from shared memory costs
// about the same issue time for any N up to 192 (and only ~25% more at 256),
// so the tensor pipe reaches its rate only when every instruction carries
// N = 256.  Token counts per expert vary (a decode batch routes a few tokens
// to each expert, a skewed prefill hundreds), while the weight side always
// has rows to spare: a tile is therefore up to 128 tokens of one expert (M)
// by 256 weight rows (N) -- gate rows n0..n0+127 followed by the same up rows
// (so SiLU(g) * u pairs two accumulator columns of one thread), or 256
// consecutive down rows.  Each MMA then does the same work whatever the token
// count is, and a tile with few tokens costs what a full one does.
//
// Formats (the "LLaDA2.2-flash-minnow" model card, "Checkpoints and
// precision"):
//   INT8 / INT4 weights with BF16 activations: the activations arrive as
//     FP16 rows with a power-of-two factor per row (an exact re-encoding of the
//     BF16 values), the converter warps dequantise each weight code to
//     fp16(q * s) with its FP16 group scale into the operand tile (one
//     rounding, relative 2^-11), FP32 accumulation over all of K, and the
//     epilogue multiplies by the row factor.  No expanded weight copy exists
//     outside shared memory.
//   BF16 weights with BF16 activations: both operands straight from the TMA.
//
// Roles (576 threads):
//   warp 0      TMA producer: 64-K token tiles (128 rows), raw weight-code
//               stages (two 128-row boxes of 128 bytes), BF16 weight tiles
//   warp 1      MMA issuer (one thread), owns the tensor memory
//   warps 2-9   converters: thread c dequantises weight row c of the tile into
//               a 64-K FP16 operand tile (128-byte swizzle) per step
//   warps 10-17 epilogue: two warps per TMEM lane quarter (32 tokens), each
//               with half of the feature columns
// Tensor memory: two accumulators of 256 columns (the next tile's MMAs fill
// one while the epilogue drains the other).
//
// Work unit (expert e, feature tile nt, token tile tt), ordered by expert,
// then feature tile, then token tile, so CTAs running at the same time share
// a weight tile (a hot expert's token tiles) or a token tile (its feature
// tiles) through L2.  Every wait is bounded (mnw_ptx.cuh).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "mnw_convert.cuh"
#include "mnw_internal.h"
#include "mnw_ptx.cuh"

namespace mnw {
namespace rows {

enum { WF_BF16 = 0, WF_INT8 = 1, WF_INT4 = 2 };

constexpr int kBM = 128;  // tokens per tile
constexpr int kBN = 256;  // weight rows per tile
// Measured on GB300 (reduced 4096 x 1536 INT4 gate/up): 16 converter warps
// and 4 epilogue warps 272 us, 8 and 8 284 us; 3 operand or token slots
// instead of 2 / 4 slower.  A token tile (128 rows of 128 bytes) takes ~3500
// cycles from TMA issue to arrival with 4 in flight per SM and ~5900 with 6:
// the token supply, not the MMA or the converters, sets the pace.
constexpr int kConvWarps = 16;  // 8: a weight row per thread; 16: half a row per thread
constexpr int kEpiWarps = 4;    // 4 or 8: one or two warps per TMEM lane quarter
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpConv0 = 2, kWarpEpi0 = kWarpConv0 + kConvWarps;
constexpr int kThreads = (kWarpEpi0 + kEpiWarps) * 32;
constexpr int kTokSlots = 4;         // 64-K token tiles (+ the BF16 weight tile for BF16 weights)
constexpr int kCodeSlots = 2;        // raw code stages: two boxes of 128 rows x 128 bytes
constexpr int kBSlots = 2;           // converted 64-K FP16 weight tiles
constexpr int kAccSlots = 2;
constexpr uint32_t kTokBytes = kBM * 128;        // 128 rows x 64 K x 2 bytes
constexpr uint32_t kWTileBytes = kBN * 128;      // 256 rows x 64 K x 2 bytes
constexpr uint32_t kCodeBytes = 2 * 128 * 128;   // two boxes
constexpr int kTmemCols = 512;

struct Args {
  const int32_t* offsets;
  int E, P, K, N, n_tiles, rows_per_tile;  // rows_per_tile: weight rows of one matrix per tile (128 or 256)
  uint32_t off_tok, tok_slot_bytes, off_code, off_b, off_tab, off_bars;
  const uint8_t* experts;
  uint64_t expert_stride;
  uint64_t scales_off[2];
  const float* a_outer;  // FP16 rows: the row's factor; nullptr for BF16 rows
  __nv_bfloat16* out;
  uint32_t* err;
};

struct Bars {
  uint64_t tfull[kTokSlots], tempty[kTokSlots];
  uint64_t cfull[kCodeSlots], cempty[kCodeSlots];
  uint64_t bfull[kBSlots], bempty[kBSlots];
  uint64_t afull[kAccSlots], aempty[kAccSlots];
  uint64_t final_mma;
  uint32_t tmem_base;
  int abort;
};

struct RingPos {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void advance(uint32_t n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

struct Unit {
  int e, nt, row0, nrows;
};

// u -> (expert, feature tile, token tile); prefix[e] = units before expert e.
__device__ __forceinline__ Unit decode(const int* prefix, const int* off, int E, int n_tiles, int u) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  Unit x;
  x.e = lo;
  const int r = u - prefix[lo];
  const int tiles = (prefix[lo + 1] - prefix[lo]) / n_tiles;  // token tiles of this expert
  x.nt = r / tiles;
  const int tt = r - x.nt * tiles;
  x.row0 = off[lo] + tt * kBM;
  x.nrows = min(kBM, off[lo + 1] - x.row0);
  return x;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

template <int WF, bool kGateUp>
__global__ void __launch_bounds__(kThreads, 1)
    rows_gemm_kernel(const __grid_constant__ CUtensorMap tmTok, const __grid_constant__ CUtensorMap tmW0,
                     const __grid_constant__ CUtensorMap tmW1, const Args args) {
  constexpr bool kConv = WF != WF_BF16;
  constexpr int kCodeK = WF == WF_INT4 ? 256 : 128;  // K per raw code stage (128-byte rows)
  constexpr int kSub = kCodeK / 64;                   // 64-K steps per code stage

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + args.off_bars);
  int* tab_prefix = reinterpret_cast<int*>(smem + args.off_tab);
  int* tab_off = tab_prefix + (args.E + 1);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E, K = args.K, n_tiles = args.n_tiles;
  const int nsteps = K / 64;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTokSlots; ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], 1);
    }
    for (int i = 0; i < kCodeSlots; ++i) {
      mbar_init(&bars->cfull[i], 1);
      mbar_init(&bars->cempty[i], kConvWarps);
    }
    for (int i = 0; i < kBSlots; ++i) {
      mbar_init(&bars->bfull[i], kConvWarps);
      mbar_init(&bars->bempty[i], 1);
    }
    for (int i = 0; i < kAccSlots; ++i) {
      mbar_init(&bars->afull[i], 1);
      mbar_init(&bars->aempty[i], kEpiWarps);
    }
    mbar_init(&bars->final_mma, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tmTok);
    tma_prefetch_desc(&tmW0);
    if (kGateUp) tma_prefetch_desc(&tmW1);
  }
  pdl_wait();
  // unit table: tab_prefix[e] = units before expert e (token tiles x feature tiles)
  if (warp == kWarpConv0) {
    const int per = (E + 31) / 32;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        const int o0 = __ldg(args.offsets + e), o1 = __ldg(args.offsets + e + 1);
        tab_off[e] = o0;
        local += max(0, (o1 - o0 + kBM - 1) / kBM) * n_tiles;
      }
    }
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        tab_prefix[e] = run;
        run += max(0, (__ldg(args.offsets + e + 1) - tab_off[e] + kBM - 1) / kBM) * n_tiles;
      }
    }
    if (lane == 31) {
      tab_prefix[E] = incl;
      tab_off[E] = __ldg(args.offsets + E);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int units = tab_prefix[E];
  uint8_t* tok_ring = smem + args.off_tok;
  uint8_t* code_ring = smem + args.off_code;
  uint8_t* b_ring = smem + args.off_b;

  if (warp == kWarpTma) {
    // ======================= producer =======================
    if (lane == 0) {
      RingPos tp, cp;
      uint32_t t_issued = 0, c_issued = 0;
      bool ok = true;
      const uint32_t tok_tx = kTokBytes + (kConv ? 0u : kWTileBytes);
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const Unit x = decode(tab_prefix, tab_off, E, n_tiles, u);
        const int n0 = x.nt * args.rows_per_tile;
        for (int step = 0; ok && step < nsteps; ++step) {
          if (kConv && step % kSub == 0) {
            // raw codes of the next kCodeK for the tile's 256 weight rows
            if (!bounded_wait(&bars->cempty[cp.slot], cp.phase ^ 1, abort, args.err)) { ok = false; break; }
            uint8_t* dst = code_ring + cp.slot * kCodeBytes;
            mbar_arrive_expect_tx(&bars->cfull[cp.slot], kCodeBytes);
            const int kx = (step / kSub) * 128;  // bytes
            tma_load_3d(dst, &tmW0, &bars->cfull[cp.slot], kx, n0, x.e);
            if (kGateUp) tma_load_3d(dst + 16384, &tmW1, &bars->cfull[cp.slot], kx, n0, x.e);
            else tma_load_3d(dst + 16384, &tmW0, &bars->cfull[cp.slot], kx, n0 + 128, x.e);
            ++c_issued;
            cp.advance(kCodeSlots);
          }
          if (!bounded_wait(&bars->tempty[tp.slot], tp.phase ^ 1, abort, args.err)) { ok = false; break; }
          uint8_t* dst = tok_ring + tp.slot * args.tok_slot_bytes;
          mbar_arrive_expect_tx(&bars->tfull[tp.slot], tok_tx);
          tma_load_2d(dst, &tmTok, &bars->tfull[tp.slot], step * 64, x.row0);
          if (!kConv) {
            tma_load_3d(dst + kTokBytes, &tmW0, &bars->tfull[tp.slot], step * 64, n0, x.e);
            if (kGateUp) tma_load_3d(dst + kTokBytes + 16384, &tmW1, &bars->tfull[tp.slot], step * 64, n0, x.e);
            else tma_load_3d(dst + kTokBytes + 16384, &tmW0, &bars->tfull[tp.slot], step * 64, n0 + 128, x.e);
          }
          ++t_issued;
          tp.advance(kTokSlots);
        }
      }
      if (!ok || *abort) {
        // let every copy already issued land before the CTA exits
        for (uint32_t j = t_issued > kTokSlots ? t_issued - kTokSlots : 0; j < t_issued; ++j)
          drain_wait(&bars->tfull[j % kTokSlots], (j / kTokSlots) & 1);
        for (uint32_t j = c_issued > kCodeSlots ? c_issued - kCodeSlots : 0; j < c_issued; ++j)
          drain_wait(&bars->cfull[j % kCodeSlots], (j / kCodeSlots) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kBM, kBN, !kConv ? true : false);
      RingPos tp, bp, ap;
      bool ok = true, issued = false;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        if (!bounded_wait(&bars->aempty[ap.slot], ap.phase ^ 1, abort, args.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + ap.slot * kBN;
        for (int step = 0; step < nsteps; ++step) {
          if (!bounded_wait(&bars->tfull[tp.slot], tp.phase, abort, args.err)) { ok = false; break; }
          if (kConv && !bounded_wait(&bars->bfull[bp.slot], bp.phase, abort, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_tile = smem_u32(tok_ring + tp.slot * args.tok_slot_bytes);
          const uint32_t b_tile = kConv ? smem_u32(b_ring + bp.slot * kWTileBytes) : a_tile + kTokBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(d, sdesc_sw128(a_tile + kk * 32), sdesc_sw128(b_tile + kk * 32), idesc, (step | kk) != 0);
          issued = true;
          mma_commit(&bars->tempty[tp.slot]);
          tp.advance(kTokSlots);
          if (kConv) {
            mma_commit(&bars->bempty[bp.slot]);
            bp.advance(kBSlots);
          }
        }
        if (!ok) break;
        mma_commit(&bars->afull[ap.slot]);
        ap.advance(kAccSlots);
      }
      if (issued) {
        mma_commit(&bars->final_mma);
        drain_wait(&bars->final_mma, 0);
      }
    }
  } else if (warp < kWarpEpi0) {
    // ======================= converters =======================
    if (kConv) {
      // kParts threads share a weight row: thread (c, part) converts K
      // [part * kKPer, (part + 1) * kKPer) of row c of every 64-K step.
      constexpr int kParts = kConvWarps / 8;
      constexpr int kKPer = 64 / kParts;
      const int ct = (warp - kWarpConv0) * 32 + lane;
      const int c = ct & (kBN - 1), part = ct / kBN;  // weight row of the tile (0..255), its K part
      const int box = c >> 7, r = c & 127;            // code box and its row
      const int G = K / 128;
      RingPos cp, bp;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const Unit x = decode(tab_prefix, tab_off, E, n_tiles, u);
        // this row's FP16 group scales, read from global memory one group ahead
        // (a select, not an index: a runtime index into the parameter array would copy it to local memory)
        const uint64_t soff = (kGateUp && box) ? args.scales_off[1] : args.scales_off[0];
        const int wrow = x.nt * args.rows_per_tile + (kGateUp ? r : c);
        const __half* srow = reinterpret_cast<const __half*>(args.experts + static_cast<uint64_t>(x.e) * args.expert_stride +
                                                             soff) +
                             static_cast<size_t>(wrow) * G;
        uint32_t s_cur = __half_as_ushort(__ldg(srow));
        uint32_t s_nxt = G > 1 ? __half_as_ushort(__ldg(srow + 1)) : 0u;
        for (int step = 0; step < nsteps; ++step) {
          const int sub = step % kSub;
          if (sub == 0 && !bounded_wait(&bars->cfull[cp.slot], cp.phase, abort, args.err)) { ok = false; break; }
          if (step > 0 && (step & 1) == 0) {  // a new 128-K group
            s_cur = s_nxt;
            const int g = step / 2;
            s_nxt = g + 1 < G ? __half_as_ushort(__ldg(srow + g + 1)) : 0u;
          }
          const uint32_t src = smem_u32(code_ring + cp.slot * kCodeBytes + box * 16384);
          const int kin = sub * 64 + part * kKPer;  // K offset inside the code stage
          // codes first: the loads overlap the wait for a free operand slot
          uint4 v[kKPer / 16];
          if (WF == WF_INT4) {
#pragma unroll
            for (int j = 0; j < kKPer / 32; ++j) v[j] = lds128(sw128(src, r, kin / 32 + j));  // 32 codes per chunk
          } else {
#pragma unroll
            for (int j = 0; j < kKPer / 16; ++j) v[j] = lds128(sw128(src, r, kin / 16 + j));  // 16 codes per chunk
          }
          if (!bounded_wait(&bars->bempty[bp.slot], bp.phase ^ 1, abort, args.err)) { ok = false; break; }
          const uint32_t dst = smem_u32(b_ring + bp.slot * kWTileBytes);
          const uint32_t s2 = s_cur | (s_cur << 16);
          uint32_t o[kKPer / 2];
#pragma unroll
          for (int j = 0; j < kKPer / 32; ++j) {
            uint32_t h[16];
            if (WF == WF_INT4) cvt_int4x32<false>(v[j], h);
            else cvt_int8x32<false>(v[2 * j], v[2 * j + 1], h);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[16 * j + i] = f16x2_mul(h[i], s2);
          }
#pragma unroll
          for (int ch = 0; ch < kKPer / 8; ++ch)
            sts128(sw128(dst, c, part * (kKPer / 8) + ch), o[4 * ch], o[4 * ch + 1], o[4 * ch + 2], o[4 * ch + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->bfull[bp.slot]);
          bp.advance(kBSlots);
          if (sub == kSub - 1) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->cempty[cp.slot]);
            cp.advance(kCodeSlots);
          }
        }
      }
    }
  } else {
    // ======================= epilogue =======================
    const int q = warp & 3;                 // TMEM lane quarter: tokens 32 q .. 32 q + 31
    const int half = (warp - kWarpEpi0) >> 2;  // which share of the feature columns (kEpiWarps / 4 shares)
    constexpr int kGuCols = 128 / (kEpiWarps / 4), kDnCols = 256 / (kEpiWarps / 4);
    const uint32_t lane_bits = static_cast<uint32_t>(q * 32) << 16;
    RingPos ap;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      const Unit x = decode(tab_prefix, tab_off, E, n_tiles, u);
      if (!bounded_wait(&bars->afull[ap.slot], ap.phase, abort, args.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d = tmem + lane_bits + ap.slot * kBN;
      const int t = q * 32 + lane;
      const bool valid = t < x.nrows;
      const int row = x.row0 + t;
      const float f = (valid && args.a_outer) ? __ldg(args.a_outer + row) : 1.f;
      if (kGateUp) {
        // features n0 + half * kGuCols ..: gate in columns j, up in 128 + j
        __nv_bfloat16* dst = args.out + static_cast<size_t>(row) * args.N + x.nt * 128 + half * kGuCols;
        for (int j0 = 0; j0 < kGuCols; j0 += 16) {
          uint32_t g[16], up[16];
          tmem_ld16(d + half * kGuCols + j0, g);
          tmem_ld16(d + 128 + half * kGuCols + j0, up);
          tmem_wait_ld();
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float hv[2];
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const float gv = __uint_as_float(g[2 * i + e2]) * f;
              const float uv = __uint_as_float(up[2 * i + e2]) * f;
              hv[e2] = __fdividef(gv, 1.f + __expf(-gv)) * uv;
            }
            pk[i] = pack_bf16x2(hv[0], hv[1]);
          }
          if (valid) {
            stg128(dst + j0, pk[0], pk[1], pk[2], pk[3]);
            stg128(dst + j0 + 8, pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else {
        // features n0 + half * kDnCols ..
        __nv_bfloat16* dst = args.out + static_cast<size_t>(row) * args.N + x.nt * 256 + half * kDnCols;
        for (int j0 = 0; j0 < kDnCols; j0 += 16) {
          uint32_t v[16];
          tmem_ld16(d + half * kDnCols + j0, v);
          tmem_wait_ld();
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * f, __uint_as_float(v[2 * i + 1]) * f);
          if (valid) {
            stg128(dst + j0, pk[0], pk[1], pk[2], pk[3]);
            stg128(dst + j0 + 8, pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->aempty[ap.slot]);
      ap.advance(kAccSlots);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

constexpr size_t kSmemLimit = 232448;

inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <int WF, bool GU>
cudaError_t launch_one(const CUtensorMap* maps, const Args& a, size_t smem, int grid, cudaStream_t st) {
  auto kern = rows_gemm_kernel<WF, GU>;
  static std::atomic<uint64_t> attr{0};
  uint64_t bit;
  if (attrs_needed(attr, &bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemLimit));
    if (e != cudaSuccess) return e;
    attrs_done(attr, bit);
  }
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, maps[0], maps[1], maps[2], a);
}

template <int WF>
cudaError_t launch_kind(bool gu, const CUtensorMap* maps, const Args& a, size_t smem, int grid, cudaStream_t st) {
  return gu ? launch_one<WF, true>(maps, a, smem, grid, st) : launch_one<WF, false>(maps, a, smem, grid, st);
}

}  // namespace rows

bool rows_gemm_applicable(const mnw_moe_layer* L, int wfmt, int act, int kind) {
  const bool gu = kind == MNW_KIND_GATE_UP;
  const int N = kind == MNW_KIND_DOWN ? L->H : L->I;
  if (gu ? (N % 128) : (N % 256)) return false;
  if (wfmt == MNW_FMT_BF16) return act == MNW_ACT_BF16;
  return (wfmt == MNW_FMT_INT8_G128 || wfmt == MNW_FMT_INT4_G128) && act == kActF16Rows;
}

int run_gemm_rows(const mnw_moe_layer* L, int wfmt, int act, int kind, const void* a0, const void* a1,
                  const int32_t* offsets, int P, void* out, uint32_t* err, cudaStream_t st) {
  using namespace rows;
  const bool gu = kind == MNW_KIND_GATE_UP;
  const int K = kind == MNW_KIND_DOWN ? L->I : L->H, N = kind == MNW_KIND_DOWN ? L->H : L->I;
  Args a{};
  a.offsets = offsets;
  a.E = L->E;
  a.P = P;
  a.K = K;
  a.N = N;
  a.rows_per_tile = gu ? 128 : 256;
  a.n_tiles = N / a.rows_per_tile;
  const bool conv = wfmt != MNW_FMT_BF16;
  a.tok_slot_bytes = kTokBytes + (conv ? 0u : kWTileBytes);
  uint32_t o = 0;
  a.off_tok = o;
  o += kTokSlots * a.tok_slot_bytes;
  a.off_code = o;
  if (conv) o += kCodeSlots * kCodeBytes;
  a.off_b = o;
  if (conv) o += kBSlots * kWTileBytes;
  a.off_tab = o;
  o += align_up(2u * (L->E + 1) * 4u, 16);
  a.off_bars = align_up(o, 16);
  const size_t smem = a.off_bars + sizeof(Bars) + 1024;
  if (smem > kSmemLimit) return MNW_E_UNSUPPORTED;
  a.experts = L->blob + L->data_offset;
  a.expert_stride = L->expert_stride;
  const int m0 = kind_matrix(kind);
  a.scales_off[0] = L->scales_off[m0];
  a.scales_off[1] = L->scales_off[gu ? 1 : m0];
  a.a_outer = act == kActF16Rows ? static_cast<const float*>(a1) : nullptr;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.err = err;

  CUtensorMap maps[3];
  memset(maps, 0, sizeof(maps));
  const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(P)};
  const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
  const uint32_t box[2] = {64, static_cast<uint32_t>(kBM)};
  if (!encode_map(&maps[0], act == kActF16Rows ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  a0, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return MNW_E_INVALID_ARG;
  maps[1] = L->tm_codes[m0];
  maps[2] = gu ? L->tm_codes[1] : L->tm_codes[m0];

  const int grid = L->num_sms;
  cudaError_t e;
  if (wfmt == MNW_FMT_INT4_G128) e = launch_kind<WF_INT4>(gu, maps, a, smem, grid, st);
  else if (wfmt == MNW_FMT_INT8_G128) e = launch_kind<WF_INT8>(gu, maps, a, smem, grid, st);
  else e = launch_kind<WF_BF16>(gu, maps, a, smem, grid, st);
  return e == cudaSuccess ? MNW_OK : MNW_E_CUDA;
}

}  // namespace mnw
