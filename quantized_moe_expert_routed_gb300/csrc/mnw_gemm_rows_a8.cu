// mnw_gemm_rows_a8.cu -- the W8A8 grouped GEMMs on tcgen05 with the tokens as
// the MMA's M and 128 weight rows as its N ("row tiles", INT8 activations).
//
// The "LLaDA2.2-flash-minnow" model card, "Checkpoints and precision"
// (W8A8/W4A8 paragraph): expert inputs are quantised to signed INT8 with an
// FP32 scale per 128 values, each 128-wide group's dot product is an exact
// integer, and the groups are combined in FP32 with the weight and activation
// scales.  Here both operands' codes enter the tensor cores as exact FP16
// integers (|dot| <= 128 * 127 * 128 < 2^24, exact in the FP32 accumulator);
// every 128-K group gets its own accumulator in tensor memory, and the
// epilogue warps fold each group into FP32 running sums they keep in
// registers: sum += (s_w * s_a) * D_g, group by group in K order.
//
// Why rows: with ~64 tokens per expert, an MMA with the tokens as N (the
// weight-tile kernel) costs nearly as much at N = 64 as at N = 256; with the
// tokens as M = 128 (half of the rows empty at 64 tokens) and 128 weight rows
// as N, each MMA carries twice the weights, and the running sums no longer
// take tensor-memory columns: four accumulator slots of 128 columns fit.
//
// Roles (448 threads: 14 warps, so that no scheduler holds more than 4 and each
// thread may keep 128 registers -- the epilogue's 64 running sums need them):
//   warp 0      TMA producer: per 128-K group one code stage (128 token rows
//               and 128 weight rows of 128 INT8 codes, 128-byte swizzle); per
//               unit the weight rows' FP16 group scales and the token rows'
//               FP32 group scales (bulk copies)
//   warp 1      MMA issuer (one thread), owns the tensor memory
//   warps 2-5   converters: thread t turns token row t and weight row t of
//               each 64-K half stage into FP16 operand tiles
//   warps 6-13  epilogue: two warps per TMEM lane quarter (32 token rows),
//               each with 64 of the 128 columns (gate/up: 32 gate and the
//               same 32 up features)
// Weight tile: gate/up: gate rows n0..n0+63 then the same up rows (a unit
// makes 64 features of h); down or one matrix: 128 consecutive rows.
// Work unit (expert, feature tile, token tile of 128 rows); every wait is
// bounded (mnw_ptx.cuh).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "mnw_convert.cuh"
#include "mnw_internal.h"
#include "mnw_ptx.cuh"

namespace mnw {
namespace rowsa8 {

constexpr int kBM = 128;  // token rows per tile (MMA M)
constexpr int kBN = 128;  // weight rows per tile (MMA N)
constexpr int kConvWarps = 4, kEpiWarps = 8;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpConv0 = 2, kWarpEpi0 = kWarpConv0 + kConvWarps;
constexpr int kThreads = (kWarpEpi0 + kEpiWarps) * 32;
constexpr int kStages = 3;    // code stages (one 128-K group each)
constexpr int kOpSlots = 2;   // converted 64-K operand slots (A and B tile)
constexpr int kAccSlots = 4;  // per-group accumulators of 128 columns
constexpr int kMaxG = 16;     // K <= 2048
constexpr uint32_t kCodeTile = 128 * 128;        // 128 rows x 128 codes
constexpr uint32_t kStageBytes = 2 * kCodeTile;  // tokens + weights
constexpr uint32_t kOpTile = 128 * 128;          // 128 rows x 64 FP16
constexpr uint32_t kOpBytes = 2 * kOpTile;       // A (tokens) + B (weights)
constexpr int kTmemCols = 512;

struct Args {
  const int32_t* offsets;
  int E, P, K, N, n_tiles, G;
  const uint8_t* experts;
  uint64_t expert_stride;
  uint64_t scales_off[2];  // weight group scales of the tile's first and (gate/up) second matrix
  const float* a_scales;   // [P][G]
  __nv_bfloat16* out;
  int32_t* dots;           // nullable: [P][C][G], C = 2I (gate, then up) or N
  int dots_c, dots_c_off;  // dots row width C and a column offset
  uint32_t off_op, off_sc, off_swt, off_tab, off_bars, sc_w_bytes, sc_bytes;
  uint32_t* err;
};

struct Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t ofull[kOpSlots], oempty[kOpSlots];
  uint64_t afull[kAccSlots], aempty[kAccSlots];
  uint64_t sfull[2], sempty[2];
  uint64_t tpose[2];  // the epilogue warps' transposed weight scales are in place
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
  const int tiles = (prefix[lo + 1] - prefix[lo]) / n_tiles;
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

// warp-uniform bounded wait: every lane polls, the warp agrees on the outcome
__device__ __forceinline__ bool wwait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* err) {
  return __all_sync(0xffffffffu, bounded_wait(bar, parity, abort, err)) != 0;
}

template <bool kGateUp>
__global__ void __launch_bounds__(kThreads, 1)
    rows_a8_kernel(const __grid_constant__ CUtensorMap tmTok, const __grid_constant__ CUtensorMap tmW0,
                   const __grid_constant__ CUtensorMap tmW1, const Args args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + args.off_bars);
  int* tab_prefix = reinterpret_cast<int*>(smem + args.off_tab);
  int* tab_off = tab_prefix + (args.E + 1);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E, G = args.G, n_tiles = args.n_tiles;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], kConvWarps);
    }
    for (int i = 0; i < kOpSlots; ++i) {
      mbar_init(&bars->ofull[i], kConvWarps);
      mbar_init(&bars->oempty[i], 1);
    }
    for (int i = 0; i < kAccSlots; ++i) {
      mbar_init(&bars->afull[i], 1);
      mbar_init(&bars->aempty[i], kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->sfull[i], 1);
      mbar_init(&bars->sempty[i], kEpiWarps);
      mbar_init(&bars->tpose[i], kEpiWarps);
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
  uint8_t* op_ring = smem + args.off_op;
  uint8_t* sc_ring = smem + args.off_sc;

  if (warp == kWarpTma) {
    // ======================= producer =======================
    if (lane == 0) {
      RingPos sp;
      uint32_t issued = 0, s_issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const Unit x = decode(tab_prefix, tab_off, E, n_tiles, u);
        const int n0 = x.nt * (kGateUp ? 64 : kBN);
        // the unit's scales: weight rows [128][G] FP16, then token rows [nrows][G] FP32
        const uint32_t sb = s_issued & 1u;
        if (!bounded_wait(&bars->sempty[sb], ((s_issued >> 1) & 1u) ^ 1u, abort, args.err)) { ok = false; break; }
        uint8_t* sc = sc_ring + sb * args.sc_bytes;
        const uint32_t wbytes = (kGateUp ? 64u : 128u) * G * 2u;
        const uint32_t abytes = static_cast<uint32_t>(x.nrows) * G * 4u;
        mbar_arrive_expect_tx(&bars->sfull[sb], (kGateUp ? 2u : 1u) * wbytes + abytes);
        const uint8_t* eb = args.experts + static_cast<uint64_t>(x.e) * args.expert_stride;
        bulk_load(sc, eb + args.scales_off[0] + static_cast<uint64_t>(n0) * G * 2, wbytes, &bars->sfull[sb]);
        if (kGateUp) bulk_load(sc + wbytes, eb + args.scales_off[1] + static_cast<uint64_t>(n0) * G * 2, wbytes,
                               &bars->sfull[sb]);
        bulk_load(sc + args.sc_w_bytes, args.a_scales + static_cast<size_t>(x.row0) * G, abytes, &bars->sfull[sb]);
        ++s_issued;
        for (int g = 0; g < G; ++g, sp.advance(kStages)) {
          if (!bounded_wait(&bars->empty[sp.slot], sp.phase ^ 1u, abort, args.err)) { ok = false; break; }
          uint8_t* st = smem + sp.slot * kStageBytes;
          mbar_arrive_expect_tx(&bars->full[sp.slot], kStageBytes);
          tma_load_2d(st, &tmTok, &bars->full[sp.slot], g * 128, x.row0);
          if (kGateUp) {
            tma_load_3d(st + kCodeTile, &tmW0, &bars->full[sp.slot], g * 128, n0, x.e);
            tma_load_3d(st + kCodeTile + 64 * 128, &tmW1, &bars->full[sp.slot], g * 128, n0, x.e);
          } else {
            tma_load_3d(st + kCodeTile, &tmW0, &bars->full[sp.slot], g * 128, n0, x.e);
          }
          ++issued;
        }
      }
      if (!ok || *abort) {
        for (uint32_t j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
          drain_wait(&bars->full[j % kStages], (j / kStages) & 1);
        for (uint32_t j = s_issued > 2 ? s_issued - 2 : 0; j < s_issued; ++j)
          drain_wait(&bars->sfull[j & 1], (j >> 1) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kBM, kBN, false);
      RingPos op, ap;
      bool ok = true, issued = false;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        for (int g = 0; ok && g < G; ++g) {
          if (!bounded_wait(&bars->aempty[ap.slot], ap.phase ^ 1u, abort, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + ap.slot * kBN;
          for (int h = 0; h < 2; ++h) {
            if (!bounded_wait(&bars->ofull[op.slot], op.phase, abort, args.err)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a_tile = smem_u32(op_ring + op.slot * kOpBytes);
            const uint32_t b_tile = a_tile + kOpTile;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(d, sdesc_sw128(a_tile + kk * 32), sdesc_sw128(b_tile + kk * 32), idesc, (h | kk) != 0);
            issued = true;
            mma_commit(&bars->oempty[op.slot]);
            op.advance(kOpSlots);
          }
          if (!ok) break;
          mma_commit(&bars->afull[ap.slot]);
          ap.advance(kAccSlots);
        }
      }
      if (issued) {
        mma_commit(&bars->final_mma);
        drain_wait(&bars->final_mma, 0);
      }
    }
  } else if (warp < kWarpEpi0) {
    // ======================= converters =======================
    // thread r: token row r (the stage's first tile) and weight row r (its second)
    const int r = (warp - kWarpConv0) * 32 + lane;
    RingPos sp, op;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      for (int g = 0; ok && g < G; ++g, sp.advance(kStages)) {
        if (!bounded_wait(&bars->full[sp.slot], sp.phase, abort, args.err)) { ok = false; break; }
        const uint32_t src = smem_u32(smem + sp.slot * kStageBytes);
        for (int h = 0; h < 2; ++h) {
          if (!bounded_wait(&bars->oempty[op.slot], op.phase ^ 1u, abort, args.err)) { ok = false; break; }
          const uint32_t dst = smem_u32(op_ring + op.slot * kOpBytes);
#pragma unroll
          for (int m = 0; m < 2; ++m) {  // tokens, then weights
            // 64 codes: chunks 4h .. 4h+3 of the 128-byte row
            uint4 v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) v[c] = lds128(sw128(src + m * kCodeTile, r, 4 * h + c));
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              uint32_t o[16];
              cvt_int8x32<false>(v[2 * c2], v[2 * c2 + 1], o);  // 32 codes -> 32 FP16 integers
#pragma unroll
              for (int ch = 0; ch < 4; ++ch)
                sts128(sw128(dst + m * kOpTile, r, 4 * c2 + ch), o[4 * ch], o[4 * ch + 1], o[4 * ch + 2],
                       o[4 * ch + 3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->ofull[op.slot]);
          op.advance(kOpSlots);
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->empty[sp.slot]);
      }
    }
  } else {
    // ======================= epilogue =======================
    const int q = warp & 3;                          // TMEM lane quarter: token rows 32q .. 32q+31
    const int hf = (warp - kWarpEpi0) >> 2;          // which 64 of the 128 columns
    const uint32_t lane_bits = static_cast<uint32_t>(q * 32) << 16;
    const int tr = q * 32 + lane;                    // token row in the tile
    // columns: gate/up: gate 32hf .. +31 and up 64 + 32hf .. +31; else 64hf .. +63
    const int ca = kGateUp ? 32 * hf : 64 * hf;
    const int cb = kGateUp ? 64 + 32 * hf : 64 * hf + 32;
    RingPos ap;
    uint32_t s_used = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      const Unit x = decode(tab_prefix, tab_off, E, n_tiles, u);
      const int n0 = x.nt * (kGateUp ? 64 : kBN);
      const bool valid = tr < x.nrows;
      const uint32_t sb = s_used & 1u;
      if (!wwait(&bars->sfull[sb], (s_used >> 1) & 1u, abort, args.err)) { ok = false; break; }
      const __half* sw = reinterpret_cast<const __half*>(sc_ring + sb * args.sc_bytes);   // [128 weight rows][G]
      const float* sa = reinterpret_cast<const float*>(sc_ring + sb * args.sc_bytes + args.sc_w_bytes) + tr * G;
      // the weight scales transposed to FP32 [G][128 columns], so that a group's 64 column
      // scales of a warp are 16 broadcast 16-byte loads; buffer sb is free: every epilogue
      // warp finished unit u - 2 before the producer refilled scale buffer sb
      float* swt = reinterpret_cast<float*>(smem + args.off_swt) + sb * (kMaxG * 128);
      for (int i = (warp - kWarpEpi0) * 32 + lane; i < 128 * G; i += kEpiWarps * 32)
        swt[i] = __half2float(sw[(i & 127) * G + (i >> 7)]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tpose[sb]);
      if (!wwait(&bars->tpose[sb], (s_used >> 1) & 1u, abort, args.err)) { ok = false; break; }
      uint64_t sum2[32];  // the 64 running sums as FP32 pairs (packed FMAs, each lane as the scalar one)
#pragma unroll
      for (int c = 0; c < 32; ++c) sum2[c] = 0ull;
      for (int g = 0; g < G; ++g) {
        if (!wwait(&bars->afull[ap.slot], ap.phase, abort, args.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + lane_bits + ap.slot * kBN;
        const float s_a = valid ? sa[g] : 0.f;
        const uint64_t sa2 = f32x2_pack(__float_as_uint(s_a), __float_as_uint(s_a));
        // four chunks of 16 columns: the gate (or first) half, then the up (or second) half
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int cbase = ch < 2 ? ca + 16 * ch : cb + 16 * (ch - 2);  // tile column = weight row of the tile
          uint32_t acc[16];
          tmem_ld16(d + cbase, acc);
          tmem_wait_ld();
          if (args.dots && valid) {
            int32_t* dr = args.dots + static_cast<size_t>(x.row0 + tr) * args.dots_c * G;
            for (int i = 0; i < 16; ++i) {
              const int col = cbase + i;
              const int gcol = kGateUp ? (col < 64 ? n0 + col : args.N + n0 + (col - 64)) : n0 + col;
              dr[static_cast<size_t>(args.dots_c_off + gcol) * G + g] = __float2int_rn(__uint_as_float(acc[i]));
            }
          }
          const uint64_t* wg2 = reinterpret_cast<const uint64_t*>(swt + g * 128 + cbase);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint64_t f2 = f32x2_mul(wg2[i], sa2);  // fl(s_w * s_a), two columns
            sum2[8 * ch + i] = f32x2_fma(f2, f32x2_pack(acc[2 * i], acc[2 * i + 1]), sum2[8 * ch + i]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->aempty[ap.slot]);
        ap.advance(kAccSlots);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->sempty[sb]);
      ++s_used;
      if (valid) {
        __nv_bfloat16* dst = args.out + static_cast<size_t>(x.row0 + tr) * args.N;
        if (kGateUp) {
          // h features n0 + 32hf .. +31: SiLU(gate) * up
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float hv[2];
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const uint64_t gp = sum2[i], upp = sum2[16 + i];
              const float gv = __uint_as_float(static_cast<uint32_t>(gp >> (32 * e2)));
              const float uv = __uint_as_float(static_cast<uint32_t>(upp >> (32 * e2)));
              hv[e2] = __fdividef(gv, 1.f + __expf(-gv)) * uv;
            }
            pk[i] = pack_bf16x2(hv[0], hv[1]);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            stg128(dst + n0 + 32 * hf + 8 * i, pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        } else {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(sum2[i])),
                                __uint_as_float(static_cast<uint32_t>(sum2[i] >> 32)));
#pragma unroll
          for (int i = 0; i < 8; ++i)
            stg128(dst + n0 + 64 * hf + 8 * i, pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
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

constexpr size_t kSmemLimit = 232448;

inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <bool GU>
cudaError_t launch_one(const CUtensorMap* maps, const Args& a, size_t smem, int grid, cudaStream_t st) {
  auto kern = rows_a8_kernel<GU>;
  static std::atomic<uint64_t> attr{0};
  uint64_t bit;
  if (attrs_needed(attr, &bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemLimit));
    if (e != cudaSuccess) return e;
    attrs_done(attr, bit);
  }
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, maps[0], maps[1], maps[2], a);
}

}  // namespace rowsa8

bool rows_a8_applicable(const mnw_moe_layer* L, int wfmt, int act, int kind) {
  if (wfmt != MNW_FMT_INT8_G128 || act != MNW_ACT_INT8_G128) return false;
  const int K = kind == MNW_KIND_DOWN ? L->I : L->H;
  const int N = kind == MNW_KIND_DOWN ? L->H : L->I;
  // K: whole 128-groups, at most kMaxG of them (larger K: the weight-tile kernel), and a multiple of 4 groups (the token
  // rows' FP32 group scales then fill whole 16-byte units for the bulk copy)
  if (K % 512 || K / 128 > rowsa8::kMaxG) return false;
  return kind == MNW_KIND_GATE_UP ? N % 64 == 0 : N % 128 == 0;
}

int run_gemm_rows_a8(const mnw_moe_layer* L, int kind, const void* a_codes, const float* a_scales,
                     const int32_t* offsets, int P, void* out, int32_t* dots, uint32_t* err, cudaStream_t st) {
  using namespace rowsa8;
  const bool gu = kind == MNW_KIND_GATE_UP;
  const int K = kind == MNW_KIND_DOWN ? L->I : L->H, N = kind == MNW_KIND_DOWN ? L->H : L->I;
  Args a{};
  a.offsets = offsets;
  a.E = L->E;
  a.P = P;
  a.K = K;
  a.N = N;
  a.G = K / 128;
  a.n_tiles = N / (gu ? 64 : kBN);
  a.experts = L->blob + L->data_offset;
  a.expert_stride = L->expert_stride;
  const int m0 = kind_matrix(kind);
  a.scales_off[0] = L->scales_off[m0];
  a.scales_off[1] = L->scales_off[gu ? 1 : m0];
  a.a_scales = a_scales;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.dots = dots;
  // the dots layout of the ABI: [P][C][G], C = 2I for the gate/up pair (gate columns, then up), else N
  a.dots_c = gu ? 2 * N : N;
  a.dots_c_off = 0;
  a.err = err;
  // shared memory: code stages | operand slots | scale buffers (x2) | unit table | barriers
  a.sc_w_bytes = align_up(128u * a.G * 2u, 16);
  a.sc_bytes = align_up(a.sc_w_bytes + 128u * a.G * 4u, 128);
  uint32_t o = kStages * kStageBytes;
  a.off_op = o;
  o += kOpSlots * kOpBytes;
  a.off_sc = o;
  o += 2 * a.sc_bytes;
  a.off_swt = o;
  o += 2 * kMaxG * 128 * 4;
  a.off_tab = o;
  o += align_up(2u * (L->E + 1) * 4u, 16);
  a.off_bars = align_up(o, 16);
  const size_t smem = a.off_bars + sizeof(Bars) + 1024;
  if (smem > kSmemLimit) return MNW_E_UNSUPPORTED;

  CUtensorMap maps[3];
  memset(maps, 0, sizeof(maps));
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(P)};
    const uint64_t strides[1] = {static_cast<uint64_t>(K)};
    const uint32_t box[2] = {128, static_cast<uint32_t>(kBM)};
    if (!encode_map(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a_codes, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
      return MNW_E_INVALID_ARG;
  }
  if (gu) {
    // 64-row boxes of the gate and up codes
    const uint8_t* experts = L->blob + L->data_offset;
    for (int m = 0; m < 2; ++m) {
      const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(L->E)};
      const uint64_t strides[2] = {static_cast<uint64_t>(K), L->expert_stride};
      const uint32_t box[3] = {128, 64, 1};
      if (!encode_map(&maps[1 + m], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, experts + L->codes_off[m], dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return MNW_E_INVALID_ARG;
    }
  } else {
    maps[1] = L->tm_codes[m0];
    maps[2] = L->tm_codes[m0];
  }
  const int grid = L->num_sms;
  const cudaError_t e = gu ? launch_one<true>(maps, a, smem, grid, st) : launch_one<false>(maps, a, smem, grid, st);
  return e == cudaSuccess ? MNW_OK : MNW_E_CUDA;
}

}  // namespace mnw
