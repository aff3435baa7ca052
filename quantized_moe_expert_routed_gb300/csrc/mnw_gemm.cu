// mnw_gemm.cu -- grouped expert GEMMs on the 5th-generation tensor cores.
//
// One persistent kernel template covers every format and mode of the
// "LLaDA2.2-flash-minnow" model card's precision table (and the activation
// modes of the coder543/minnow README, "Quantization"):
//
//   weights BF16  + activations BF16   (A from smem via TMA,            BF16 MMA)
//   weights INT8/INT4 + BF16            (codes as exact BF16 integers in TMEM,
//                                        one accumulator per 128-group, FP16 group
//                                        scale applied in FP32)
//   weights INT8/INT4 + INT8 per 128    (codes as exact FP16 integers in TMEM/smem,
//                                        INT32-exact group dots, FP32 rescale by s_w*s_a)
//   weights NVFP4 + NVFP4               (E2M1 codes straight from shared memory into
//                                        the block-scaled FP4 MMA, E4M3 scales per 16
//                                        in tensor memory, FP32 outer scales applied
//                                        in the epilogue)
//
// Dequantisation happens in registers on the way into the tensor cores; no
// expanded weight copy exists in memory.  INT codes are exact in BF16/FP16, so
// the weights themselves are never rounded: each 128-wide group's dot product
// is accumulated in FP32 on the tensor cores (exact for INT8 activations,
// since |D| < 2^24) and is scaled and summed in FP32.
//
// Layout of the problem ("swap AB"): the weight matrix supplies the M = 128
// rows of the MMA (128 output features per tile) and the tokens routed to one
// expert supply N (16..128 columns).  Decode batches route only a few tokens
// to each expert, so this keeps the MMA full while the weights stream
// through once.  A work unit is (expert, token tile of BN rows, 128-feature
// tile); every CTA walks units blockIdx.x, blockIdx.x + gridDim.x, ... over
// the device-side tile table built from expert_offsets (no host sync).
//
// Warp roles (576 threads):
//   warp 0      TMA producer: weight tiles (raw codes) + group scales + token tiles
//   warp 1      MMA issuer (one thread); owns the TMEM allocation
//   warps 2-9   converters: raw weight codes -> BF16/FP16 operand in TMEM
//               (tcgen05.st); INT8 token codes -> FP16 operand in shared memory.
//               NVFP4: warps 2-5 move each stage's E4M3 block scales of weights
//               and tokens into tensor memory for the block-scaled MMA; the
//               codes themselves are MMA operands as the TMA left them.
//   warps 10-17 epilogue: TMEM accumulators -> (group rescale) -> SiLU(g)*u or y
//               -> BF16 global; two warps per TMEM lane quarter, each with half
//               of the token columns
//
// TMEM (512 columns): operand-A ring (slots of 64 K per matrix), then the
// accumulators; in the grouped modes two per-group accumulators (one drains
// while the next fills) and the FP32 running sum.  With BF16 weights A never
// enters TMEM and the accumulators may use all 512 columns.  NVFP4: the
// accumulators, then a ring of scale-factor slots, one per stage.
//
// Every wait is bounded (mnw_ptx.cuh); on a timeout all roles leave their
// loops, outstanding copies and MMAs are drained with a time limit, TMEM is
// freed and MNW_DEVERR_TIMEOUT is reported through the error word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdio>

#include "mnw_convert.cuh"
#include "mnw_internal.h"
#include "mnw_ptx.cuh"

namespace mnw {

enum { WF_BF16 = 0, WF_INT8 = 1, WF_INT4 = 2, WF_NVFP4 = 3 };
// AM_F16S: activations already in FP16 with a power-of-two factor per row
// (launch_gather_f16); INT weights are dequantised to FP16 q * s by the
// converters, so one accumulator covers the whole K (used by the forward path).
enum { AM_BF16 = 0, AM_INT8 = 1, AM_FP4 = 2, AM_F16S = 3 };

constexpr int kBM = 128;
constexpr int kConvWarps = 8;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each taking half the token columns
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpConv0 = 2, kWarpEpi0 = kWarpConv0 + kConvWarps;
constexpr int kThreads = (kWarpEpi0 + kEpiWarps) * 32;
constexpr int kMaxStages = 8;
constexpr int kMaxASlots = 8;   // operand-A ring slots in TMEM (runtime count <= this)
constexpr int kMaxAcc = 8;      // accumulator slots (runtime count <= this)
constexpr int kBSlots = 4;      // converted-token ring slots (INT8 activations)
constexpr int kMaxSf = 8;       // scale-factor ring slots in TMEM (NVFP4; runtime count <= this)
constexpr int kSfWarps = 4;     // NVFP4: converter warps that move block scales into TMEM, one per lane quarter
constexpr int kTmemCols = 512;


struct GemmArgs {
  const int32_t* offsets;
  int E, P, K, N, BN, n_tiles, stages, nmat, acc_slots, acc_base, aslots, sum_base;
  int sf_base, sf_slots, sf_cols;  // NVFP4: TMEM scale-factor ring (first column, slots, columns per slot)
  uint32_t stage_bytes, off_a[2], off_asf[2], off_b, off_braw, off_bsf, off_bring;
  uint32_t off_scales, scale_mat_bytes, off_tab, off_sa, off_bars;
  const uint8_t* experts;
  uint64_t expert_stride;
  uint64_t scales_off[2], outer_off[2];
  const float* a_scales;
  const float* a_outer;
  __nv_bfloat16* out;
  int32_t* dots;
  uint32_t* err;
};

struct Bars {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t bfull[kBSlots], bempty[kBSlots];  // converted-token ring
  uint64_t afull[kMaxASlots], aempty[kMaxASlots];
  uint64_t accfull[kMaxAcc], accempty[kMaxAcc];
  uint64_t sfull[2], sempty[2];
  uint64_t sffull[kMaxSf], sfempty[kMaxSf];  // NVFP4 scale factors in TMEM
  uint64_t final_mma;
  uint32_t tmem_base;
  int abort;
};

template <int WF>
struct WT {
  static constexpr int kStage = WF == WF_BF16 ? 64 : (WF == WF_INT8 ? 128 : 256);  // K per stage
  static constexpr int kSub = kStage / 64;                                          // 64-K sub-chunks
  static constexpr bool kTs = WF == WF_INT8 || WF == WF_INT4;                        // A from TMEM
  static constexpr bool kScales = WF == WF_INT8 || WF == WF_INT4;                    // FP16 group scales
};

// ---------------------------------------------------------------------------
// work decomposition
// ---------------------------------------------------------------------------

struct Unit {
  int e, tt, nt, row0, nrows;
};

__device__ __forceinline__ Unit decode_unit(const int* tab_prefix, const int* tab_off, int E, int n_tiles, int BN,
                                            int u) {
  Unit x;
  const int t = u / n_tiles;
  x.nt = u - t * n_tiles;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tab_prefix[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  x.e = lo;
  x.tt = t - tab_prefix[lo];
  x.row0 = tab_off[lo] + x.tt * BN;
  x.nrows = min(BN, tab_off[lo + 1] - x.row0);
  return x;
}

// Position in a ring of n slots: the slot and the parity of its current use,
// advanced without a division.  The MMA-issuing thread runs alone and every
// instruction between two MMAs delays the next one, so none of the rings of
// this kernel is indexed with a runtime modulo.
struct RingPos {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void advance(uint32_t n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Drain wait used on the way out: ignores the abort flag, bounded in time.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <int WF, int AM, bool kGateUp>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmS1,
                    const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBs,
                    const GemmArgs args) {
  using T = WT<WF>;
  constexpr int kNmat = kGateUp ? 2 : 1;
  constexpr bool kBconv = AM == AM_INT8;                  // tokens converted by the converter warps
  constexpr bool kFp4 = WF == WF_NVFP4;                   // block-scaled FP4 MMA on the raw codes
  constexpr bool kScaleConv = AM == AM_F16S;              // converters apply the FP16 group scales
  // Grouped: one accumulator per 128-wide K group, rescaled in FP32 (INT weights).
  constexpr bool kGrouped = AM == AM_INT8 || (AM == AM_BF16 && T::kScales);
  constexpr bool kBf16Mma = AM == AM_BF16;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + args.off_bars);
  int* tab_prefix = reinterpret_cast<int*>(smem + args.off_tab);
  int* tab_off = tab_prefix + (args.E + 1);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E, BN = args.BN, S = args.stages;
  const int nks = args.K / T::kStage;
  const int G = args.K / 128;

  // ---- set-up ----
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], ((T::kTs || kBconv) ? kConvWarps : (kFp4 ? kSfWarps : 0)) + 1);
    }
    for (int i = 0; i < kBSlots; ++i) {
      mbar_init(&bars->bfull[i], kConvWarps);
      mbar_init(&bars->bempty[i], 1);
    }
    for (int i = 0; i < kMaxASlots; ++i) {
      mbar_init(&bars->afull[i], kConvWarps);
      mbar_init(&bars->aempty[i], 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(&bars->accfull[i], 1);
      mbar_init(&bars->accempty[i], kEpiWarps);
    }
    for (int i = 0; i < kMaxSf; ++i) {
      mbar_init(&bars->sffull[i], kSfWarps);
      mbar_init(&bars->sfempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->sfull[i], 1);
      mbar_init(&bars->sempty[i], kScaleConv ? kConvWarps : kEpiWarps);
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
    tma_prefetch_desc(&tmA0);
    if (kGateUp) tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB);
    if (kFp4) {
      tma_prefetch_desc(&tmS0);
      if (kGateUp) tma_prefetch_desc(&tmS1);
      tma_prefetch_desc(&tmBs);
    }
  }
  // everything below reads or writes global memory the previous kernel may own
  pdl_wait();
  // Tile table: tab_prefix[e] = first tile of expert e, tab_off = expert_offsets.
  if (warp == 2) {
    const int per = (E + 31) / 32;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        const int o0 = __ldg(args.offsets + e), o1 = __ldg(args.offsets + e + 1);
        tab_off[e] = o0;
        local += max(0, (o1 - o0 + BN - 1) / BN);
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
        const int o0 = tab_off[e], o1 = __ldg(args.offsets + e + 1);
        run += max(0, (o1 - o0 + BN - 1) / BN);
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
  const int units = tab_prefix[E] * args.n_tiles;

  if (warp == kWarpTma) {
    // ======================= producer =======================
    if (lane == 0) {
      uint32_t it = 0, uit = 0, sit = 0;  // stages issued, units visited, scale loads issued
      RingPos sp;
      bool ok = true;
      const uint32_t a_bytes = kNmat * 16384u + (WF == WF_NVFP4 ? kNmat * 2048u : 0u);
      uint32_t b_bytes;
      if (AM == AM_BF16 || AM == AM_F16S) b_bytes = T::kSub * BN * 128u;
      else if (AM == AM_INT8) b_bytes = (T::kStage / 128) * BN * 128u;
      else b_bytes = BN * 128u + BN * 16u;
      const uint32_t tx = a_bytes + b_bytes;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++uit) {
        const Unit x = decode_unit(tab_prefix, tab_off, E, args.n_tiles, BN, u);
        const int n0 = x.nt * kBM;
        if (T::kScales) {
          const uint32_t sb = uit & 1;
          if (!bounded_wait(&bars->sempty[sb], ((uit >> 1) & 1) ^ 1, abort, args.err)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars->sfull[sb], kNmat * args.scale_mat_bytes);
          for (int m = 0; m < kNmat; ++m) {
            const uint8_t* src = args.experts + static_cast<uint64_t>(x.e) * args.expert_stride +
                                 args.scales_off[m] + static_cast<uint64_t>(n0) * G * 2;
            bulk_load(smem + args.off_scales + (sb * kNmat + m) * args.scale_mat_bytes, src, args.scale_mat_bytes,
                      &bars->sfull[sb]);
          }
          ++sit;
        }
        for (int ks = 0; ks < nks; ++ks, ++it, sp.advance(S)) {
          const int s = sp.slot;
          if (!bounded_wait(&bars->empty[s], sp.phase ^ 1, abort, args.err)) { ok = false; break; }
          uint8_t* st = smem + s * args.stage_bytes;
          mbar_arrive_expect_tx(&bars->full[s], tx);
          const int kx = WF == WF_BF16 ? ks * 64 : ks * 128;  // elements (BF16) or bytes (codes)
          tma_load_3d(st + args.off_a[0], &tmA0, &bars->full[s], kx, n0, x.e);
          if (kGateUp) tma_load_3d(st + args.off_a[1], &tmA1, &bars->full[s], kx, n0, x.e);
          if (WF == WF_NVFP4) {
            tma_load_3d(st + args.off_asf[0], &tmS0, &bars->full[s], ks * 16, n0, x.e);
            if (kGateUp) tma_load_3d(st + args.off_asf[1], &tmS1, &bars->full[s], ks * 16, n0, x.e);
          }
          if (AM == AM_BF16 || AM == AM_F16S) {
            for (int b = 0; b < T::kSub; ++b)
              tma_load_2d(st + args.off_b + b * BN * 128, &tmB, &bars->full[s], ks * T::kStage + b * 64, x.row0);
          } else if (AM == AM_INT8) {
            for (int b = 0; b < T::kStage / 128; ++b)
              tma_load_2d(st + args.off_braw + b * BN * 128, &tmB, &bars->full[s], ks * T::kStage + b * 128,
                          x.row0);
          } else {
            tma_load_2d(st + args.off_braw, &tmB, &bars->full[s], ks * 128, x.row0);
            tma_load_2d(st + args.off_bsf, &tmBs, &bars->full[s], ks * 16, x.row0);
          }
        }
      }
      if (!ok || *abort) {
        // Let every copy already issued land before the CTA exits.
        const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
        for (uint32_t j = first; j < it; ++j) drain_wait(&bars->full[j % S], (j / S) & 1);
        if (T::kScales)
          for (uint32_t j = sit > 2 ? sit - 2 : 0; j < sit; ++j) drain_wait(&bars->sfull[j & 1], (j >> 1) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ======================= MMA issuer =======================
    if (lane == 0 && kFp4) {
      // Block-scaled FP4: per stage, both operands as the TMA left them (128-byte
      // rows of 256 E2M1 codes) and the stage's scale factors in TMEM slot fp;
      // 4 MMAs of K = 64 per matrix.
      const uint32_t idesc = idesc_fp4(kBM, BN);
      const uint32_t S_ = static_cast<uint32_t>(S), nacc = static_cast<uint32_t>(args.acc_slots),
                     nsf = static_cast<uint32_t>(args.sf_slots);
      RingPos sp, cp, fp;  // stages, accumulator slots, scale-factor slots
      bool ok = true, issued = false;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        if (!bounded_wait(&bars->accempty[cp.slot], cp.phase ^ 1, abort, args.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_base = tmem + args.acc_base + cp.slot * kNmat * BN;
        for (int ks = 0; ks < nks; ++ks, sp.advance(S_), fp.advance(nsf)) {
          const int s = sp.slot;
          if (!bounded_wait(&bars->full[s], sp.phase, abort, args.err) ||
              !bounded_wait(&bars->sffull[fp.slot], fp.phase, abort, args.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * args.stage_bytes);
          // [SFA m0 | SFA m1]: 16 columns each; SFB: 8 columns per 64-K step
          const uint32_t sf = tmem + args.sf_base + fp.slot * args.sf_cols;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = sdesc_sw128(st + args.off_braw + kk * 32);
            const uint32_t acc = (ks != 0 || kk != 0);
#pragma unroll
            for (int m = 0; m < kNmat; ++m)
              mma_fp4_ss(d_base + m * BN, sdesc_sw128(st + args.off_a[m] + kk * 32), bdesc, idesc, sf + m * 16 + kk * 4,
                         sf + kNmat * 16 + kk * 8, acc);
          }
          issued = true;
          mma_commit(&bars->sfempty[fp.slot]);
          mma_commit(&bars->empty[s]);
        }
        if (!ok) break;
        mma_commit(&bars->accfull[cp.slot]);
        cp.advance(nacc);
      }
      if (issued) {
        mma_commit(&bars->final_mma);
        drain_wait(&bars->final_mma, 0);
      }
    } else if (lane == 0) {
      const uint32_t idesc = idesc_f16(kBM, BN, kBf16Mma);
      const uint32_t S_ = static_cast<uint32_t>(S), na = static_cast<uint32_t>(args.aslots),
                     nacc = static_cast<uint32_t>(args.acc_slots);
      RingPos sp, ap, cp, bp;  // stages, operand-A slots, accumulator slots, token slots
      bool ok = true, issued = false;
      uint32_t d_base = 0;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        if (!kGrouped) {
          if (!bounded_wait(&bars->accempty[cp.slot], cp.phase ^ 1, abort, args.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          d_base = tmem + args.acc_base + cp.slot * kNmat * BN;
        }
        for (int ks = 0; ok && ks < nks; ++ks, sp.advance(S_)) {
          const int s = sp.slot;
          // with converted tokens both operands come from rings; the stage itself is not read here
          if (!kBconv) {
            if (!bounded_wait(&bars->full[s], sp.phase, abort, args.err)) { ok = false; break; }
            tc_fence_after();
          }
          const uint32_t st = smem_u32(smem + s * args.stage_bytes);
          for (int sc = 0; sc < T::kSub; ++sc) {
            const int kg = ks * T::kStage + sc * 64;
            if (kGrouped) {
              if ((kg & 127) == 0) {
                if (!bounded_wait(&bars->accempty[cp.slot], cp.phase ^ 1, abort, args.err)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              d_base = tmem + args.acc_base + cp.slot * kNmat * BN;
            }
            const uint32_t aslot = ap.slot;
            if (T::kTs) {
              if (!bounded_wait(&bars->afull[aslot], ap.phase, abort, args.err)) { ok = false; break; }
              tc_fence_after();
            }
            uint32_t b_tile = st + args.off_b + sc * BN * 128;
            const uint32_t bslot = bp.slot;
            if (kBconv) {
              if (!bounded_wait(&bars->bfull[bslot], bp.phase, abort, args.err)) { ok = false; break; }
              tc_fence_after();
              b_tile = smem_u32(smem + args.off_bring) + bslot * BN * 128;
            }
            const uint32_t a_tmem = tmem + aslot * (kNmat * 32);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bdesc = sdesc_sw128(b_tile + kk * 32);
              const uint32_t acc = kGrouped ? ((kg & 127) != 0 || kk != 0) : (ks != 0 || sc != 0 || kk != 0);
#pragma unroll
              for (int m = 0; m < kNmat; ++m) {
                if (T::kTs) {
                  mma_ts(d_base + m * BN, a_tmem + m * 32 + kk * 8, bdesc, idesc, acc);
                } else {
                  mma_ss(d_base + m * BN, sdesc_sw128(st + args.off_a[m] + kk * 32), bdesc, idesc, acc);
                }
              }
            }
            issued = true;
            if (T::kTs) {
              mma_commit(&bars->aempty[aslot]);
              ap.advance(na);
            }
            if (kBconv) {
              mma_commit(&bars->bempty[bslot]);
              bp.advance(kBSlots);
            }
            if (kGrouped && ((kg + 64) & 127) == 0) {
              mma_commit(&bars->accfull[cp.slot]);
              cp.advance(nacc);
            }
          }
          if (!ok) break;
          mma_commit(&bars->empty[s]);
        }
        if (ok && !kGrouped) {
          mma_commit(&bars->accfull[cp.slot]);
          cp.advance(nacc);
        }
      }
      if (issued) {
        mma_commit(&bars->final_mma);
        drain_wait(&bars->final_mma, 0);
      }
    }
  } else if (warp < kWarpEpi0) {
    // ======================= converters =======================
    const int cw = warp - kWarpConv0;   // 0..7
    const int q = warp & 3;             // TMEM lane quarter this warp may access
    const int h = cw >> 2;              // which 32-K half of each 64-K sub-chunk
    const int r = q * 32 + lane;        // weight row within the tile
    const int ctid = cw * 32 + lane;    // 0..255
    const uint32_t S_ = static_cast<uint32_t>(S), na = static_cast<uint32_t>(args.aslots);
    RingPos sp, ap, bp;  // stages, operand-A slots, token slots
    bool ok = true;
    if (kFp4 && cw < kSfWarps) {
      // Block scales of one stage (256 K: four 64-K MMA steps) into TMEM slot fp.
      // A (weights): lane quarter q holds rows 32q..32q+31; row r's four scales
      // of step kk (one 32-bit word, first 16 K in the low byte) go to the four
      // columns m*16 + 4kk .. +3 of lane r.  B (tokens): every lane quarter
      // holds all BN (<= 256) token rows, token 32j + l in lane l of column
      // 16 nmat + 8kk + j; rows past BN read as zero.
      const uint32_t nsf = static_cast<uint32_t>(args.sf_slots);
      const uint32_t lane_bits = static_cast<uint32_t>(q * 32) << 16;
      RingPos fp;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        for (int ks = 0; ks < nks; ++ks, sp.advance(S_), fp.advance(nsf)) {
          const int s = sp.slot;
          if (!bounded_wait(&bars->full[s], sp.phase, abort, args.err) ||
              !bounded_wait(&bars->sfempty[fp.slot], fp.phase ^ 1, abort, args.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * args.stage_bytes);
          const uint32_t sf = tmem + lane_bits + args.sf_base + fp.slot * args.sf_cols;
          uint32_t o[16];
#pragma unroll
          for (int m = 0; m < kNmat; ++m) {
            const uint4 v = lds128(st + args.off_asf[m] + r * 16);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = w[i >> 2];
            tmem_st16(sf + m * 16, o);
          }
          uint4 tv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int row = 32 * j + lane;
            tv[j] = row < BN ? lds128(st + args.off_bsf + row * 16) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int hk = 0; hk < 2; ++hk) {  // steps 2hk and 2hk + 1: 16 columns
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
              const int kk = 2 * hk + k2;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const uint4 v = tv[j];
                o[k2 * 8 + j] = kk == 0 ? v.x : (kk == 1 ? v.y : (kk == 2 ? v.z : v.w));
              }
            }
            tmem_st16(sf + kNmat * 16 + hk * 16, o);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bars->sffull[fp.slot]);
            mbar_arrive(&bars->empty[s]);
          }
        }
      }
    } else if (T::kTs || kBconv) {
      for (uint32_t uit = 0, u = blockIdx.x; ok && static_cast<int>(u) < units; u += gridDim.x, ++uit) {
        // FP16 operand mode: this unit's FP16 group scales, applied here to the weights
        const uint32_t sbuf = uit & 1;
        if (kScaleConv && !bounded_wait(&bars->sfull[sbuf], (uit >> 1) & 1, abort, args.err)) { ok = false; break; }
        for (int ks = 0; ks < nks; ++ks, sp.advance(S_)) {
          const int s = sp.slot;
          if (!bounded_wait(&bars->full[s], sp.phase, abort, args.err)) { ok = false; break; }
          const uint32_t st = smem_u32(smem + s * args.stage_bytes);
          if (T::kTs) {
            for (int sc = 0; sc < T::kSub; ++sc, ap.advance(na)) {
              if (kBconv) {
                // this sub-chunk's token codes -> FP16 operand tile in the next token slot
                // (128-byte swizzle, BN rows of 64 K)
                const uint32_t bslot = bp.slot;
                if (!bounded_wait(&bars->bempty[bslot], bp.phase ^ 1, abort, args.err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tile = smem_u32(smem + args.off_bring) + bslot * BN * 128;
                const uint32_t braw = st + args.off_braw;
                // 64 K = four 16-code chunks of raw box sc / 2 (128 codes per row)
                for (int i = ctid; i < BN * 4; i += kConvWarps * 32) {
                  const int row = i >> 2, c = 4 * (sc & 1) + (i & 3);
                  const uint4 v = lds128(sw128(braw + (sc >> 1) * BN * 128, row, c));
                  uint32_t o[16];
                  const uint4 zero = make_uint4(0, 0, 0, 0);
                  cvt_int8x32<false>(v, zero, o);  // first 8 words hold the 16 converted values
                  const int cc = (c & 3) * 2;
                  sts128(sw128(tile, row, cc), o[0], o[1], o[2], o[3]);
                  sts128(sw128(tile, row, cc + 1), o[4], o[5], o[6], o[7]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->bfull[bslot]);
                bp.advance(kBSlots);
              }
              const uint32_t aslot = ap.slot;
              if (!bounded_wait(&bars->aempty[aslot], ap.phase ^ 1, abort, args.err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const int kin = sc * 64 + h * 32;            // K offset inside the stage
#pragma unroll
              for (int m = 0; m < kNmat; ++m) {
                const uint32_t abase = st + args.off_a[m];
                uint32_t o[16];
                if (WF == WF_INT4) {
                  const uint4 v = lds128(sw128(abase, r, kin >> 5));  // 32 codes = one 16-byte chunk
                  cvt_int4x32<AM == AM_BF16>(v, o);
                } else if (WF == WF_INT8) {
                  const uint4 v0 = lds128(sw128(abase, r, kin >> 4));  // 32 codes = two chunks
                  const uint4 v1 = lds128(sw128(abase, r, (kin >> 4) + 1));
                  cvt_int8x32<AM == AM_BF16>(v0, v1, o);
                }
                if (kScaleConv && (WF == WF_INT4 || WF == WF_INT8)) {
                  // exact FP16 integers q -> fp16(q * s), s the row's scale of this 128-K group
                  const __half* scl = reinterpret_cast<const __half*>(smem + args.off_scales +
                                                                      (sbuf * kNmat + m) * args.scale_mat_bytes);
                  const uint32_t sh = __half_as_ushort(scl[r * G + ((ks * T::kStage + kin) >> 7)]);
                  const uint32_t s2 = sh | (sh << 16);
#pragma unroll
                  for (int i = 0; i < 16; ++i) o[i] = f16x2_mul(o[i], s2);
                }
                tmem_st16(tmem + (static_cast<uint32_t>(q * 32) << 16) + aslot * (kNmat * 32) + m * 32 + h * 16, o);
              }
              tmem_wait_st();
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars->afull[aslot]);
            }
            if (!ok) break;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->empty[s]);
        }
        if (kScaleConv && ok) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->sempty[sbuf]);
        }
      }
    }
  } else {
    // ======================= epilogue =======================
    // Warp e (0..7) reads TMEM lane quarter warp % 4 (row r of the tile) and
    // the token columns [c0, c1): the first or second half of the tile, or,
    // for tiles narrower than 32 columns, all of them (the second warp of the
    // pair then only keeps the barrier phases in step).
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int ew = warp - kWarpEpi0;
    const int half = ew >> 2;
    const int cpw = BN >= 32 ? BN / 2 : BN;
    const int c0 = BN >= 32 ? half * cpw : (half ? BN : 0);
    const int c1 = BN >= 32 ? c0 + cpw : (half ? BN : BN);
    const uint32_t lane_bits = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t nacc = static_cast<uint32_t>(args.acc_slots);
    RingPos cp;  // accumulator slots
    uint32_t uit = 0;
    bool ok = true;
    // each epilogue warp keeps its own copy of its columns' activation scales
    float* sa = reinterpret_cast<float*>(smem + args.off_sa) + ew * cpw * G;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++uit) {
      const Unit x = decode_unit(tab_prefix, tab_off, E, args.n_tiles, BN, u);
      const int n0 = x.nt * kBM;
      const int col = n0 + r;
      const int jend = min(c1, x.nrows);  // live columns of this warp: [c0, jend)
      if (!kGrouped) {
        const uint32_t slot = cp.slot;
        // The unit's scale factors, loaded before the wait so their latency overlaps it:
        // the expert matrices' outer scales, and the row factors of this warp's tokens
        // c0 + lane and c0 + 32 + lane (up to 64 columns per warp).
        float ow[2] = {1.f, 1.f};
        if (AM == AM_FP4) {
          for (int m = 0; m < kNmat; ++m)
            ow[m] = __ldg(reinterpret_cast<const float*>(args.experts + static_cast<uint64_t>(x.e) * args.expert_stride +
                                                         args.outer_off[m]));
        }
        float oa_r[4] = {1.f, 1.f, 1.f, 1.f};  // row factors of tokens c0 + 32 i + lane (up to 128 columns)
        if (AM == AM_FP4 || AM == AM_F16S) {
#pragma unroll
          for (int h2 = 0; h2 < 4; ++h2)
            if (32 * h2 < c1 - c0) oa_r[h2] = __ldg(args.a_outer + min(x.row0 + c0 + 32 * h2 + lane, args.P - 1));
        }
        if (!bounded_wait(&bars->accfull[slot], cp.phase, abort, args.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + lane_bits + args.acc_base + slot * kNmat * BN;
        // Each 16-token chunk goes through this warp's staging tile [16 tokens][32 features]
        // (BF16), then out as 16-byte row pieces: 64 bytes of a token's row per 4 lanes.
        uint16_t* stage = reinterpret_cast<uint16_t*>(smem + args.off_sa) + ew * (16 * 32);
        const uint32_t stage_s = smem_u32(stage);
        for (int j0 = c0; j0 < jend; j0 += 16) {
          uint32_t g[16], up[16];
          tmem_ld16(d + j0, g);
          if (kGateUp) tmem_ld16(d + BN + j0, up);
          tmem_wait_ld();
          // the chunk's tokens j0 .. j0+15 are this warp's columns (j0 - c0) .. +15: held by lanes (j0 - c0 + i) % 32
          const int oc = (j0 - c0) >> 5;
          const float oa_c = oc == 0 ? oa_r[0] : (oc == 1 ? oa_r[1] : (oc == 2 ? oa_r[2] : oa_r[3]));
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float oa = __shfl_sync(0xffffffffu, oa_c, ((j0 - c0) & 31) + i);
            float gv = __uint_as_float(g[i]);
            if (AM == AM_FP4) gv = gv * (ow[0] * oa);
            else if (AM == AM_F16S) gv = gv * oa;
            float val = gv;
            if (kGateUp) {
              float uv = __uint_as_float(up[i]);
              if (AM == AM_FP4) uv = uv * (ow[1] * oa);
              else if (AM == AM_F16S) uv = uv * oa;
              val = __fdividef(gv, 1.f + __expf(-gv)) * uv;
            }
            stage[i * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
          }
          __syncwarp();
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int c = lane + 32 * h2;  // 16-byte piece: token c / 4, features 8 (c % 4) ..
            const int j = j0 + (c >> 2);
            if (j < jend && x.row0 + j < args.P) {
              const uint4 v = lds128(stage_s + c * 16);
              stg128(args.out + static_cast<size_t>(x.row0 + j) * args.N + n0 + q * 32 + (c & 3) * 8, v.x, v.y,
                     v.z, v.w);
            }
          }
          __syncwarp();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->accempty[slot]);
        cp.advance(nacc);
      } else {
        // Grouped: one accumulator per 128-wide K group.  Each group's exact
        // dot products D_g are scaled in FP32 (by s_w, times s_a in the A8
        // mode) and added to a running sum held in TMEM.
        const uint32_t sb = uit & 1;
        if (!bounded_wait(&bars->sfull[sb], (uit >> 1) & 1, abort, args.err)) { ok = false; break; }
        if (AM == AM_INT8) {
          for (int i = lane; i < cpw * G; i += 32) {
            const int j = c0 + i / G, gg = i - (i / G) * G;
            sa[i] = (j < x.nrows && x.row0 + j < args.P)
                        ? __ldg(args.a_scales + static_cast<size_t>(x.row0 + j) * G + gg)
                        : 0.f;
          }
          __syncwarp();
        }
        const __half* sw0 =
            reinterpret_cast<const __half*>(smem + args.off_scales + (sb * kNmat + 0) * args.scale_mat_bytes) + r * G;
        const __half* sw1 =
            reinterpret_cast<const __half*>(smem + args.off_scales + (sb * kNmat + (kNmat - 1)) * args.scale_mat_bytes) +
            r * G;
        const uint32_t dsum = tmem + lane_bits + args.sum_base;
        const bool want_dots = AM == AM_INT8 && args.dots != nullptr;
        for (int g = 0; g < G; ++g) {
          const uint32_t slot = cp.slot;
          if (!bounded_wait(&bars->accfull[slot], cp.phase, abort, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + lane_bits + args.acc_base + slot * kNmat * BN;
          const float w0 = __half2float(sw0[g]), w1 = __half2float(sw1[g]);
          const bool last = g == G - 1;
          for (int j0 = c0; j0 < jend; j0 += 16) {
            uint32_t d0[16], d1[16], s0[16], s1[16];
            tmem_ld16(d + j0, d0);
            if (kGateUp) tmem_ld16(d + BN + j0, d1);
            if (g > 0) {
              tmem_ld16(dsum + j0, s0);
              if (kGateUp) tmem_ld16(dsum + BN + j0, s1);
            }
            tmem_wait_ld();
            if (want_dots) {
              const size_t C = static_cast<size_t>(kNmat) * args.N;
              for (int i = 0; i < 16; ++i) {
                const int j = j0 + i;
                if (j >= jend) break;
                const size_t base = (static_cast<size_t>(x.row0 + j) * C) * G;
                args.dots[base + static_cast<size_t>(col) * G + g] = __float2int_rn(__uint_as_float(d0[i]));
                if (kGateUp)
                  args.dots[base + static_cast<size_t>(args.N + col) * G + g] = __float2int_rn(__uint_as_float(d1[i]));
              }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float f0 = w0, f1 = w1;
              if (AM == AM_INT8) {
                const float s_a = sa[(j0 - c0 + i) * G + g];
                f0 = __fmul_rn(w0, s_a);
                f1 = __fmul_rn(w1, s_a);
              }
              const float a0 = __fmaf_rn(f0, __uint_as_float(d0[i]), g > 0 ? __uint_as_float(s0[i]) : 0.f);
              float a1 = 0.f;
              if (kGateUp) a1 = __fmaf_rn(f1, __uint_as_float(d1[i]), g > 0 ? __uint_as_float(s1[i]) : 0.f);
              s0[i] = __float_as_uint(a0);
              s1[i] = __float_as_uint(a1);
            }
            if (!last) {
              tmem_st16(dsum + j0, s0);
              if (kGateUp) tmem_st16(dsum + BN + j0, s1);
            } else {
              for (int i = 0; i < 16; ++i) {
                const int j = j0 + i;
                if (j >= jend || x.row0 + j >= args.P) break;
                const float a0 = __uint_as_float(s0[i]), a1 = __uint_as_float(s1[i]);
                const float val = kGateUp ? __fdividef(a0, 1.f + __expf(-a0)) * a1 : a0;
                args.out[static_cast<size_t>(x.row0 + j) * args.N + col] = __float2bfloat16_rn(val);
              }
            }
          }
          if (!last) tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->accempty[slot]);
          cp.advance(nacc);
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->sempty[sb]);
      }
    }
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

constexpr size_t kSmemLimit = 232448;  // max dynamic shared memory per block on sm_103

inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

struct Plan {
  GemmArgs args;
  size_t smem;
};

// Lay out one stage and the fixed areas for a given BN; returns false if
// fewer than two stages fit.
bool plan_smem(int wf, int am, bool gate_up, int K, int E, int BN, Plan* p) {
  const int nmat = gate_up ? 2 : 1;
  const int kstage = wf == WF_BF16 ? 64 : (wf == WF_INT8 ? 128 : 256);
  GemmArgs& a = p->args;
  uint32_t off = 0;
  for (int m = 0; m < 2; ++m) {
    a.off_a[m] = off;
    if (m < nmat) off += 16384;
  }
  for (int m = 0; m < 2; ++m) {
    a.off_asf[m] = off;
    if (wf == WF_NVFP4 && m < nmat) off += 2048;
  }
  off = align_up(off, 1024);
  a.off_b = off;
  if (am == AM_BF16 || am == AM_F16S) off += (kstage / 64) * BN * 128;  // 16-bit tokens copied in operand layout
  off = align_up(off, 1024);
  a.off_braw = off;
  if (am == AM_INT8) off += (kstage / 128) * BN * 128;
  if (am == AM_FP4) off += BN * 128;
  off = align_up(off, 1024);
  a.off_bsf = off;
  if (am == AM_FP4) off += BN * 16;
  off = align_up(off, 1024);
  a.stage_bytes = off;

  const int G = K / 128;
  uint32_t fixed = 0;
  a.scale_mat_bytes = (wf == WF_INT8 || wf == WF_INT4) ? 128u * G * 2u : 0u;
  const uint32_t scales = 2 * nmat * a.scale_mat_bytes;
  const uint32_t tab = align_up(2u * (E + 1) * 4u, 16);
  const uint32_t cpw = BN >= 32 ? BN / 2 : BN;  // token columns per epilogue warp
  // A8: the epilogue warps' activation scales; non-grouped modes: their BF16 staging tiles [16][32]
  const bool grouped = am == AM_INT8 || (am == AM_BF16 && (wf == WF_INT8 || wf == WF_INT4));
  const uint32_t sa = am == AM_INT8 ? align_up(kEpiWarps * cpw * G * 4u, 16) : (grouped ? 0u : kEpiWarps * 16u * 32u * 2u);
  const uint32_t bars = align_up(sizeof(Bars), 16);
  const uint32_t bring = am == AM_INT8 ? kBSlots * BN * 128u : 0u;  // converted-token ring
  fixed = bring + scales + tab + sa + bars;
  const size_t budget = kSmemLimit - 1024;  // alignment slack
  if (fixed + 2 * a.stage_bytes > budget) return false;
  int stages = static_cast<int>((budget - fixed) / a.stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  a.stages = stages;
  uint32_t o = stages * a.stage_bytes;
  a.off_bring = o;  // a multiple of 1024: stage_bytes is
  o += bring;
  a.off_scales = o;
  o += scales;
  a.off_tab = o;
  o += tab;
  a.off_sa = o;
  o += sa;
  a.off_bars = align_up(o, 16);
  o = a.off_bars + bars;
  p->smem = o + 1024;
  return true;
}

template <int WF, int AM, bool GU>
cudaError_t launch_one(const CUtensorMap* maps, const GemmArgs& a, size_t smem, int grid, cudaStream_t st) {
  auto kern = moe_gemm_kernel<WF, AM, GU>;
  static std::atomic<uint64_t> attr{0};
  uint64_t bit;
  if (attrs_needed(attr, &bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemLimit));
    if (e != cudaSuccess) return e;
    attrs_done(attr, bit);
  }
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                    a);
}

template <int WF, int AM>
cudaError_t launch_kind(bool gate_up, const CUtensorMap* maps, const GemmArgs& a, size_t smem, int grid,
                        cudaStream_t st) {
  return gate_up ? launch_one<WF, AM, true>(maps, a, smem, grid, st) : launch_one<WF, AM, false>(maps, a, smem, grid, st);
}

}  // namespace

int warp_gemm_nt(int P, int E) {
  const int mean_rows = (P + E - 1) / E;
  return mean_rows <= 4 ? 1 : (mean_rows <= 16 ? 2 : 4);
}

int run_gemm(const mnw_moe_layer* L, int wfmt, int act, int kind, const void* a0, const void* a1, const void* a2,
             const int32_t* offsets, int P, void* out, int32_t* dots, uint32_t* err, cudaStream_t st,
             uint32_t* sched, const WarpDep* dep) {
  if (!L || kind < MNW_KIND_GATE_UP || kind > MNW_KIND_UP || P < 0) return MNW_E_INVALID_ARG;
  if (L->wfmt != wfmt) return MNW_E_MODE;
  if (P == 0) return MNW_OK;
  if (!a0 || !offsets || !out || !aligned(a0, 16) || !aligned(out, 16)) return MNW_E_INVALID_ARG;
  if (act == MNW_ACT_INT8_G128 && (!a1 || !aligned(a1, 16))) return MNW_E_INVALID_ARG;
  if (act == MNW_ACT_NVFP4_G16 && (!a1 || !a2 || !aligned(a1, 16) || !aligned(a2, 16))) return MNW_E_INVALID_ARG;
  // the FP16 operand mode: INT weights, row factors in a1
  if (act == kActF16Rows && ((wfmt != MNW_FMT_INT8_G128 && wfmt != MNW_FMT_INT4_G128) || !a1 || !aligned(a1, 4)))
    return MNW_E_INVALID_ARG;
  // INT8/INT4 weights with few tokens per expert: the warp-MMA kernel (see
  // mnw_gemm_warp.cu for why).  From 32 tokens per expert on average the
  // tcgen05 kernel below is as fast or faster (measured on GB300: 64 tokens
  // per expert W8A8 369 vs 486 us for gate/up; 128 per expert W4A16 down
  // 1036 vs 1463 us), and BF16/NVFP4 weights always use it.
  const int mean_rows = (P + L->E - 1) / L->E;
  const int path = gemm_path();
  const bool warp_ok = warp_gemm_applicable(L, wfmt, act, kind);
  if (warp_ok && (path == MNW_PATH_WARP_MMA || (path != MNW_PATH_TCGEN05 && path != MNW_PATH_ROWS && mean_rows < 32))) {
    return run_gemm_warp(L, wfmt, act, kind, a0, a1, offsets, P, warp_gemm_nt(P, L->E), out, dots, err, sched, st,
                         dep);
  }
  if (dep && dep->role != kDepNone) return MNW_E_INVALID_ARG;  // only the warp-MMA kernel takes a dependency
  // FP16 rows on INT weights, and BF16 on BF16: the row-tile kernel (tokens as
  // M, 256 weight rows as N; mnw_gemm_rows.cu) unless the swap-AB kernel below
  // is forced.
  if (path != MNW_PATH_TCGEN05 && rows_gemm_applicable(L, wfmt, act, kind))
    return run_gemm_rows(L, wfmt, act, kind, a0, a1, offsets, P, out, err, st);
  // W8A8: the row-tile kernel with per-group accumulators (mnw_gemm_rows_a8.cu)
  if (path != MNW_PATH_TCGEN05 && rows_a8_applicable(L, wfmt, act, kind))
    return run_gemm_rows_a8(L, kind, a0, static_cast<const float*>(a1), offsets, P, out, dots, err, st);
  const bool gate_up = kind == MNW_KIND_GATE_UP;
  const int K = kind == MNW_KIND_DOWN ? L->I : L->H;
  const int N = kind == MNW_KIND_DOWN ? L->H : L->I;
  const int nmat = gate_up ? 2 : 1;
  const int am = act;  // MNW_ACT_* match AM_*; kActF16Rows is AM_F16S
  const int wf = wfmt;

  // Token tile: the power of two (16..max) nearest above the mean rows per expert.
  const bool grouped = am == AM_INT8 || (am == AM_BF16 && (wf == WF_INT8 || wf == WF_INT4));
  // TMEM budget (512 columns): operand-A ring + accumulators (+ running sums when grouped).
  const int max_bn = grouped ? (gate_up ? 64 : 128) : 128;
  const int mean = (P + L->E - 1) / L->E;
  int BN = 16;
  while (BN < mean && BN < max_bn) BN *= 2;
  // A non-grouped gate/up tile of 128 tokens leaves TMEM room for one
  // accumulator slot only (the MMA then stalls while the epilogue drains);
  // 96 tokens fit two slots beside a two-slot operand-A ring.
  if (!grouped && gate_up && BN == 128 && wf != WF_BF16) BN = 96;
  // NVFP4 down: the block-scaled MMA costs about the same for any N up to 256,
  // so wider token tiles pay; 192 leaves room for two accumulators and two
  // scale-factor slots (gate/up keeps 96: two matrices per tile).
  if (wf == WF_NVFP4 && !gate_up && mean > 128) BN = 192;
  Plan plan{};
  while (!plan_smem(wf, am, gate_up, K, L->E, BN, &plan)) {
    if (BN == 16) return MNW_E_UNSUPPORTED;
    BN /= 2;
  }
  GemmArgs& a = plan.args;
  const bool ts = wf == WF_INT8 || wf == WF_INT4;  // A through TMEM (converted codes)
  a.offsets = offsets;
  a.E = L->E;
  a.P = P;
  a.K = K;
  a.N = N;
  a.BN = BN;
  a.n_tiles = N / kBM;
  a.nmat = nmat;
  if (wf == WF_NVFP4) {
    // TMEM columns: [accumulator slots | scale-factor slots].  A scale-factor
    // slot holds one stage's block scales: 16 columns per weight matrix and 16
    // for the tokens.  At least two of each, so the epilogue drains one
    // accumulator while the MMAs fill the other and the scale-factor warps
    // fill one slot while the MMAs read the other.
    const int d_cols = nmat * BN, sf_cols = 16 * nmat + 32;
    int nacc = 2, nsf = 2;
    if (2 * d_cols + 2 * sf_cols > kTmemCols) return MNW_E_UNSUPPORTED;
    while (nacc < 4 && (nacc + 1) * d_cols + 2 * sf_cols <= kTmemCols) ++nacc;
    while (nsf < kMaxSf && nsf < a.stages && nacc * d_cols + (nsf + 1) * sf_cols <= kTmemCols) ++nsf;
    a.aslots = 1;
    a.acc_slots = nacc;
    a.acc_base = 0;
    a.sum_base = 0;
    a.sf_base = nacc * d_cols;
    a.sf_slots = nsf;
    a.sf_cols = sf_cols;
  } else {
    // TMEM columns: [A ring | accumulator slots | running sum (grouped)].
    // Deep rings hide the converter -> MMA -> epilogue hand-off latency; small
    // token tiles leave room for more slots.
    const int a_cols = ts ? nmat * 32 : 0;
    const int d_cols = nmat * BN;
    const int sum_cols = grouped ? nmat * BN : 0;
    int na = ts ? 2 : 0, nacc = grouped ? 2 : 1;
    auto fits = [&](int x, int y) { return x * a_cols + y * d_cols + sum_cols <= kTmemCols; };
    if (!fits(na, nacc)) return MNW_E_UNSUPPORTED;
    // grow in turn: accumulators to 2, A ring to 4, accumulators to 4, A ring to 8, accumulators to 8
    const int steps[5][2] = {{0, 2}, {4, 0}, {0, 4}, {8, 0}, {0, 8}};
    for (const auto& st : steps) {
      if (st[0]) while (ts && na < st[0] && fits(na + 1, nacc)) ++na;
      if (st[1]) while (nacc < st[1] && fits(na, nacc + 1)) ++nacc;
    }
    a.aslots = ts ? na : 1;
    a.acc_slots = nacc;
    a.acc_base = na * a_cols;
    a.sum_base = a.acc_base + nacc * d_cols;
  }
  a.experts = L->blob + L->data_offset;
  a.expert_stride = L->expert_stride;
  const int m0 = kind_matrix(kind);  // first (or only) matrix of the launch
  for (int m = 0; m < nmat; ++m) {
    a.scales_off[m] = L->scales_off[m0 + m];
    a.outer_off[m] = L->outer_off[m0 + m];
  }
  a.a_scales = am == AM_INT8 ? static_cast<const float*>(a1) : nullptr;
  a.a_outer = am == AM_FP4 ? static_cast<const float*>(a2) : (am == AM_F16S ? static_cast<const float*>(a1) : nullptr);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.dots = am == AM_INT8 ? dots : nullptr;
  a.err = err;

  // Tensor maps: 0/1 weight codes, 2/3 NVFP4 weight scales, 4 tokens, 5 token scales.
  CUtensorMap maps[6];
  memset(maps, 0, sizeof(maps));
  maps[0] = L->tm_codes[m0];
  if (gate_up) maps[1] = L->tm_codes[1];
  if (wf == WF_NVFP4) {
    maps[2] = L->tm_sf[m0];
    if (gate_up) maps[3] = L->tm_sf[1];
  }
  const uint64_t Pu = static_cast<uint64_t>(P);
  bool ok;
  if (am == AM_BF16 || am == AM_F16S) {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), Pu};
    const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(BN)};
    ok = encode_map(&maps[4], am == AM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a0,
                    dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else if (am == AM_INT8) {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), Pu};
    const uint64_t strides[1] = {static_cast<uint64_t>(K)};
    const uint32_t box[2] = {128, static_cast<uint32_t>(BN)};
    ok = encode_map(&maps[4], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a0, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const uint64_t dims[2] = {static_cast<uint64_t>(K / 2), Pu};
    const uint64_t strides[1] = {static_cast<uint64_t>(K / 2)};
    const uint32_t box[2] = {128, static_cast<uint32_t>(BN)};
    ok = encode_map(&maps[4], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a0, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    const uint64_t dims2[2] = {static_cast<uint64_t>(K / 16), Pu};
    const uint64_t strides2[1] = {static_cast<uint64_t>(K / 16)};
    const uint32_t box2[2] = {16, static_cast<uint32_t>(BN)};
    ok = ok && encode_map(&maps[5], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a1, dims2, strides2, box2,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!ok) return MNW_E_INVALID_ARG;

  const int grid = L->num_sms;
  cudaError_t e = cudaErrorInvalidValue;
  switch (wf * 4 + am) {
    case WF_BF16 * 4 + AM_BF16: e = launch_kind<WF_BF16, AM_BF16>(gate_up, maps, a, plan.smem, grid, st); break;
    case WF_INT8 * 4 + AM_BF16: e = launch_kind<WF_INT8, AM_BF16>(gate_up, maps, a, plan.smem, grid, st); break;
    case WF_INT4 * 4 + AM_BF16: e = launch_kind<WF_INT4, AM_BF16>(gate_up, maps, a, plan.smem, grid, st); break;
    case WF_INT8 * 4 + AM_INT8: e = launch_kind<WF_INT8, AM_INT8>(gate_up, maps, a, plan.smem, grid, st); break;
    case WF_INT4 * 4 + AM_INT8: e = launch_kind<WF_INT4, AM_INT8>(gate_up, maps, a, plan.smem, grid, st); break;
    case WF_NVFP4 * 4 + AM_FP4: e = launch_kind<WF_NVFP4, AM_FP4>(gate_up, maps, a, plan.smem, grid, st); break;
    case WF_INT8 * 4 + AM_F16S: e = launch_kind<WF_INT8, AM_F16S>(gate_up, maps, a, plan.smem, grid, st); break;
    case WF_INT4 * 4 + AM_F16S: e = launch_kind<WF_INT4, AM_F16S>(gate_up, maps, a, plan.smem, grid, st); break;
    default: return MNW_E_MODE;
  }
  return e == cudaSuccess ? MNW_OK : MNW_E_CUDA;
}

}  // namespace mnw
