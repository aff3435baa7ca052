// mnw_gemm_warp.cuh -- the warp-MMA grouped GEMM kernel (device code and the
// launch template), shared by mnw_gemm_warp.cu and mnw_gemm_warp_dep.cu.
//
// Grouped expert GEMMs for INT8/INT4 weights when few
// tokens are routed to each expert (decode batches, the INT8-activation mode
// at moderate batch).
//
// Measured on GB300 (sm_103a): a tcgen05.mma of kind::f16 with M = 128 costs
// ~96 SM cycles whatever N <= 64 is, so with 8-16 tokens per expert one MMA
// moves only 2048 weights per ~96 cycles -- under half of what streaming INT4
// weights at HBM rate requires.  The warp-level m16n8k16 MMA moves 256
// weights per cycle per SM at N = 8 (16 warps), so for this regime the
// weights are dequantised straight into MMA operand registers:
//
//   TMA (one producer warp)  raw weight codes of a 128-K group for 256 weight
//                            rows, and the group's slice of the expert's
//                            token tile, into a shared-memory ring
//   8 MMA warps (x2 CTAs/SM) codes -> exact BF16/FP16 integers in registers,
//                            m16n8k16 MMAs into a per-group accumulator, then
//                            acc += s_w (* s_a) * group_dot in FP32; SiLU(g)*u
//                            or y written as BF16 straight from registers
//
// Weight format and numerics follow the "LLaDA2.2-flash-minnow" model card,
// "Checkpoints and precision" (signed INT8/INT4, one FP16 scale per 128
// weights; the W8A8/W4A8 mode's INT32 group dot products combined in FP32).
// The weights are never rounded (integer codes are exact in BF16/FP16); each
// 128-wide group's dot product is accumulated in FP32 (exact for INT8
// activations) and combined exactly as in the tcgen05 path (mnw_gemm.cu), so
// the two kernels give identical bits in the INT8-activation mode.
//
// Operand mapping.  Within one 128-K group, lane (g = lane/4, t = lane%4)
// owns K = 32t .. 32t+31 of its rows (16 contiguous code bytes for INT4, 32
// for INT8, 64 bytes of 16-bit activations).  For k-step s (0..7) its A/B
// fragment slots {2t, 2t+1} hold K = 32t+4s+{0,1} and slots {2t+8, 2t+9}
// hold K = 32t+4s+{2,3}.  A and B use the same assignment, so the dot
// product is unchanged and no shuffle is needed.
//
// FP16 rows (activations fp16 with a power-of-two factor per row) with INT4
// weights pair K differently: k-steps 2c and 2c+1 cover the 8 K of code word
// c (K = 32t+8c .. +7, nibble i = K 8c+i), slots {2t, 2t+1} holding K
// {0,4} / {2,6} and slots {2t+8, 2t+9} K {1,5} / {3,7} of the word.  With
// FP16's 10-bit mantissa, one AND-XOR places nibbles 0 and 4 (or 1 and 5,
// 16 times larger) of a word under the exponent of 1024, so a word becomes
// four operand registers in 1 shift + 4 AND-XOR + 2 subtractions + 2 FMAs,
// against 9 integer instructions + 4 subtractions for the BF16 operands.
// The token fragment then takes its pairs {x_j, x_j+4} from one 16-byte load
// by two byte permutes per register pair.
//
// Work unit: (expert, token tile of 8*NT rows, block of 256 weight rows).
// gate/up: rows are 128 gate features + the same 128 up features, so each
// thread ends with gate and up of the same (token, feature) and applies
// SiLU(g)*u in registers.  down: 256 consecutive rows of Wd.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "mnw_convert.cuh"
#include "mnw_internal.h"
#include "mnw_ptx.cuh"

namespace mnw {
namespace warpmma {

enum { WF_INT8 = 1, WF_INT4 = 2 };
// AM_F16R: FP16 activation rows with a float factor per row (kActF16Rows)
enum { AM_BF16 = 0, AM_INT8 = 1, AM_F16R = 3 };

constexpr int kMmaWarps = 8;
constexpr int kThreads = (1 + kMmaWarps) * 32;  // warp 0 = producer
// A launch that releases token tiles to a dependent launch has one more warp
// (the releaser, after the MMA warps).
constexpr int threads_for(int dep) { return kThreads + (dep == 1 ? 32 : 0); }
constexpr int kMaxStages = 12;
constexpr int kRowsPerBox = 128;
// 128-K groups per pipeline stage: one for INT4 (a 64-byte code box per
// 128-row block, 64-byte swizzle: small stages, so a deeper ring fits), two
// for INT8 (one 128-byte box per group).
__host__ __device__ constexpr int groups_per_stage(int wf) { return wf == 2 ? 1 : 2; }
constexpr int kBoxBytes = 128 * 128;    // INT8: one TMA box, 128 rows x 128 bytes
constexpr int kBox64Bytes = 128 * 64;   // INT4: one TMA box, 128 rows x 64 bytes
// CTAs per SM: two (16 MMA warps) for INT4 with 8- and 16-token tiles, whose
// registers fit in 96 and whose stages fit in half the shared memory; one
// otherwise (INT8 stages are twice as large, 32-token accumulators need more).
constexpr int ctas_per_sm(int wf, int nt) { return (nt <= 2 && wf == 2) ? 2 : 1; }

struct Args {
  const int32_t* offsets;
  int E, P, K, N, BN, n_blocks, stages;
  uint32_t stage_bytes, off_b, box_bytes, off_scales, scale_box_bytes, off_tab, off_bars;
  const uint8_t* experts;
  uint64_t expert_stride;
  uint64_t scales_off[2];  // box 0 / box 1 matrices (gate, up) or (down, down)
  int box_row_off[2];      // row offset of box 1 within its matrix (0 for gate/up, 128 for down)
  const float* a_scales;   // INT8 activations: [P][K/128]
  const float* a_outer;    // FP16 rows: the row factors [P]
  __nv_bfloat16* out;
  int32_t* dots;
  uint32_t* err;
  // [claim, done]: zero at launch; the last CTA to finish zeroes it again.
  // NULL: units are handed out statically (CTA c takes c, c + grid, ...).
  uint32_t* sched;
  uint32_t* dep;    // tile dependency counters (WarpDep), or null
  int dep_role;     // kDepNone / kDepProduce / kDepConsume
  uint32_t dep_need;
};

struct Bars {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t sfull[2], sempty[2];
  uint64_t udone[2];  // per unit slot: the MMA warps have written the unit's output rows
  int unit[2];  // unit handed from the producer to the MMA warps, per scale buffer
  int abort;
};

__device__ __forceinline__ void hmma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void hmma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Work unit -> (expert, token tile, row block).
struct Unit {
  int e, rb, row0, nrows;
};
__device__ __forceinline__ Unit decode(const int* tab_prefix, const int* tab_off, int E, int n_blocks, int BN,
                                       int u) {
  Unit x;
  const int t = u / n_blocks;
  x.rb = u - t * n_blocks;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tab_prefix[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  x.e = lo;
  x.row0 = tab_off[lo] + (t - tab_prefix[lo]) * BN;
  x.nrows = min(BN, tab_off[lo + 1] - x.row0);
  return x;
}

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

// Two (even, odd) operand words from byte pair (2p, 2p+1) of 8 INT4 codes.
template <bool kBf16>
__device__ __forceinline__ void int4_pair(uint32_t w, int p, uint32_t& lo, uint32_t& hi) {
  const uint32_t sh = w >> 4;
  const int b0 = 2 * p, b1 = 2 * p + 1;
  const uint32_t x0 = prmt(w, sh, 0x0400u + 0x0101u * b0), x1 = prmt(w, sh, 0x0400u + 0x0101u * b1);
  if (kBf16) {
    lo = bf16x2_sub(and_xor(x0, 0x000F000Fu, 0x43084308u), 0x43084308u);
    hi = bf16x2_sub(and_xor(x1, 0x000F000Fu, 0x43084308u), 0x43084308u);
  } else {
    lo = f16x2_sub(and_xor(x0, 0x000F000Fu, 0x64086408u), 0x64086408u);
    hi = f16x2_sub(and_xor(x1, 0x000F000Fu, 0x64086408u), 0x64086408u);
  }
}
// Two FP16 operand words from INT4 code word w (nibble i = K i): K {0,4} and
// {1,5} (odd = false) or K {2,6} and {3,7} (odd = true), exact integers.
template <bool kOdd>
__device__ __forceinline__ void int4_j4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t v = kOdd ? w >> 8 : w;
  // 0x6400 | (n ^ 8) = 1024 + (n ^ 8); minus 1032 gives the signed code
  lo = f16x2_sub(and_xor(v, 0x000F000Fu, 0x64086408u), 0x64086408u);
  // 0x6400 | (n ^ 8) << 4 = 1024 + 16 (n ^ 8); times 1/16 (0x2C00) minus 72 (0xD480)
  hi = f16x2_fma(and_xor(v, 0x00F000F0u, 0x64806480u), 0x2C002C00u, 0xD480D480u);
}
// Two operand words from the 4 INT8 codes of one 32-bit word.
template <bool kBf16>
__device__ __forceinline__ void int8_pair(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  if (kBf16) {
    float f[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) f[b] = __fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7540u + b)), 8388736.0f);
    lo = pack_bf16x2(f[0], f[1]);
    hi = pack_bf16x2(f[2], f[3]);
  } else {
    lo = f16x2_sub(prmt(u, 0x64646464u, 0x4140u), 0x64806480u);
    hi = f16x2_sub(prmt(u, 0x64646464u, 0x4342u), 0x64806480u);
  }
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One 128-K group of a stage for one warp: its 16 rows of both row blocks
// against the first NTA token tiles (NTA is fixed per unit, so the body has
// no branches and the compiler can interleave all of it), then the FP32
// group combine tot += (s_w [* s_a]) * exact group dot.
template <int WF, int AM, bool kGateUp, int NT, int NTA>
__device__ __forceinline__ void group_step(const Args& args, uint32_t st, uint32_t stb,
                                           const uint32_t (&a_off)[2][2][2], const uint32_t (&b_off)[NT][4],
                                           const __half* scl0, const __half* scl1, int w, int g, int t, int grp,
                                           int G, const Unit& x, int nb, float (&tot)[2][NT][4]) {
  constexpr bool kBf16 = AM == AM_BF16;
  constexpr bool kJ4 = AM == AM_F16R && WF == WF_INT4;  // (j, j+4) K pairing
  // raw codes: [box i][row g / g+8]
  uint4 ar[2][2][WF == WF_INT4 ? 1 : 2];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      ar[i][hh][0] = lds128(st + a_off[i][hh][0]);
      if constexpr (WF != WF_INT4) ar[i][hh][1] = lds128(st + a_off[i][hh][1]);
    }
  float cg[2][NTA][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < NTA; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) cg[i][j][q] = 0.f;
  uint4 bv[NTA];  // kJ4: the 8 activations of the current code word, per n-tile
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    // token operand of this k-step: K = 32t + 4ks .. +3 of each n-tile's row
    // (kJ4: K {0,4},{1,5} or {2,6},{3,7} of K = 32t + 8(ks/2) .. +7)
    uint32_t b0[NTA], b1[NTA];
#pragma unroll
    for (int j = 0; j < NTA; ++j) {
      if constexpr (kJ4) {
        if ((ks & 1) == 0) bv[j] = lds128(stb + b_off[j][ks >> 1]);
        const uint32_t p = (ks & 1) ? bv[j].y : bv[j].x, q = (ks & 1) ? bv[j].w : bv[j].z;
        b0[j] = prmt(p, q, 0x5410u);
        b1[j] = prmt(p, q, 0x7632u);
      } else if constexpr (AM != AM_INT8) {
        const uint2 v = lds64(stb + b_off[j][ks >> 1] + 8 * (ks & 1));
        b0[j] = v.x;
        b1[j] = v.y;
      } else {
        int8_pair<false>(lds32(stb + b_off[j][ks >> 2] + 4 * (ks & 3)), b0[j], b1[j]);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t a[4];  // {row g, slots 2t..}, {row g+8, 2t..}, {row g, 2t+8..}, {row g+8, 2t+8..}
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t lo, hi;
        if constexpr (kJ4) {
          if (ks & 1) int4_j4<true>(word_of(ar[i][hh][0], ks >> 1), lo, hi);
          else int4_j4<false>(word_of(ar[i][hh][0], ks >> 1), lo, hi);
        } else if constexpr (WF == WF_INT4) {
          int4_pair<kBf16>(word_of(ar[i][hh][0], ks >> 1), ks & 1, lo, hi);
        } else {
          int8_pair<kBf16>(word_of(ar[i][hh][ks >> 2], ks & 3), lo, hi);
        }
        a[hh] = lo;
        a[2 + hh] = hi;
      }
#pragma unroll
      for (int j = 0; j < NTA; ++j) {
        if constexpr (kBf16) hmma_bf16(cg[i][j], a, b0[j], b1[j]);
        else hmma_f16(cg[i][j], a, b0[j], b1[j]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const __half* scl = i == 0 ? scl0 : scl1;
    const float sw0 = __half2float(scl[(16 * w + g) * G + grp]);
    const float sw1 = __half2float(scl[(16 * w + g + 8) * G + grp]);
#pragma unroll
    for (int j = 0; j < NTA; ++j) {
      const int tok0 = j * 8 + 2 * t;
      float f00 = sw0, f01 = sw0, f10 = sw1, f11 = sw1;
      if constexpr (AM == AM_INT8) {
        const float sa0 = tok0 < x.nrows ? __ldg(args.a_scales + static_cast<size_t>(x.row0 + tok0) * G + grp) : 0.f;
        const float sa1 =
            tok0 + 1 < x.nrows ? __ldg(args.a_scales + static_cast<size_t>(x.row0 + tok0 + 1) * G + grp) : 0.f;
        f00 = __fmul_rn(sw0, sa0); f01 = __fmul_rn(sw0, sa1);
        f10 = __fmul_rn(sw1, sa0); f11 = __fmul_rn(sw1, sa1);
      }
      tot[i][j][0] = __fmaf_rn(f00, cg[i][j][0], tot[i][j][0]);
      tot[i][j][1] = __fmaf_rn(f01, cg[i][j][1], tot[i][j][1]);
      tot[i][j][2] = __fmaf_rn(f10, cg[i][j][2], tot[i][j][2]);
      tot[i][j][3] = __fmaf_rn(f11, cg[i][j][3], tot[i][j][3]);
      if (AM == AM_INT8 && args.dots) {
        // exact group dot products, layout [P][C][G]; C = 2N (gate, up) or N
        const size_t C = kGateUp ? 2 * static_cast<size_t>(args.N) : static_cast<size_t>(args.N);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int tok = tok0 + (q & 1);
          const int feat = nb + args.box_row_off[i] + 16 * w + g + 8 * (q >> 1);
          const size_t col = kGateUp ? static_cast<size_t>(i) * args.N + feat : static_cast<size_t>(feat);
          if (tok < x.nrows)
            args.dots[(static_cast<size_t>(x.row0 + tok) * C + col) * G + grp] = __float2int_rn(cg[i][j][q]);
        }
      }
    }
  }
}

// The releaser warp of a launch that releases token tiles (kDepProduce): per
// unit, once all MMA warps have written its output rows, one release add on
// the token tile's counter; CTA 0 first sets the ready flag (every thread has
// passed the wait on the previous kernel before the roles split).  Kept out of
// line so that its code takes no part in the MMA warps' register allocation.
static __device__ __noinline__ void release_loop(Bars* bars, volatile int* abort, uint32_t* err, uint32_t* dep, int n_blocks,
                                          int units) {
  if (blockIdx.x == 0) {
    __threadfence();
    atomicExch(dep, 1u);
  }
  for (uint32_t uit = 0;; ++uit) {
    const uint32_t sb = uit & 1, par = (uit >> 1) & 1;
    if (!bounded_wait(&bars->sfull[sb], par, abort, err)) break;
    const int u = *reinterpret_cast<volatile int*>(&bars->unit[sb]);
    if (u >= units) break;
    if (!bounded_wait(&bars->udone[sb], par, abort, err)) break;
    __threadfence();
    atomicAdd(dep + 1 + u / n_blocks, 1u);
    mbar_arrive(&bars->sempty[sb]);
  }
}

// kDep: kDepNone, or the launch's role in a gate/up -> down tile dependency
// (WarpDep).  A template parameter so that launches without one compile to
// the same code (and registers) as if the feature did not exist.
template <int WF, int AM, bool kGateUp, int NT, int kDep>
__global__ void __launch_bounds__(threads_for(kDep), ctas_per_sm(WF, NT))
    moe_gemm_warp_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                         const __grid_constant__ CUtensorMap tmB, const Args args) {
  constexpr bool k16 = AM != AM_INT8;  // 16-bit activation rows (BF16 or FP16)
  // A stage holds kG 128-K groups: per weight row 64 contiguous code bytes
  // (INT4, one group, 64-byte swizzle) or two 128-byte pieces (INT8, two
  // groups, 128-byte swizzle).
  constexpr int kG = groups_per_stage(WF);
  constexpr int kABoxes = WF == WF_INT4 ? 1 : 2;  // code boxes per 128-row block per stage
  constexpr uint32_t kABox = WF == WF_INT4 ? kBox64Bytes : kBoxBytes;
  constexpr int kABoxX = WF == WF_INT4 ? 64 : 128;  // code bytes per box row
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + args.off_bars);
  int* tab_prefix = reinterpret_cast<int*>(smem + args.off_tab);
  int* tab_off = tab_prefix + (args.E + 1);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E, BN = args.BN, S = args.stages, G = args.K / 128;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], kMmaWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->sfull[i], 1);
      // with a releaser, a unit slot is free again only once its tile is released
      mbar_init(&bars->sempty[i], kMmaWarps + (kDep == kDepProduce ? 1 : 0));
      mbar_init(&bars->udone[i], kMmaWarps);
    }
    bars->abort = 0;
    fence_barrier_init();
  }
  // everything below reads or writes global memory the previous kernel may own
  if constexpr (kDep == kDepConsume) {
    // Started behind the gate/up launch: flags[0] is set only once that launch's
    // own wait has returned, so every kernel before it has completed.
    __syncthreads();  // the barriers and the abort flag are initialised
    if (threadIdx.x == 0 && !bounded_poll_ge(args.dep, 1u, abort, args.err)) bars->abort = 1;
    __syncthreads();
    if (bars->abort) return;  // nothing issued yet: leave without touching memory
  } else {
    pdl_wait();
  }
  if (warp == 1) {  // tile table: first tile of each expert
    const int per = (E + 31) / 32;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        // L2 loads: with a dependency the writer may have run concurrently with this kernel's start
        const int o0 = __ldcg(args.offsets + e), o1 = __ldcg(args.offsets + e + 1);
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
        run += max(0, (__ldcg(args.offsets + e + 1) - tab_off[e] + BN - 1) / BN);
      }
    }
    if (lane == 31) {
      tab_prefix[E] = incl;
      tab_off[E] = __ldcg(args.offsets + E);
    }
  }
  __syncthreads();
  const int units = tab_prefix[E] * args.n_blocks;
  const int rows_per_block = kGateUp ? kRowsPerBox : 2 * kRowsPerBox;

  if (warp == 0) {
    // ======================= producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tmA0);
      tma_prefetch_desc(&tmA1);
      tma_prefetch_desc(&tmB);
      const uint32_t b_bytes = (k16 ? 2u : 1u) * kG * BN * 128u;
      const uint32_t tx = 2u * kABoxes * kABox + b_bytes;
      const int nstages = (G + kG - 1) / kG;
      uint32_t it = 0, uit = 0, sit = 0;
      int s = 0;
      uint32_t ph = 0;  // stage index and phase of `it`, kept without divisions
      bool ok = true;
      // Units are claimed from a counter shared by the CTAs (the last wave
      // stays balanced) and passed to the MMA warps through shared memory
      // under the scale-buffer barrier.  The next unit is claimed while the
      // current unit's last two stages are issued, so the atomic's latency
      // hides behind them and the next unit's loads follow without a gap.
      const int claim_at = nstages >= 2 ? nstages - 2 : 0;
      // Without a counter (a standalone call) the order is static, so launches
      // share no state and may overlap or be replayed on any stream.
      int static_next = static_cast<int>(blockIdx.x);
      auto claim = [&]() -> int {
        if (args.sched) return static_cast<int>(atomicAdd(args.sched, 1u));
        const int u = static_next;
        static_next += static_cast<int>(gridDim.x);
        return u;
      };
      int u_next = claim();
      for (;; ++uit) {
        const int u = u_next;
        const uint32_t sb = uit & 1;
        if (!bounded_wait(&bars->sempty[sb], ((uit >> 1) & 1) ^ 1, abort, args.err)) { ok = false; break; }
        bars->unit[sb] = u;
        if (u >= units) {  // no more work: release the MMA warps
          mbar_arrive(&bars->sfull[sb]);
          break;
        }
        const Unit x = decode(tab_prefix, tab_off, E, args.n_blocks, BN, u);
        const int nb = x.rb * rows_per_block;
        mbar_arrive_expect_tx(&bars->sfull[sb], 2 * args.scale_box_bytes);
        for (int i = 0; i < 2; ++i) {
          const uint8_t* src = args.experts + static_cast<uint64_t>(x.e) * args.expert_stride + args.scales_off[i] +
                               static_cast<uint64_t>(nb + args.box_row_off[i]) * G * 2;
          bulk_load(smem + args.off_scales + (sb * 2 + i) * args.scale_box_bytes, src, args.scale_box_bytes,
                    &bars->sfull[sb]);
        }
        ++sit;
        if constexpr (kDep == kDepConsume) {
          // this unit reads h rows of token tile u / n_blocks: wait until every
          // gate/up MMA warp of every row block has written its part
          if (!bounded_poll_ge(args.dep + 1 + u / args.n_blocks, args.dep_need, abort, args.err)) { ok = false; break; }
          fence_proxy_async();
        }
        for (int ss = 0; ss < nstages; ++ss, ++it) {
          if (ss == claim_at) u_next = claim();
          if (!bounded_wait(&bars->empty[s], ph ^ 1, abort, args.err)) { ok = false; break; }
          uint8_t* st = smem + s * args.stage_bytes;
          mbar_arrive_expect_tx(&bars->full[s], tx);
          // weight codes: box (i, q) holds rows of block i, kABoxX bytes at byte (ss*kABoxes + q)*kABoxX
#pragma unroll
          for (int q = 0; q < kABoxes; ++q) {
            tma_load_3d(st + (0 * kABoxes + q) * kABox, &tmA0, &bars->full[s], (ss * kABoxes + q) * kABoxX,
                        nb + args.box_row_off[0], x.e);
            tma_load_3d(st + (1 * kABoxes + q) * kABox, &tmA1, &bars->full[s], (ss * kABoxes + q) * kABoxX,
                        nb + args.box_row_off[1], x.e);
          }
          // tokens: 64-element 16-bit boxes or 128-element INT8 boxes covering the stage's kG * 128 K
#pragma unroll
          for (int b = 0; b < (k16 ? 2 : 1) * kG; ++b)
            tma_load_2d(st + args.off_b + b * BN * 128, &tmB, &bars->full[s], ss * (kG * 128) + b * (k16 ? 64 : 128),
                        x.row0);
          if (++s == S) { s = 0; ph ^= 1; }
        }
      }
      // The last CTA to stop claiming resets the counter for its next user.
      if (args.sched && atomicAdd(args.sched + 1, 1u) == gridDim.x - 1) {
        atomicExch(args.sched, 0u);
        atomicExch(args.sched + 1, 0u);
      }
      if (!ok || *abort) {
        const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
        for (uint32_t j = first; j < it; ++j) drain(&bars->full[j % S], (j / S) & 1);
        for (uint32_t j = sit > 2 ? sit - 2 : 0; j < sit; ++j) drain(&bars->sfull[j & 1], (j >> 1) & 1);
      }
    }
    return;
  }

  if constexpr (kDep == kDepProduce) {
    if (warp == 1 + kMmaWarps) {
      // ======================= releaser =======================
      if (lane == 0) release_loop(bars, abort, args.err, args.dep, args.n_blocks, units);
      return;
    }
  }

  // ======================= MMA warps =======================
  const int w = warp - 1;            // 0..7: rows 16w .. 16w+15 of both boxes
  const int g = lane >> 2, t = lane & 3;
  uint32_t it = 0, uit = 0;
  int s = 0;
  uint32_t ph = 0;
  // lane-constant shared-memory offsets (swizzled chunk positions)
  uint32_t b_off[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int row = j * 8 + g;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      b_off[j][c] = k16 ? args.off_b + (t >> 1) * BN * 128 + row * 128 + (((4 * (t & 1) + c) ^ (row & 7)) << 4)
                        : args.off_b + row * 128 + (((2 * t + (c & 1)) ^ (row & 7)) << 4);
  }
  // a_off[gi][i][hh][c]: code chunk c of row 16w+g+8hh of block i for group gi of a stage
  // (INT4: 64-byte rows, 16-byte chunk t xor (row / 2) % 4; INT8: 128-byte rows, chunk xor row % 8)
  uint32_t a_off[kG][2][2][2];
#pragma unroll
  for (int gi = 0; gi < kG; ++gi)
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * w + g + 8 * hh;
#pragma unroll
        for (int c = 0; c < 2; ++c)
          a_off[gi][i][hh][c] =
              WF == WF_INT4 ? i * kABox + r * 64 + ((t ^ ((r >> 1) & 3)) << 4)
                            : (2 * i + gi) * kABox + r * 128 + (((2 * t + c) ^ (r & 7)) << 4);
      }
  const uint32_t b_gstep = (k16 ? 2u : 1u) * BN * 128u;  // token boxes per group
  for (;; ++uit) {
    const uint32_t sb = uit & 1;
    if (!bounded_wait(&bars->sfull[sb], (uit >> 1) & 1, abort, args.err)) return;
    const int u = *reinterpret_cast<volatile int*>(&bars->unit[sb]);
    if (u >= units) break;
    const Unit x = decode(tab_prefix, tab_off, E, args.n_blocks, BN, u);
    const int nb = x.rb * rows_per_block;
    const __half* scl[2] = {
        reinterpret_cast<const __half*>(smem + args.off_scales + (sb * 2 + 0) * args.scale_box_bytes),
        reinterpret_cast<const __half*>(smem + args.off_scales + (sb * 2 + 1) * args.scale_box_bytes)};
    float tot[2][NT][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) tot[i][j][q] = 0.f;

    const int nstages = (G + kG - 1) / kG;
    for (int ss = 0; ss < nstages; ++ss, ++it) {
      if (!bounded_wait(&bars->full[s], ph, abort, args.err)) return;
      const uint32_t st = smem_u32(smem + s * args.stage_bytes);
      const int s_now = s;
      if (++s == S) { s = 0; ph ^= 1; }
#pragma unroll
      for (int gi = 0; gi < kG; ++gi) {
      const int grp = ss * kG + gi;
      if (grp >= G) break;
      const uint32_t stb = st + gi * b_gstep;
      // active token tiles of this unit (uniform across the CTA)
      const int nta = NT == 1 ? 1 : min(NT, (x.nrows + 7) >> 3);
      if (nta <= 1) {
        group_step<WF, AM, kGateUp, NT, 1>(args, st, stb, a_off[gi], b_off, scl[0], scl[1], w, g, t, grp, G, x, nb, tot);
      } else if constexpr (NT >= 2) {
        if (nta == 2 || NT == 2) {
          group_step<WF, AM, kGateUp, NT, (NT >= 2 ? 2 : 1)>(args, st, stb, a_off[gi], b_off, scl[0], scl[1], w, g, t,
                                                            grp, G, x, nb, tot);
        } else if (nta == 3) {
          group_step<WF, AM, kGateUp, NT, (NT >= 3 ? 3 : 1)>(args, st, stb, a_off[gi], b_off, scl[0], scl[1], w, g, t,
                                                            grp, G, x, nb, tot);
        } else {
          group_step<WF, AM, kGateUp, NT, NT>(args, st, stb, a_off[gi], b_off, scl[0], scl[1], w, g, t, grp, G, x, nb,
                                              tot);
        }
      }
      }  // groups of the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[s_now]);  // this stage's codes and tokens are consumed
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->sempty[sb]);
    // epilogue straight from registers
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int tok = j * 8 + 2 * t + (q & 1);
        if (tok >= x.nrows || x.row0 + tok >= args.P) continue;
        const int r = 16 * w + g + 8 * (q >> 1);
        __nv_bfloat16* orow = args.out + static_cast<size_t>(x.row0 + tok) * args.N;
        const float f = AM == AM_F16R ? __ldg(args.a_outer + x.row0 + tok) : 1.f;  // the row's 2^e
        if (kGateUp) {
          const float gv = tot[0][j][q] * f, uv = tot[1][j][q] * f;
          orow[nb + r] = __float2bfloat16_rn(__fdividef(gv, 1.f + __expf(-gv)) * uv);
        } else {
          orow[nb + r] = __float2bfloat16_rn(tot[0][j][q] * f);
          orow[nb + kRowsPerBox + r] = __float2bfloat16_rn(tot[1][j][q] * f);
        }
      }
    }
    if constexpr (kDep == kDepProduce) {
      // this warp's output rows of the unit, visible at GPU scope, to the releaser
      __threadfence();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->udone[sb]);
    }
  }
}

constexpr size_t kSmemPerSm = 232448;
inline size_t smem_limit(int wf, int nt) { return ctas_per_sm(wf, nt) == 2 ? kSmemPerSm / 2 - 1024 : kSmemPerSm; }

// One launch of an instance (sets its shared-memory limit on first use per device).
template <int WF, int AM, bool GU, int NT, int DEP>
cudaError_t launch(const CUtensorMap* maps, const Args& a, size_t smem, int grid, cudaStream_t st) {
  auto kern = moe_gemm_warp_kernel<WF, AM, GU, NT, DEP>;
  static std::atomic<uint64_t> attr{0};
  uint64_t bit;
  if (attrs_needed(attr, &bit)) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_limit(WF, NT)));
    if (e != cudaSuccess) return e;
    attrs_done(attr, bit);
  }
  return launch_pdl(kern, dim3(grid), dim3(threads_for(DEP)), smem, st, maps[0], maps[1], maps[2], a);
}

// The instances that take part in a gate/up -> down tile dependency, compiled
// in their own translation unit (mnw_gemm_warp_dep.cu) to keep builds parallel.
#define MNW_WARP_DEP_INSTANCES(X)                                                                        \
  X(WF_INT4, AM_BF16, true, 1, kDepProduce) X(WF_INT4, AM_BF16, true, 2, kDepProduce)                   \
  X(WF_INT4, AM_BF16, true, 4, kDepProduce) X(WF_INT8, AM_BF16, true, 1, kDepProduce)                   \
  X(WF_INT8, AM_BF16, true, 2, kDepProduce) X(WF_INT8, AM_BF16, true, 4, kDepProduce)                   \
  X(WF_INT4, AM_F16R, true, 1, kDepProduce) X(WF_INT4, AM_F16R, true, 2, kDepProduce)                   \
  X(WF_INT4, AM_F16R, true, 4, kDepProduce) X(WF_INT8, AM_F16R, true, 1, kDepProduce)                   \
  X(WF_INT8, AM_F16R, true, 2, kDepProduce) X(WF_INT8, AM_F16R, true, 4, kDepProduce)                   \
  X(WF_INT4, AM_BF16, false, 1, kDepConsume) X(WF_INT4, AM_BF16, false, 2, kDepConsume)                 \
  X(WF_INT4, AM_BF16, false, 4, kDepConsume) X(WF_INT8, AM_BF16, false, 1, kDepConsume)                 \
  X(WF_INT8, AM_BF16, false, 2, kDepConsume) X(WF_INT8, AM_BF16, false, 4, kDepConsume)

}  // namespace warpmma
}  // namespace mnw
