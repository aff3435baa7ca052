// mnw_internal.h -- host-side state shared by the library's translation units.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/mnw_moe.h"

struct mnw_moe_layer {
  int wfmt, E, H, I, group;
  const uint8_t* blob;        // device, borrowed
  size_t blob_bytes;
  uint64_t data_offset, expert_stride;
  uint64_t codes_off[3], scales_off[3], outer_off[3];
  int device, num_sms;
  // INT weights: every fp16(q * s) of the gate/up (resp. down) matrices is
  // finite and normal (checked once at init), so those GEMMs may run on FP16
  // operands.
  bool f16_gate_up_ok, f16_down_ok;
  // Weight tensor maps (built once): codes per matrix, NVFP4 block scales per matrix.
  CUtensorMap tm_codes[3];
  CUtensorMap tm_codes64[3];  // INT4 codes in 64-byte boxes (one 128-K group), 64-byte swizzle
  CUtensorMap tm_sf[3];
};

namespace mnw {

// The expert matrix a grouped GEMM of `kind` reads first (gate/up: gate, then up).
inline int kind_matrix(int kind) { return kind == MNW_KIND_DOWN ? 2 : (kind == MNW_KIND_UP ? 1 : 0); }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Number of SMs of the current device, looked up once per device.
int current_sm_count();

// Launch a kernel of this library with programmatic stream serialisation: it
// may start while the previous kernel on the stream finishes (its set-up
// overlaps that kernel's tail), and waits for that kernel's completion with
// pdl_wait() before it touches global memory.  After a non-kernel stream
// operation (a copy, a memset, an event) the launch is an ordinary one.
// Kernel attributes are per device: `done` keeps one bit per device (0..63)
// on which a kernel's attributes have been set.  Setting them twice, from two
// threads, is harmless.
inline bool attrs_needed(const std::atomic<uint64_t>& done, uint64_t* bit) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *bit = 0;
    return true;  // unknown device: set them every time
  }
  *bit = 1ull << dev;
  return (done.load(std::memory_order_acquire) & *bit) == 0;
}
inline void attrs_done(std::atomic<uint64_t>& done, uint64_t bit) { done.fetch_or(bit, std::memory_order_release); }

// An NVTX range named after the C-ABI call it covers, for profiler timelines
// (a no-op unless a tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define MNW_RANGE(name) ::mnw::NvtxRange mnw_nvtx_range_(name)

// Count of kernels this library has enqueued (mnw_moe_launch_count).
void note_launch();

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
  if (e == cudaSuccess) note_launch();
  return e;
}

// Encode a tiled tensor map; returns false on failure.
bool encode_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle);

// Launchers (arguments already validated by the ABI functions).
cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets, int32_t* sorted_assign,
                           int32_t* assign_pos, const void* x, int H, void* x_perm, uint32_t* err,
                           cudaStream_t st);
// h = bf16(SiLU(g) * u) elementwise over n BF16 values (n % 8 == 0, 16-byte aligned).
cudaError_t launch_silu_mul(const void* g, const void* u, size_t n, void* h, cudaStream_t st);
// Process-wide: the forward's gate/up runs fused (SiLU in the GEMM epilogue) or
// as two single-matrix GEMMs and the activation step.
bool fused_activation();
// x_perm[p] = x[sorted_assign[p] / k] (zero rows where sorted_assign[p] < 0).
cudaError_t launch_gather_rows(const void* x, int H, const int32_t* sorted_assign, int P, int k, void* x_perm,
                               cudaStream_t st);
// GPU routing fused with the permutation (mnw_router.cu): ids/w for every
// token and the permutation of them; scratch = [arrival counters | logits].
size_t route_scratch_bytes(int T, int E);
bool route_shape_ok(int T, int H, int E, int k);
cudaError_t launch_route(const void* x, const void* wr, int T, int H, int E, int k, int32_t* ids, float* w,
                         int32_t* offsets, int32_t* sorted_assign, int32_t* assign_pos, void* scratch, uint32_t* err,
                         cudaStream_t st);
// Host routing (a comparison path): the router's logits only, then the top-k
// and softmax on the host with the same rule.
cudaError_t launch_route_logits(const void* x, const void* wr, int T, int H, int E, float* logits, cudaStream_t st);
void route_topk_host(const float* logits, int T, int E, int k, int32_t* ids, float* w);
bool host_routing();
// Bytes at the start of the route scratch that hold its arrival counters.
inline size_t route_counter_bytes(int T) { return ((1 + (static_cast<size_t>(T) + 15) / 16) * 4 + 255) / 256 * 256; }
// MNW_ACT_F16_ROWS encoding of P rows (row p reads x[row_index[p] / div], or
// x[p] without row_index): FP16 codes into x_perm, power-of-two factors.
cudaError_t launch_gather_f16(const void* x, int H, const int32_t* row_index, int P, int div, void* x_perm,
                              float* factor, cudaStream_t st);
cudaError_t launch_combine(const void* y, const int32_t* assign_pos, const float* w, int T, int k, int H,
                           void* out, cudaStream_t st);
cudaError_t launch_quantize(int act, const void* x, int R, int K, const int32_t* row_index, int index_div,
                            void* codes, void* scales, float* row_outer, cudaStream_t st);
// The forward path's form: each of the R source rows (tokens) is quantised
// once and written to the output rows row_index[r * index_div + j] >= 0
// (row_index = assign_pos, index_div = k).
cudaError_t launch_quantize_scatter(int act, const void* x, int R, int K, const int32_t* row_index, int index_div,
                            void* codes, void* scales, float* row_outer, cudaStream_t st);
// Activation mode of the FP16 operand gate/up GEMM (INT weights): a0 = FP16
// rows from launch_gather_f16, a1 = their float factors.
constexpr int kActF16Rows = MNW_ACT_F16_ROWS;
// Tile-level dependency between the gate/up and the down warp-MMA launches of
// one forward step.  The gate/up launch (kDepProduce) adds one to flags[1 + t]
// when all its MMA warps have written token tile t's h rows of a row block,
// and sets flags[0] once its own wait on the previous kernel has returned.  The down launch (kDepConsume) waits for flags[0] instead of for
// the gate/up launch to complete, so its CTAs start as gate/up CTAs retire,
// and reads token tile t only once flags[1 + t] >= need.  flags is zeroed
// before the gate/up launch; both launches use the same token tile.
enum { kDepNone = 0, kDepProduce = 1, kDepConsume = 2 };
struct WarpDep {
  uint32_t* flags;
  int role;
  uint32_t need;
};
// Token tiles of any warp-MMA launch over P rows of E experts (8-row tiles at least).
inline size_t warp_dep_words(int P, int E) { return static_cast<size_t>(P) / 8 + E + 2; }
// Count a token tile's counter reaches when the gate/up launch has written all its h rows
// (its number of row blocks).
uint32_t warp_dep_need_gate_up(const mnw_moe_layer* L);
// Grouped GEMM for weight format wfmt and activation mode act.
// sched (nullable): a zeroed device counter that lets the kernel's CTAs claim
// work units dynamically; NULL gives a static round-robin order.
int run_gemm(const mnw_moe_layer* L, int wfmt, int act, int kind, const void* a0, const void* a1,
             const void* a2, const int32_t* offsets, int P, void* out, int32_t* dots, uint32_t* err,
             cudaStream_t st, uint32_t* sched = nullptr, const WarpDep* dep = nullptr);
// Warp-MMA grouped GEMM (INT8/INT4 weights, few tokens per expert); nt = token tile / 8.
bool warp_gemm_applicable(const mnw_moe_layer* L, int wfmt, int act, int kind);
int run_gemm_warp(const mnw_moe_layer* L, int wfmt, int act, int kind, const void* a0, const void* a1,
                  const int32_t* offsets, int P, int nt, void* out, int32_t* dots, uint32_t* err, uint32_t* sched,
                  cudaStream_t st, const WarpDep* dep = nullptr);
// Row-tile tcgen05 GEMM (tokens as M, 256 weight rows as N; mnw_gemm_rows.cu):
// FP16 rows on INT8/INT4 weights, BF16 rows on BF16 weights.
bool rows_gemm_applicable(const mnw_moe_layer* L, int wfmt, int act, int kind);
int run_gemm_rows(const mnw_moe_layer* L, int wfmt, int act, int kind, const void* a0, const void* a1,
                  const int32_t* offsets, int P, void* out, uint32_t* err, cudaStream_t st);
// Row-tile tcgen05 GEMM for INT8 weights with INT8 activations (tokens as M,
// 128 weight rows as N, one accumulator per 128-K group; mnw_gemm_rows_a8.cu).
bool rows_a8_applicable(const mnw_moe_layer* L, int wfmt, int act, int kind);
int run_gemm_rows_a8(const mnw_moe_layer* L, int kind, const void* a_codes, const float* a_scales,
                     const int32_t* offsets, int P, void* out, int32_t* dots, uint32_t* err, cudaStream_t st);
// Token tile (in 8-row units) the warp-MMA kernel uses for P rows over E experts.
int warp_gemm_nt(int P, int E);
// Process-wide GEMM path selection (MNW_PATH_*).
int gemm_path();

}  // namespace mnw
