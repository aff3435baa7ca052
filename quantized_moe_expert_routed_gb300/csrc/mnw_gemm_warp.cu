// mnw_gemm_warp.cu -- host side of the warp-MMA grouped GEMM (mnw_gemm_warp.cuh):
// launch shapes, shared-memory plan, tensor maps, dispatch.
#include "mnw_gemm_warp.cuh"

namespace mnw {
namespace warpmma {

// compiled in mnw_gemm_warp_dep.cu
#define MNW_WARP_DEP_EXTERN(WF, AM, GU, NT, DEP) \
  extern template cudaError_t launch<WF, AM, GU, NT, DEP>(const CUtensorMap*, const Args&, size_t, int, cudaStream_t);
MNW_WARP_DEP_INSTANCES(MNW_WARP_DEP_EXTERN)
#undef MNW_WARP_DEP_EXTERN

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {
inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <int WF, int AM, bool GU, int DEP>
cudaError_t launch_nt(int nt, const CUtensorMap* maps, const Args& a, size_t smem, int grid, cudaStream_t st) {
  switch (nt) {
    case 1: return launch<WF, AM, GU, 1, DEP>(maps, a, smem, grid, st);
    case 2: return launch<WF, AM, GU, 2, DEP>(maps, a, smem, grid, st);
    default: return launch<WF, AM, GU, 4, DEP>(maps, a, smem, grid, st);
  }
}
// Dependency roles exist for the forward path's pairing only: a gate/up launch
// on 16-bit rows produces, a down launch on BF16 rows consumes.
template <int WF, int AM>
cudaError_t launch_kind(bool gu, int nt, int dep, const CUtensorMap* maps, const Args& a, size_t smem, int grid,
                        cudaStream_t st) {
  if (gu) {
    if constexpr (AM != AM_INT8) {
      if (dep == kDepProduce) return launch_nt<WF, AM, true, kDepProduce>(nt, maps, a, smem, grid, st);
    }
    if (dep != kDepNone) return cudaErrorInvalidValue;
    return launch_nt<WF, AM, true, kDepNone>(nt, maps, a, smem, grid, st);
  }
  if constexpr (AM == AM_BF16) {
    if (dep == kDepConsume) return launch_nt<WF, AM, false, kDepConsume>(nt, maps, a, smem, grid, st);
  }
  if (dep != kDepNone) return cudaErrorInvalidValue;
  return launch_nt<WF, AM, false, kDepNone>(nt, maps, a, smem, grid, st);
}
}  // namespace

}  // namespace warpmma

uint32_t warp_dep_need_gate_up(const mnw_moe_layer* L) {
  return static_cast<uint32_t>(L->I / warpmma::kRowsPerBox);  // one release per row block of a token tile
}

bool warp_gemm_applicable(const mnw_moe_layer* L, int wfmt, int act, int kind) {
  if (wfmt != MNW_FMT_INT8_G128 && wfmt != MNW_FMT_INT4_G128) return false;
  if (act != MNW_ACT_BF16 && act != MNW_ACT_INT8_G128 && act != kActF16Rows) return false;
  if (kind == MNW_KIND_GATE_UP) return L->I % warpmma::kRowsPerBox == 0;
  return (kind == MNW_KIND_DOWN ? L->H : L->I) % (2 * warpmma::kRowsPerBox) == 0;
}

int run_gemm_warp(const mnw_moe_layer* L, int wfmt, int act, int kind, const void* a0, const void* a1,
                  const int32_t* offsets, int P, int nt, void* out, int32_t* dots, uint32_t* err, uint32_t* sched,
                  cudaStream_t st, const WarpDep* dep) {
  using namespace warpmma;
  const bool gu = kind == MNW_KIND_GATE_UP;
  const int K = kind == MNW_KIND_DOWN ? L->I : L->H, N = kind == MNW_KIND_DOWN ? L->H : L->I, G = K / 128;
  const int BN = 8 * nt;
  Args a{};
  a.offsets = offsets;
  a.E = L->E;
  a.P = P;
  a.K = K;
  a.N = N;
  a.BN = BN;
  a.n_blocks = gu ? N / kRowsPerBox : N / (2 * kRowsPerBox);
  const bool int4 = wfmt == MNW_FMT_INT4_G128;
  const int a_boxes = int4 ? 1 : 2;                // code boxes per 128-row block per stage
  const int kg = groups_per_stage(int4 ? WF_INT4 : WF_INT8);
  a.box_bytes = int4 ? kBox64Bytes : kBoxBytes;
  a.off_b = 2 * a_boxes * a.box_bytes;
  const bool act16 = act != MNW_ACT_INT8_G128;  // BF16 or FP16 rows
  const uint32_t b_bytes = (act16 ? 2u : 1u) * kg * BN * 128u;
  a.stage_bytes = align_up(a.off_b + b_bytes, 1024);
  a.scale_box_bytes = kRowsPerBox * G * 2;
  const uint32_t fixed = 4 * a.scale_box_bytes + align_up(2u * (L->E + 1) * 4u, 16) + align_up(sizeof(Bars), 16);
  const size_t budget = smem_limit(wfmt, nt) - 1024;
  if (fixed + 2 * a.stage_bytes > budget) return MNW_E_UNSUPPORTED;
  int stages = static_cast<int>((budget - fixed) / a.stage_bytes);
  a.stages = stages > kMaxStages ? kMaxStages : stages;
  a.off_scales = a.stages * a.stage_bytes;
  a.off_tab = a.off_scales + 4 * a.scale_box_bytes;
  a.off_bars = align_up(a.off_tab + 2u * (L->E + 1) * 4u, 16);
  const size_t smem = a.off_bars + sizeof(Bars) + 1024;
  a.experts = L->blob + L->data_offset;
  a.expert_stride = L->expert_stride;
  const int m0 = kind_matrix(kind), m1 = gu ? 1 : m0;
  a.scales_off[0] = L->scales_off[m0];
  a.scales_off[1] = L->scales_off[m1];
  a.box_row_off[0] = 0;
  a.box_row_off[1] = gu ? 0 : kRowsPerBox;
  a.a_scales = act == MNW_ACT_INT8_G128 ? static_cast<const float*>(a1) : nullptr;
  a.a_outer = act == kActF16Rows ? static_cast<const float*>(a1) : nullptr;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.dots = act == MNW_ACT_INT8_G128 ? dots : nullptr;
  a.err = err;
  a.sched = sched;  // NULL (a standalone call): static work order
  if (dep && dep->role != kDepNone) {
    if (!dep->flags || !sched) return MNW_E_INVALID_ARG;
    a.dep = dep->flags;
    a.dep_role = dep->role;
    a.dep_need = dep->need;
  }

  CUtensorMap maps[3];
  maps[0] = int4 ? L->tm_codes64[m0] : L->tm_codes[m0];
  maps[1] = int4 ? L->tm_codes64[m1] : L->tm_codes[m1];
  const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(P)};
  bool ok;
  if (act16) {
    const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(BN)};
    ok = encode_map(&maps[2], act == MNW_ACT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    a0, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const uint64_t strides[1] = {static_cast<uint64_t>(K)};
    const uint32_t box[2] = {128, static_cast<uint32_t>(BN)};
    ok = encode_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a0, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return MNW_E_INVALID_ARG;
  const int grid = L->num_sms * ctas_per_sm(wfmt, nt);
  cudaError_t e;
  const int role = a.dep_role;
  if (wfmt == MNW_FMT_INT4_G128 && act == MNW_ACT_BF16) e = launch_kind<WF_INT4, AM_BF16>(gu, nt, role, maps, a, smem, grid, st);
  else if (wfmt == MNW_FMT_INT8_G128 && act == MNW_ACT_BF16) e = launch_kind<WF_INT8, AM_BF16>(gu, nt, role, maps, a, smem, grid, st);
  else if (wfmt == MNW_FMT_INT4_G128 && act == kActF16Rows) e = launch_kind<WF_INT4, AM_F16R>(gu, nt, role, maps, a, smem, grid, st);
  else if (wfmt == MNW_FMT_INT8_G128 && act == kActF16Rows) e = launch_kind<WF_INT8, AM_F16R>(gu, nt, role, maps, a, smem, grid, st);
  else if (wfmt == MNW_FMT_INT4_G128) e = launch_kind<WF_INT4, AM_INT8>(gu, nt, role, maps, a, smem, grid, st);
  else e = launch_kind<WF_INT8, AM_INT8>(gu, nt, role, maps, a, smem, grid, st);
  return e == cudaSuccess ? MNW_OK : MNW_E_CUDA;
}

}  // namespace mnw
