// mnw_api.cu -- the C ABI of include/mnw_moe.h: argument checks, the expert
// blob header, workspace layout and the whole-layer orchestration.  No call
// here synchronises except mnw_moe_read_error() and mnw_moe_forward_host().
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "mnw_internal.h"

namespace mnw {

static std::atomic<uint64_t> g_launch_count{0};
void note_launch() { g_launch_count.fetch_add(1, std::memory_order_relaxed); }

// ---- tensor maps ------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i < rank - 1) s[i] = strides_bytes[i];
  }
  CUresult r = fn(map, dtype, rank, const_cast<void*>(base), d, s, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---- weight scale range ------------------------------------------------------

// Largest |s| and smallest non-zero |s| over the FP16 group scales of
// `nmat` matrices of every expert (scale arrays at off0 and, for a second
// matrix, off1), as the bits of non-negative FP16 values (their order is the
// order of magnitudes; a NaN compares above every finite value).
static __device__ uint32_t g_scale_max_bits;
static __device__ uint32_t g_scale_min_bits;
__global__ void scale_range_kernel(const uint8_t* experts, uint64_t expert_stride, uint64_t off0, uint64_t off1,
                                   int nmat, uint64_t halfs_per_matrix, int E) {
  uint32_t m = 0, lo = 0xFFFFu;
  const uint64_t per_expert = static_cast<uint64_t>(nmat) * halfs_per_matrix;
  const uint64_t total = static_cast<uint64_t>(E) * per_expert;
  for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const uint64_t e = i / per_expert, rem = i - e * per_expert;
    const uint64_t mat = rem / halfs_per_matrix, j = rem - mat * halfs_per_matrix;
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(experts + e * expert_stride + (mat ? off1 : off0));
    const uint32_t a = __ldg(sc + j) & 0x7FFFu;
    m = max(m, a);
    if (a) lo = min(lo, a);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, d));
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMax(&g_scale_max_bits, m);
    atomicMin(&g_scale_min_bits, lo);
  }
}

// True when fp16(q * s) is finite and, for q != 0 and s != 0, a normal FP16
// number (so it keeps 11 significant bits) for every code q and scale s of the
// gate and up matrices (down = false) or of the down matrix (down = true).
static std::mutex g_scale_range_mu;  // the two device words above serve one check at a time
static bool scales_fit_f16(const mnw_moe_layer& L, bool down) {
  if (L.wfmt != MNW_FMT_INT8_G128 && L.wfmt != MNW_FMT_INT4_G128) return false;
  std::lock_guard<std::mutex> lock(g_scale_range_mu);
  const uint32_t zero = 0, top = 0xFFFFu;
  if (cudaMemcpyToSymbol(g_scale_max_bits, &zero, sizeof(zero)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_scale_min_bits, &top, sizeof(top)) != cudaSuccess)
    return false;
  // gate/up: [I rows][H/128 groups] each; down: [H rows][I/128 groups]
  const uint64_t halfs = static_cast<uint64_t>(L.I) * (L.H / 128);
  if (down)
    scale_range_kernel<<<256, 256>>>(L.blob + L.data_offset, L.expert_stride, L.scales_off[2], L.scales_off[2], 1,
                                     halfs, L.E);
  else
    scale_range_kernel<<<256, 256>>>(L.blob + L.data_offset, L.expert_stride, L.scales_off[0], L.scales_off[1], 2,
                                     halfs, L.E);
  note_launch();
  uint32_t bits = 0xFFFF, lo_bits = 0;
  if (cudaGetLastError() != cudaSuccess || cudaMemcpyFromSymbol(&bits, g_scale_max_bits, sizeof(bits)) != cudaSuccess ||
      cudaMemcpyFromSymbol(&lo_bits, g_scale_min_bits, sizeof(lo_bits)) != cudaSuccess)
    return false;
  if (bits >= 0x7C00u) return false;     // an infinite or NaN scale
  if (lo_bits < 0x0400u) return false;   // a subnormal scale: below 2^-14
  const float smax = __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
  const float qmax = L.wfmt == MNW_FMT_INT8_G128 ? 127.f : 8.f;
  return smax * qmax < 65504.f;
}

// ---- blob header ------------------------------------------------------------

static uint32_t rd32(const uint8_t* p) {
  return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) | (static_cast<uint32_t>(p[2]) << 16) |
         (static_cast<uint32_t>(p[3]) << 24);
}
static uint64_t rd64(const uint8_t* p) { return rd32(p) | (static_cast<uint64_t>(rd32(p + 4)) << 32); }

// CRC-32, reflected polynomial 0xEDB88320, table driven.
static uint32_t crc32(const uint8_t* p, size_t n) {
  static uint32_t table[256];
  static std::once_flag once;
  std::call_once(once, [] {
    for (uint32_t i = 0; i < 256; ++i) {
      uint32_t c = i;
      for (int k = 0; k < 8; ++k) c = (c & 1) ? 0xEDB88320u ^ (c >> 1) : c >> 1;
      table[i] = c;
    }
  });
  uint32_t c = 0xFFFFFFFFu;
  for (size_t i = 0; i < n; ++i) c = table[(c ^ p[i]) & 0xFF] ^ (c >> 8);
  return c ^ 0xFFFFFFFFu;
}

static uint64_t code_bytes(int wfmt, uint64_t N, uint64_t K) {
  switch (wfmt) {
    case MNW_FMT_BF16: return N * K * 2;
    case MNW_FMT_INT8_G128: return N * K;
    default: return N * K / 2;
  }
}
static uint64_t scale_bytes(int wfmt, uint64_t N, uint64_t K) {
  switch (wfmt) {
    case MNW_FMT_INT8_G128:
    case MNW_FMT_INT4_G128: return N * (K / 128) * 2;
    case MNW_FMT_NVFP4_G16: return N * (K / 16);
    default: return 0;
  }
}

static bool act_allowed(int wfmt, int act) {
  if (act == MNW_ACT_BF16) return wfmt != MNW_FMT_NVFP4_G16;
  if (act == MNW_ACT_INT8_G128) return wfmt == MNW_FMT_INT8_G128 || wfmt == MNW_FMT_INT4_G128;
  if (act == MNW_ACT_NVFP4_G16) return wfmt == MNW_FMT_NVFP4_G16;
  return false;
}

// ---- workspace layout ----------------------------------------------------------

struct WsLayout {
  size_t err, dep, rt, rt_zero_end, offsets, sorted, pos;
  size_t xa, xb, xc;   // x operand: bf16 rows | codes, scales, outer
  size_t h, ha, hb, hc;
  size_t y;
  size_t hx, hids, hw, hout;  // staging for the host-buffer entry point
  size_t total, total_host;
};

static size_t al(size_t x) { return (x + 255) / 256 * 256; }

// routed: room for the GPU router's scratch (arrival counters, zeroed with the
// error word, then the logits [T, E]).
static WsLayout ws_layout(const mnw_moe_layer* L, int act, int T, int k, bool routed = false) {
  WsLayout w{};
  const size_t P = static_cast<size_t>(T) * k, H = L->H, I = L->I, E = L->E;
  size_t o = 0;
  w.err = o; o += 256;
  w.dep = o; o = al(o + warp_dep_words(static_cast<int>(P), static_cast<int>(E)) * 4);  // zeroed with err
  w.rt = o;
  if (routed) o = al(o + route_scratch_bytes(T, L->E));
  w.rt_zero_end = routed ? w.rt + route_counter_bytes(T) : w.rt;  // [err, rt_zero_end) is zeroed per call
  w.offsets = o; o = al(o + (E + 1) * 4);
  w.sorted = o; o = al(o + P * 4);
  w.pos = o; o = al(o + P * 4);
  if (act == MNW_ACT_BF16) {
    w.xa = o; o = al(o + P * H * 2);  // BF16 rows, or FP16 rows for the FP16 operand path
    w.xc = o; o = al(o + P * 4);      // their row factors (FP16 operand path)
  } else if (act == MNW_ACT_INT8_G128) {
    w.xa = o; o = al(o + P * H);
    w.xb = o; o = al(o + P * (H / 128) * 4);
  } else {
    w.xa = o; o = al(o + P * H / 2);
    w.xb = o; o = al(o + P * H / 16);
    w.xc = o; o = al(o + P * 4);
  }
  w.h = o; o = al(o + P * I * 2);
  if (act == MNW_ACT_BF16 && (L->wfmt == MNW_FMT_INT8_G128 || L->wfmt == MNW_FMT_INT4_G128)) {
    w.ha = o; o = al(o + P * I * 2);  // h as FP16 rows (FP16 operand down GEMM)
    w.hc = o; o = al(o + P * 4);      // their row factors
  } else if (act == MNW_ACT_INT8_G128) {
    w.ha = o; o = al(o + P * I);
    w.hb = o; o = al(o + P * (I / 128) * 4);
  } else if (act == MNW_ACT_NVFP4_G16) {
    w.ha = o; o = al(o + P * I / 2);
    w.hb = o; o = al(o + P * I / 16);
    w.hc = o; o = al(o + P * 4);
  }
  w.y = o; o = al(o + P * (H > 2 * I ? H : 2 * I) * 2);  // y, or g and u of the unfused gate/up
  w.total = o;
  w.hx = o; o = al(o + static_cast<size_t>(T) * H * 2);
  w.hids = o; o = al(o + P * 4);
  w.hw = o; o = al(o + P * 4);
  w.hout = o; o = al(o + static_cast<size_t>(T) * H * 2);
  w.total_host = o;
  return w;
}

static int gemm_for(const mnw_moe_layer* L, int act, int kind, const void* a0, const void* a1, const void* a2,
                    const int32_t* offsets, int P, void* out, uint32_t* err, uint32_t* sched, cudaStream_t st) {
  return run_gemm(L, L->wfmt, act, kind, a0, a1, a2, offsets, P, out, nullptr, err, st, sched);
}

}  // namespace mnw

namespace mnw {
int gemm_path();
}
using namespace mnw;

extern "C" {

static int g_gemm_path = MNW_PATH_AUTO;
static std::atomic<int> g_fused_activation{1};
static std::atomic<int> g_host_routing{0};
int mnw_moe_set_host_routing(int on) {
  if (on != 0 && on != 1) return MNW_E_INVALID_ARG;
  g_host_routing.store(on);
  return MNW_OK;
}
int mnw_moe_set_fused_activation(int fused) {
  if (fused != 0 && fused != 1) return MNW_E_INVALID_ARG;
  g_fused_activation.store(fused);
  return MNW_OK;
}

int mnw_moe_silu_mul(const void* g, const void* u, size_t n, void* h, mnw_stream stream) {
  MNW_RANGE("mnw_moe_silu_mul");
  if (n == 0) return MNW_OK;
  if (!g || !u || !h || n % 8 || !aligned(g, 16) || !aligned(u, 16) || !aligned(h, 16)) return MNW_E_INVALID_ARG;
  return launch_silu_mul(g, u, n, h, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MNW_OK : MNW_E_CUDA;
}
int mnw_moe_set_gemm_path(int path) {
  if (path < MNW_PATH_AUTO || path > MNW_PATH_ROWS) return MNW_E_INVALID_ARG;
  g_gemm_path = path;
  return MNW_OK;
}

uint64_t mnw_moe_launch_count(void) { return g_launch_count.load(std::memory_order_relaxed); }

const char* mnw_status_string(int status) {
  switch (status) {
    case MNW_OK: return "ok";
    case MNW_E_INVALID_ARG: return "invalid argument";
    case MNW_E_UNSUPPORTED: return "unsupported shape";
    case MNW_E_BAD_BLOB: return "bad expert blob";
    case MNW_E_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MNW_E_CUDA: return "CUDA error";
    case MNW_E_MODE: return "activation mode not allowed for this weight format";
    default: return "unknown status";
  }
}

int mnw_moe_layer_init(const void* header_host, const void* blob_dev, size_t blob_bytes, mnw_moe_layer** out) {
  MNW_RANGE("mnw_moe_layer_init");
  if (!header_host || !blob_dev || !out) return MNW_E_INVALID_ARG;
  *out = nullptr;
  if (!aligned(blob_dev, 256)) return MNW_E_INVALID_ARG;
  const uint8_t* h = static_cast<const uint8_t*>(header_host);
  if (std::memcmp(h, "MNWB", 4) != 0 || rd32(h + 4) != 1 || rd32(h + 28) != 256) return MNW_E_BAD_BLOB;
  if (crc32(h, 252) != rd32(h + 252)) return MNW_E_BAD_BLOB;
  mnw_moe_layer L{};
  L.wfmt = static_cast<int>(rd32(h + 8));
  L.E = static_cast<int>(rd32(h + 12));
  L.H = static_cast<int>(rd32(h + 16));
  L.I = static_cast<int>(rd32(h + 20));
  L.group = static_cast<int>(rd32(h + 24));
  L.data_offset = rd64(h + 32);
  L.expert_stride = rd64(h + 40);
  for (int m = 0; m < 3; ++m) {
    L.codes_off[m] = rd64(h + 48 + 8 * m);
    L.scales_off[m] = rd64(h + 72 + 8 * m);
    L.outer_off[m] = rd64(h + 96 + 8 * m);
  }
  const uint64_t total = rd64(h + 120);
  if (L.wfmt < 0 || L.wfmt > 3 || L.E < 1 || L.E > 1024 || L.H <= 0 || L.I <= 0) return MNW_E_BAD_BLOB;
  const int want_group[4] = {0, 128, 128, 16};
  if (L.group != want_group[L.wfmt]) return MNW_E_BAD_BLOB;
  if (L.H % 128 || L.I % 128) return MNW_E_UNSUPPORTED;
  // INT4 and NVFP4 stream 256 K values (128 bytes) per row and stage.
  if ((L.wfmt == MNW_FMT_NVFP4_G16 || L.wfmt == MNW_FMT_INT4_G128) && (L.H % 256 || L.I % 256))
    return MNW_E_UNSUPPORTED;
  if (total > blob_bytes || L.data_offset % 256 || L.expert_stride % 256 ||
      L.data_offset + static_cast<uint64_t>(L.E) * L.expert_stride > total)
    return MNW_E_BAD_BLOB;
  L.blob = static_cast<const uint8_t*>(blob_dev);
  L.blob_bytes = blob_bytes;
  for (int m = 0; m < 3; ++m) {
    const uint64_t N = m == 2 ? L.H : L.I, K = m == 2 ? L.I : L.H;
    if (L.codes_off[m] % 256 || L.codes_off[m] + code_bytes(L.wfmt, N, K) > L.expert_stride) return MNW_E_BAD_BLOB;
    if (scale_bytes(L.wfmt, N, K) &&
        (L.scales_off[m] % 256 || L.scales_off[m] + scale_bytes(L.wfmt, N, K) > L.expert_stride))
      return MNW_E_BAD_BLOB;
    if (L.wfmt == MNW_FMT_NVFP4_G16 && (L.outer_off[m] % 4 || L.outer_off[m] + 4 > L.expert_stride))
      return MNW_E_BAD_BLOB;
  }
  if (cudaGetDevice(&L.device) != cudaSuccess) return MNW_E_CUDA;
  if (cudaDeviceGetAttribute(&L.num_sms, cudaDevAttrMultiProcessorCount, L.device) != cudaSuccess)
    return MNW_E_CUDA;
  // Weight tensor maps: every expert's matrix m seen as one 3-D tensor [E][N][row].
  const uint8_t* experts = L.blob + L.data_offset;
  for (int m = 0; m < 3; ++m) {
    const uint64_t N = m == 2 ? L.H : L.I, K = m == 2 ? L.I : L.H;
    bool ok;
    if (L.wfmt == MNW_FMT_BF16) {
      const uint64_t dims[3] = {K, N, static_cast<uint64_t>(L.E)};
      const uint64_t strides[2] = {K * 2, L.expert_stride};
      const uint32_t box[3] = {64, 128, 1};
      ok = encode_map(&L.tm_codes[m], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, experts + L.codes_off[m], dims, strides,
                      box, CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
      const uint64_t row = code_bytes(L.wfmt, 1, K);
      const uint64_t dims[3] = {row, N, static_cast<uint64_t>(L.E)};
      const uint64_t strides[2] = {row, L.expert_stride};
      const uint32_t box[3] = {128, 128, 1};
      ok = encode_map(&L.tm_codes[m], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, experts + L.codes_off[m], dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B);
      if (ok && L.wfmt == MNW_FMT_INT4_G128) {  // the warp-MMA kernel's one-group stages
        const uint32_t box64[3] = {64, 128, 1};
        ok = encode_map(&L.tm_codes64[m], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, experts + L.codes_off[m], dims, strides,
                        box64, CU_TENSOR_MAP_SWIZZLE_64B);
      }
    }
    if (ok && L.wfmt == MNW_FMT_NVFP4_G16) {
      const uint64_t dims[3] = {K / 16, N, static_cast<uint64_t>(L.E)};
      const uint64_t strides[2] = {K / 16, L.expert_stride};
      const uint32_t box[3] = {16, 128, 1};
      ok = encode_map(&L.tm_sf[m], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, experts + L.scales_off[m], dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (!ok) return MNW_E_CUDA;
  }
  // one small reduction over the gate/up scales (reads the blob, synchronises)
  L.f16_gate_up_ok = scales_fit_f16(L, false);
  L.f16_down_ok = scales_fit_f16(L, true);
  mnw_moe_layer* p = new (std::nothrow) mnw_moe_layer(L);
  if (!p) return MNW_E_INVALID_ARG;
  *out = p;
  return MNW_OK;
}

void mnw_moe_layer_destroy(mnw_moe_layer* layer) { delete layer; }

int mnw_moe_layer_info(const mnw_moe_layer* L, int* wfmt, int* E, int* H, int* I) {
  if (!L) return MNW_E_INVALID_ARG;
  if (wfmt) *wfmt = L->wfmt;
  if (E) *E = L->E;
  if (H) *H = L->H;
  if (I) *I = L->I;
  return MNW_OK;
}

int mnw_moe_permute(const int32_t* ids, int T, int k, int E, int32_t* expert_offsets, int32_t* sorted_assign,
                    int32_t* assign_pos, const void* x, int H, void* x_perm, uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_moe_permute");
  if (T < 0 || k < 1 || k > 32 || E < 1 || E > 1024) return MNW_E_INVALID_ARG;
  if (static_cast<long long>(T) * k > (1LL << 24)) return MNW_E_UNSUPPORTED;
  if (T == 0) return MNW_OK;
  if (!ids || !expert_offsets || !sorted_assign || !assign_pos) return MNW_E_INVALID_ARG;
  if ((x == nullptr) != (x_perm == nullptr)) return MNW_E_INVALID_ARG;
  if (x && (H <= 0 || H % 8 || !aligned(x, 16) || !aligned(x_perm, 16))) return MNW_E_INVALID_ARG;
  cudaError_t e = launch_permute(ids, T, k, E, expert_offsets, sorted_assign, assign_pos, x, H, x_perm, err,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MNW_OK : MNW_E_CUDA;
}

int mnw_moe_permute_host(const int32_t* ids, int T, int k, int E, int32_t* expert_offsets, int32_t* sorted_assign,
                         int32_t* assign_pos, uint32_t* dropped) {
  MNW_RANGE("mnw_moe_permute_host");
  if (T < 0 || k < 1 || k > 32 || E < 1 || E > 1024) return MNW_E_INVALID_ARG;
  if (static_cast<long long>(T) * k > (1LL << 24)) return MNW_E_UNSUPPORTED;
  if (dropped) *dropped = 0;
  if (T == 0) return MNW_OK;
  if (!ids || !expert_offsets || !sorted_assign || !assign_pos) return MNW_E_INVALID_ARG;
  const int P = T * k;
  // counting sort by expert: counts, exclusive offsets, then one stable pass
  for (int e = 0; e <= E; ++e) expert_offsets[e] = 0;
  uint32_t bad = 0;
  for (int a = 0; a < P; ++a) {
    const int id = ids[a];
    if (id >= 0 && id < E) ++expert_offsets[id + 1];
    else ++bad;
  }
  for (int e = 0; e < E; ++e) expert_offsets[e + 1] += expert_offsets[e];
  std::vector<int32_t> next(expert_offsets, expert_offsets + E);
  for (int a = 0; a < P; ++a) {
    const int id = ids[a];
    if (id >= 0 && id < E) {
      const int pos = next[id]++;
      assign_pos[a] = pos;
      sorted_assign[pos] = a;
    } else {
      assign_pos[a] = -1;
    }
  }
  for (int p = expert_offsets[E]; p < P; ++p) sorted_assign[p] = -1;  // slots past the valid count
  if (dropped) *dropped = bad;
  return MNW_OK;
}

int mnw_moe_quantize_act(int act, const void* x, int R, int K, const int32_t* row_index, int index_div, void* codes,
                         void* scales, float* row_outer, mnw_stream stream) {
  MNW_RANGE("mnw_moe_quantize_act");
  if (R < 0 || K <= 0) return MNW_E_INVALID_ARG;
  if (row_index && index_div < 1) return MNW_E_INVALID_ARG;
  if (act == MNW_ACT_F16_ROWS) {
    if (K % 8) return MNW_E_UNSUPPORTED;
    if (R == 0) return MNW_OK;
    if (!x || !codes || !row_outer || !aligned(x, 16) || !aligned(codes, 16) || !aligned(row_outer, 4))
      return MNW_E_INVALID_ARG;
    cudaError_t e = launch_gather_f16(x, K, row_index, R, row_index ? index_div : 1, codes, row_outer,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MNW_OK : MNW_E_CUDA;
  }
  if (act == MNW_ACT_INT8_G128) {
    if (K % 128) return MNW_E_UNSUPPORTED;
  } else if (act == MNW_ACT_NVFP4_G16) {
    if (K % 16) return MNW_E_UNSUPPORTED;
    if (!row_outer || !aligned(row_outer, 4)) return MNW_E_INVALID_ARG;
  } else {
    return MNW_E_INVALID_ARG;
  }
  if (R == 0) return MNW_OK;
  if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4))
    return MNW_E_INVALID_ARG;
  cudaError_t e = launch_quantize(act, x, R, K, row_index, index_div, codes, scales, row_outer,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MNW_OK : MNW_E_CUDA;
}

int mnw_moe_grouped_gemm_bf16(const mnw_moe_layer* L, int kind, const void* a, const int32_t* offs, int P, void* out,
                              uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_moe_grouped_gemm_bf16");
  return run_gemm(L, MNW_FMT_BF16, MNW_ACT_BF16, kind, a, nullptr, nullptr, offs, P, out, nullptr, err,
                  static_cast<cudaStream_t>(stream));
}
int mnw_moe_grouped_gemm_w8a16(const mnw_moe_layer* L, int kind, const void* a, const int32_t* offs, int P, void* out,
                               uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_moe_grouped_gemm_w8a16");
  return run_gemm(L, MNW_FMT_INT8_G128, MNW_ACT_BF16, kind, a, nullptr, nullptr, offs, P, out, nullptr, err,
                  static_cast<cudaStream_t>(stream));
}
int mnw_moe_grouped_gemm_w4a16(const mnw_moe_layer* L, int kind, const void* a, const int32_t* offs, int P, void* out,
                               uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_moe_grouped_gemm_w4a16");
  return run_gemm(L, MNW_FMT_INT4_G128, MNW_ACT_BF16, kind, a, nullptr, nullptr, offs, P, out, nullptr, err,
                  static_cast<cudaStream_t>(stream));
}
static int gemm_f16rows(const mnw_moe_layer* L, int wfmt, int kind, const void* a, const float* f,
                        const int32_t* offs, int P, void* out, uint32_t* err, cudaStream_t st) {
  if (!L || kind < MNW_KIND_GATE_UP || kind > MNW_KIND_UP) return MNW_E_INVALID_ARG;
  if (L->wfmt != wfmt) return MNW_E_MODE;
  if (!(kind == MNW_KIND_DOWN ? L->f16_down_ok : L->f16_gate_up_ok)) return MNW_E_UNSUPPORTED;
  return run_gemm(L, wfmt, kActF16Rows, kind, a, f, nullptr, offs, P, out, nullptr, err, st);
}
int mnw_moe_grouped_gemm_w8a16_f16rows(const mnw_moe_layer* L, int kind, const void* a, const float* f,
                                       const int32_t* offs, int P, void* out, uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_moe_grouped_gemm_w8a16_f16rows");
  return gemm_f16rows(L, MNW_FMT_INT8_G128, kind, a, f, offs, P, out, err, static_cast<cudaStream_t>(stream));
}
int mnw_moe_grouped_gemm_w4a16_f16rows(const mnw_moe_layer* L, int kind, const void* a, const float* f,
                                       const int32_t* offs, int P, void* out, uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_moe_grouped_gemm_w4a16_f16rows");
  return gemm_f16rows(L, MNW_FMT_INT4_G128, kind, a, f, offs, P, out, err, static_cast<cudaStream_t>(stream));
}
int mnw_moe_grouped_gemm_w8a8(const mnw_moe_layer* L, int kind, const int8_t* q, const float* s, const int32_t* offs,
                              int P, void* out, int32_t* dots, uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_moe_grouped_gemm_w8a8");
  return run_gemm(L, MNW_FMT_INT8_G128, MNW_ACT_INT8_G128, kind, q, s, nullptr, offs, P, out, dots, err,
                  static_cast<cudaStream_t>(stream));
}
int mnw_moe_grouped_gemm_w4a8(const mnw_moe_layer* L, int kind, const int8_t* q, const float* s, const int32_t* offs,
                              int P, void* out, int32_t* dots, uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_moe_grouped_gemm_w4a8");
  return run_gemm(L, MNW_FMT_INT4_G128, MNW_ACT_INT8_G128, kind, q, s, nullptr, offs, P, out, dots, err,
                  static_cast<cudaStream_t>(stream));
}
int mnw_moe_grouped_gemm_nvfp4(const mnw_moe_layer* L, int kind, const uint8_t* c, const uint8_t* sf, const float* o,
                               const int32_t* offs, int P, void* out, uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_moe_grouped_gemm_nvfp4");
  return run_gemm(L, MNW_FMT_NVFP4_G16, MNW_ACT_NVFP4_G16, kind, c, sf, o, offs, P, out, nullptr, err,
                  static_cast<cudaStream_t>(stream));
}

int mnw_moe_combine(const void* y, const int32_t* assign_pos, const float* w, int T, int k, int H, void* out,
                    mnw_stream stream) {
  MNW_RANGE("mnw_moe_combine");
  if (T < 0 || k < 1 || k > 32 || H <= 0 || H % 8) return MNW_E_INVALID_ARG;
  if (T == 0) return MNW_OK;
  if (!y || !assign_pos || !w || !out || !aligned(y, 16) || !aligned(out, 16)) return MNW_E_INVALID_ARG;
  cudaError_t e = launch_combine(y, assign_pos, w, T, k, H, out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MNW_OK : MNW_E_CUDA;
}

size_t mnw_moe_workspace_size(const mnw_moe_layer* L, int act, int T, int k) {
  if (!L || T < 0 || k < 1) return 0;
  return ws_layout(L, act, T, k).total;
}
size_t mnw_moe_workspace_size_host(const mnw_moe_layer* L, int act, int T, int k) {
  if (!L || T < 0 || k < 1) return 0;
  return ws_layout(L, act, T, k).total_host;
}
uint32_t* mnw_moe_workspace_error_word(void* ws) { return static_cast<uint32_t*>(ws); }

}  // extern "C"

// The layer.  With wr (router weights) non-null the ids and weights come from
// the GPU router (written to ids_out / w_out), whose launch also produces the
// permutation; the steps that would permute then only gather rows.
static int forward_impl(const mnw_moe_layer* L, int act, const void* x, const int32_t* ids, const float* w,
                        const void* wr, int32_t* ids_out, float* w_out, int T, int k, void* out, void* ws,
                        size_t ws_bytes, mnw_stream stream) {
  if (!L || T < 0 || k < 1 || k > 32 || k > L->E) return MNW_E_INVALID_ARG;
  if (!act_allowed(L->wfmt, act)) return MNW_E_MODE;
  if (T == 0) return MNW_OK;
  const bool routed = wr != nullptr;
  if (routed && (!ids_out || !w_out || !aligned(wr, 16) || !route_shape_ok(T, L->H, L->E, k)))
    return MNW_E_INVALID_ARG;
  if (!routed && (!ids || !w)) return MNW_E_INVALID_ARG;
  if (!x || !out || !ws || !aligned(x, 16) || !aligned(out, 16) || !aligned(ws, 256)) return MNW_E_INVALID_ARG;
  const WsLayout W = ws_layout(L, act, T, k, routed);
  if (ws_bytes < W.total) return MNW_E_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* b = static_cast<uint8_t*>(ws);
  uint32_t* err = reinterpret_cast<uint32_t*>(b + W.err);
  int32_t* offs = reinterpret_cast<int32_t*>(b + W.offsets);
  int32_t* sorted = reinterpret_cast<int32_t*>(b + W.sorted);
  int32_t* pos = reinterpret_cast<int32_t*>(b + W.pos);
  const int P = T * k, H = L->H, I = L->I;
  // The first 256 bytes of ws: error word, then a [claim, done] work counter per GEMM launch.
  uint32_t* sched_gu = err + 16;
  uint32_t* sched_dn = err + 18;
  if (cudaMemsetAsync(err, 0, W.rt_zero_end - W.err, st) != cudaSuccess) return MNW_E_CUDA;  // error word, counters
  int rc0;
  if (routed && !host_routing()) {
    if (launch_route(x, wr, T, L->H, L->E, k, ids_out, w_out, offs, sorted, pos, b + W.rt, err, st) != cudaSuccess)
      return MNW_E_CUDA;
  } else if (routed) {
    // Host routing: logits on the GPU, copied to the host; top-k, softmax and
    // the permutation on the host; the results copied back (synchronises).
    float* logits = reinterpret_cast<float*>(b + W.rt + route_counter_bytes(T));
    const size_t TE = static_cast<size_t>(T) * L->E, Pk = static_cast<size_t>(P);
    std::vector<float> lg(TE), wh(Pk);
    std::vector<int32_t> ih(Pk), oh(L->E + 1), sh(Pk), ph(Pk);
    if (launch_route_logits(x, wr, T, L->H, L->E, logits, st) != cudaSuccess ||
        cudaMemcpyAsync(lg.data(), logits, TE * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return MNW_E_CUDA;
    route_topk_host(lg.data(), T, L->E, k, ih.data(), wh.data());
    rc0 = mnw_moe_permute_host(ih.data(), T, k, L->E, oh.data(), sh.data(), ph.data(), nullptr);
    if (rc0) return rc0;
    if (cudaMemcpyAsync(ids_out, ih.data(), Pk * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(w_out, wh.data(), Pk * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(offs, oh.data(), (L->E + 1) * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(sorted, sh.data(), Pk * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(pos, ph.data(), Pk * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)  // the host vectors go out of scope below
      return MNW_E_CUDA;
  }
  if (routed) {
    ids = ids_out;
    w = w_out;
  }
  // gate/up: fused (SiLU in the GEMM epilogue), or the unfused comparison path:
  // gate and up as single-matrix GEMMs into the y region, then the activation
  const bool fused = fused_activation();
  auto gate_up = [&](int gact, const void* a0, const void* a1, const void* a2, const WarpDep* dep) -> int {
    if (fused)
      return run_gemm(L, L->wfmt, gact, MNW_KIND_GATE_UP, a0, a1, a2, offs, P, b + W.h, nullptr, err, st, sched_gu,
                      dep);
    uint8_t* g = b + W.y;
    uint8_t* u = g + static_cast<size_t>(P) * I * 2;
    int r = run_gemm(L, L->wfmt, gact, MNW_KIND_GATE, a0, a1, a2, offs, P, g, nullptr, err, st);
    if (r) return r;
    r = run_gemm(L, L->wfmt, gact, MNW_KIND_UP, a0, a1, a2, offs, P, u, nullptr, err, st);
    if (r) return r;
    return launch_silu_mul(g, u, static_cast<size_t>(P) * I, b + W.h, st) == cudaSuccess ? MNW_OK : MNW_E_CUDA;
  };
  // the permutation, optionally gathering x rows (routed: already permuted, gather only)
  auto permute = [&](const void* gx, void* gx_perm) -> int {
    if (!routed) return mnw_moe_permute(ids, T, k, L->E, offs, sorted, pos, gx, gx ? H : 0, gx_perm, err, stream);
    if (!gx) return MNW_OK;
    return launch_gather_rows(gx, H, sorted, P, k, gx_perm, st) == cudaSuccess ? MNW_OK : MNW_E_CUDA;
  };
  int rc;
  if (act == MNW_ACT_BF16) {
    // INT weights: the GEMMs run on FP16 rows (scaled into FP16 range by a
    // power of two per row).  On the tcgen05 kernel (enough tokens per
    // expert) the weights are dequantised on chip to fp16(q * s), so one
    // accumulator spans all of K; on the warp-MMA kernel the INT4 codes
    // convert to FP16 operands in fewer instructions than to BF16.
    const int mean_rows = (P + L->E - 1) / L->E;
    const int path = gemm_path();
    const bool tc = path != MNW_PATH_WARP_MMA && (path == MNW_PATH_TCGEN05 || path == MNW_PATH_ROWS || mean_rows >= 32);
    const int gu_act = L->f16_gate_up_ok ? kActF16Rows : act;
    // Both GEMMs on the warp-MMA kernel (same token tile): the down launch
    // follows the gate/up launch tile by tile instead of waiting for all of it.
    const bool warp_down = fused && !tc && warp_gemm_applicable(L, L->wfmt, gu_act, MNW_KIND_GATE_UP) &&
                           warp_gemm_applicable(L, L->wfmt, act, MNW_KIND_DOWN);
    const WarpDep gu_dep{reinterpret_cast<uint32_t*>(b + W.dep), kDepProduce, 0};
    if (L->f16_gate_up_ok) {
      rc = permute(nullptr, nullptr);
      if (rc) return rc;
      float* factor = reinterpret_cast<float*>(b + W.xc);
      rc = mnw_moe_quantize_act(MNW_ACT_F16_ROWS, x, P, H, sorted, k, b + W.xa, nullptr, factor, stream);
      if (rc) return rc;
      rc = gate_up(kActF16Rows, b + W.xa, factor, nullptr, warp_down ? &gu_dep : nullptr);
    } else {
      rc = permute(x, b + W.xa);
      if (rc) return rc;
      rc = gate_up(act, b + W.xa, nullptr, nullptr, warp_down ? &gu_dep : nullptr);
    }
    if (rc) return rc;
    if (warp_down) {
      // both GEMMs on the warp-MMA kernel: down starts tile by tile behind gate/up
      const WarpDep dn{reinterpret_cast<uint32_t*>(b + W.dep), kDepConsume, warp_dep_need_gate_up(L)};
      rc = run_gemm(L, L->wfmt, act, MNW_KIND_DOWN, b + W.h, nullptr, nullptr, offs, P, b + W.y, nullptr, err, st,
                    sched_dn, &dn);
    } else if (tc && L->f16_down_ok) {
      float* hf = reinterpret_cast<float*>(b + W.hc);
      rc = mnw_moe_quantize_act(MNW_ACT_F16_ROWS, b + W.h, P, I, nullptr, 1, b + W.ha, nullptr, hf, stream);
      if (rc) return rc;
      rc = gemm_for(L, kActF16Rows, MNW_KIND_DOWN, b + W.ha, hf, nullptr, offs, P, b + W.y, err, sched_dn, st);
    } else {
      rc = gemm_for(L, act, MNW_KIND_DOWN, b + W.h, nullptr, nullptr, offs, P, b + W.y, err, sched_dn, st);
    }
    if (rc) return rc;
  } else {
    rc = permute(nullptr, nullptr);
    if (rc) return rc;
    float* xo = act == MNW_ACT_NVFP4_G16 ? reinterpret_cast<float*>(b + W.xc) : nullptr;
    float* ho = act == MNW_ACT_NVFP4_G16 ? reinterpret_cast<float*>(b + W.hc) : nullptr;
    // each token row quantised once, its codes written to its k positions
    if (launch_quantize_scatter(act, x, T, H, pos, k, b + W.xa, b + W.xb, xo, st) != cudaSuccess) return MNW_E_CUDA;
    rc = gate_up(act, b + W.xa, b + W.xb, xo, nullptr);
    if (rc) return rc;
    rc = mnw_moe_quantize_act(act, b + W.h, P, I, nullptr, 1, b + W.ha, b + W.hb, ho, stream);
    if (rc) return rc;
    rc = gemm_for(L, act, MNW_KIND_DOWN, b + W.ha, b + W.hb, ho, offs, P, b + W.y, err, sched_dn, st);
    if (rc) return rc;
  }
  return mnw_moe_combine(b + W.y, pos, w, T, k, H, out, stream);
}

extern "C" {

int mnw_moe_forward(const mnw_moe_layer* L, int act, const void* x, const int32_t* ids, const float* w, int T, int k,
                    void* out, void* ws, size_t ws_bytes, mnw_stream stream) {
  MNW_RANGE("mnw_moe_forward");
  if (T > 0 && (!ids || !w)) return MNW_E_INVALID_ARG;
  return forward_impl(L, act, x, ids, w, nullptr, nullptr, nullptr, T, k, out, ws, ws_bytes, stream);
}

size_t mnw_moe_workspace_size_routed(const mnw_moe_layer* L, int act, int T, int k) {
  if (!L || T < 0 || k < 1) return 0;
  return ws_layout(L, act, T, k, true).total;
}

int mnw_moe_forward_routed(const mnw_moe_layer* L, int act, const void* x, const void* w_router, int T, int k,
                           int32_t* ids_out, float* w_out, void* out, void* ws, size_t ws_bytes, mnw_stream stream) {
  MNW_RANGE("mnw_moe_forward_routed");
  if (T > 0 && !w_router) return MNW_E_INVALID_ARG;
  return forward_impl(L, act, x, nullptr, nullptr, w_router, ids_out, w_out, T, k, out, ws, ws_bytes, stream);
}

size_t mnw_moe_route_scratch_size(int T, int E) {
  if (T < 0 || E < 1) return 0;
  return route_scratch_bytes(T, E);
}

int mnw_moe_route(const void* x, const void* w_router, int T, int H, int E, int k, int32_t* ids, float* w,
                  int32_t* expert_offsets, int32_t* sorted_assign, int32_t* assign_pos, void* scratch,
                  size_t scratch_bytes, uint32_t* err, mnw_stream stream) {
  MNW_RANGE("mnw_moe_route");
  if (!route_shape_ok(T, H, E, k)) return MNW_E_INVALID_ARG;
  if (T == 0) return MNW_OK;
  if (!x || !w_router || !ids || !w || !expert_offsets || !sorted_assign || !assign_pos || !scratch ||
      !aligned(x, 16) || !aligned(w_router, 16) || !aligned(scratch, 256))
    return MNW_E_INVALID_ARG;
  if (scratch_bytes < route_scratch_bytes(T, E)) return MNW_E_WORKSPACE_TOO_SMALL;
  const cudaError_t e = launch_route(x, w_router, T, H, E, k, ids, w, expert_offsets, sorted_assign, assign_pos,
                                     scratch, err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MNW_OK : MNW_E_CUDA;
}

// The device address of a host buffer the GPU can read and write in place
// (page-locked and mapped into the unified address space), or null for
// pageable memory, which then goes through a staging copy.
static void* mapped_alias(const void* host, size_t align) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();  // clear the error of a pointer CUDA does not know
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer || !aligned(a.devicePointer, align)) return nullptr;
  return a.devicePointer;
}

int mnw_moe_forward_host(const mnw_moe_layer* L, int act, const void* x_host, const int32_t* ids_host,
                         const float* w_host, int T, int k, void* out_host, void* ws, size_t ws_bytes,
                         mnw_stream stream) {
  MNW_RANGE("mnw_moe_forward_host");
  if (!L || T < 0 || k < 1) return MNW_E_INVALID_ARG;
  if (T == 0) return MNW_OK;
  if (!x_host || !ids_host || !w_host || !out_host || !ws) return MNW_E_INVALID_ARG;
  const WsLayout W = ws_layout(L, act, T, k);
  if (ws_bytes < W.total_host) return MNW_E_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* b = static_cast<uint8_t*>(ws);
  const size_t xb = static_cast<size_t>(T) * L->H * 2, ib = static_cast<size_t>(T) * k * 4;
  // ids and w (read once, by the permute and the combine) and out (written
  // once, by the combine) are used in place when they are mapped page-locked
  // memory; x is always staged, as the gather reads each row k times.
  const void* ids_d = mapped_alias(ids_host, 4);
  const void* w_d = mapped_alias(w_host, 4);
  void* out_d = mapped_alias(out_host, 16);
  if (cudaMemcpyAsync(b + W.hx, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess) return MNW_E_CUDA;
  if (!ids_d) {
    if (cudaMemcpyAsync(b + W.hids, ids_host, ib, cudaMemcpyHostToDevice, st) != cudaSuccess) return MNW_E_CUDA;
    ids_d = b + W.hids;
  }
  if (!w_d) {
    if (cudaMemcpyAsync(b + W.hw, w_host, ib, cudaMemcpyHostToDevice, st) != cudaSuccess) return MNW_E_CUDA;
    w_d = b + W.hw;
  }
  int rc = mnw_moe_forward(L, act, b + W.hx, static_cast<const int32_t*>(ids_d), static_cast<const float*>(w_d), T,
                           k, out_d ? out_d : b + W.hout, ws, W.total, stream);
  if (rc) return rc;
  if (!out_d && cudaMemcpyAsync(out_host, b + W.hout, xb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MNW_E_CUDA;
  // The error word goes to host stack memory: a stream-ordered copy into
  // pageable memory returns only once it, and so everything before it on the
  // stream (the output copy included), has completed -- one wait, not two.
  uint32_t e = 0;
  if (cudaMemcpyAsync(&e, b + W.err, sizeof(e), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MNW_E_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MNW_E_CUDA;
  return e ? MNW_E_CUDA : MNW_OK;
}

int mnw_moe_read_error(const uint32_t* err, uint32_t* out_host, mnw_stream stream) {
  if (!err || !out_host) return MNW_E_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MNW_E_CUDA;
  if (cudaMemcpy(out_host, err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MNW_E_CUDA;
  return MNW_OK;
}

}  // extern "C"

namespace mnw {
int gemm_path() { return g_gemm_path; }
bool fused_activation() { return g_fused_activation.load() != 0; }
bool host_routing() { return g_host_routing.load() != 0; }

int current_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];  // 0 = not looked up yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}
}  // namespace mnw
