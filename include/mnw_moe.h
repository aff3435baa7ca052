/*
 * mnw_moe.h -- C ABI of the GB300 (sm_103a) routed-expert MoE layer.
 *
 * The layer: every token t has k routed experts ids[t, 0..k) with routing
 * weights w[t, 0..k).  Each expert e is a SwiGLU feed-forward block,
 *   h = SiLU(x . Wg[e]^T) * (x . Wu[e]^T)      Wg, Wu: [I, H]
 *   y = h . Wd[e]^T                             Wd: [H, I]
 * and out[t] = sum_j w[t, j] * y(t, j).  The expert matrices are stored in one
 * of the quantised formats of the "LLaDA2.2-flash-minnow" model card,
 * section "Checkpoints and precision" (precision table): BF16; signed INT8 or
 * signed INT4 with one FP16 scale per 128 weights; NVFP4 (E2M1 values, E4M3
 * scale per 16, FP32 outer scale per expert matrix).  The "coder543/minnow"
 * README, section "Quantization", gives the execution modes: INT4/INT8
 * weights dequantised to BF16 (W4A16/W8A16); the optional INT8 activation
 * mode (W4A8/W8A8: activations quantised per group of 128 with an FP32 scale,
 * INT32 group dot products, scales applied in FP32); NVFP4 W4A4 with
 * activations quantised to E2M1 / E4M3-per-16 / FP32-per-row.  The
 * README also names a fused gate/up/SiLU step and grouping the tokens of a
 * 32-token decode block by expert on the GPU.
 *
 * Conventions for every call below
 *  - Pointers marked "device" are CUDA device pointers owned by the caller;
 *    the library never allocates, frees or keeps them.  Device buffers must be
 *    16-byte aligned; the expert blob must be 256-byte aligned.
 *  - Work is enqueued on `stream` and the call returns without synchronising,
 *    except mnw_moe_read_error() and mnw_moe_forward_host(), which say so.
 *  - BF16 tensors are row-major arrays of 16-bit bfloat16 values.
 *  - A return value other than MNW_OK means nothing was enqueued.  Errors that
 *    only the device can see (an expert id outside [0, E), a wait that ran out)
 *    are OR-ed into a caller-provided 32-bit device error word (MNW_DEVERR_*)
 *    that the caller zeroes beforehand and reads with mnw_moe_read_error().
 *  - Results are deterministic: no floating-point atomics.
 *  - The grouped-GEMM entry points keep no state between calls: calls may
 *    overlap on different streams and may be captured in a CUDA graph and
 *    replayed on any stream.  (mnw_moe_forward keeps its work counters in the
 *    caller's workspace: calls sharing one workspace must not overlap.)
 *  - Per-device state (kernel attributes, the address of
 *    mnw_moe_forward_static's array) is set up on first use; do not use the
 *    library after cudaDeviceReset() in the same process.
 *  - Kernels are launched with programmatic stream serialisation: one may
 *    start its set-up while the kernel before it on the stream finishes, but
 *    waits for that kernel's completion before it reads or writes any global
 *    memory, so ordering against the caller's own work on the stream is the
 *    usual one.  They also allow the next kernel to start early; a caller
 *    that launches its next kernel with the same attribute must wait
 *    (griddepcontrol.wait / cudaGridDependencySynchronize) before reading
 *    this library's outputs.
 *
 * Expert blob layout (defined by this library; little-endian):
 *   bytes [0, 256): header.  char[4] "MNWB"; u32 version = 1; u32 wfmt
 *   (mnw_wfmt); u32 E; u32 H; u32 I; u32 group (0 BF16, 128 INT8/INT4, 16
 *   NVFP4); u32 header_bytes = 256; u64 data_offset; u64 expert_stride;
 *   u64 codes_off[3]; u64 scales_off[3]; u64 outer_off[3] (gate, up, down,
 *   relative to the expert's start); u64 total_bytes; zero padding; u32
 *   CRC-32 (IEEE 802.3) of bytes [0, 252) stored at byte 252.
 *   Expert e starts at data_offset + e * expert_stride (a multiple of 256).
 *   Each matrix [N][K] (gate/up: N = I, K = H; down: N = H, K = I) is stored
 *   row-major, K fastest, every section 256-byte aligned:
 *     BF16:  u16 codes [N][K]
 *     INT8:  i8 codes [N][K];   f16 scales [N][K/128]
 *     INT4:  u8 codes [N][K/2] (element 2c in the low nibble of byte c);
 *            f16 scales [N][K/128]
 *     NVFP4: u8 codes [N][K/2] (same nibble order); E4M3 scales [N][K/16];
 *            f32 outer scale (one per matrix)
 *   H and I must be multiples of 128 (INT4 and NVFP4: multiples of 256).
 */
#ifndef MNW_MOE_H
#define MNW_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif
/* The library is built with hidden visibility: only what this header
 * declares is exported. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

/* A CUDA stream (cudaStream_t); 0 is the legacy default stream. */
typedef void* mnw_stream;

enum mnw_status {
  MNW_OK = 0,
  MNW_E_INVALID_ARG = 1,        /* null/misaligned pointer, negative size, bad enum */
  MNW_E_UNSUPPORTED = 2,        /* shape outside what the kernels support */
  MNW_E_BAD_BLOB = 3,           /* header magic/version/CRC/sizes do not check out */
  MNW_E_WORKSPACE_TOO_SMALL = 4,
  MNW_E_CUDA = 5,               /* a CUDA runtime call failed */
  MNW_E_MODE = 6                /* activation mode not allowed for the weight format */
};

/* Bits of the device error word. */
#define MNW_DEVERR_BAD_EXPERT_ID 0x1u  /* an id outside [0, E); that assignment was dropped */
#define MNW_DEVERR_TIMEOUT 0x2u        /* a kernel-internal wait ran out; its output is invalid */

enum mnw_wfmt { MNW_FMT_BF16 = 0, MNW_FMT_INT8_G128 = 1, MNW_FMT_INT4_G128 = 2, MNW_FMT_NVFP4_G16 = 3 };
/* MNW_ACT_F16_ROWS is an operand form, not a layer mode: BF16 rows re-encoded
 * as FP16 with a power-of-two factor per row (mnw_moe_quantize_act), read by
 * the *_f16rows gate/up GEMMs.  mnw_moe_forward picks it by itself. */
enum mnw_afmt { MNW_ACT_BF16 = 0, MNW_ACT_INT8_G128 = 1, MNW_ACT_NVFP4_G16 = 2, MNW_ACT_F16_ROWS = 3 };
/* GATE / UP: the gate or the up matrix alone, out (bf16 [P, I]) = bf16(a .
 * W^T) -- the unfused-activation comparison path ("coder543/minnow" README,
 * "Quantization": --unfused-activation), whose activation then runs as
 * mnw_moe_silu_mul(). */
enum mnw_kind { MNW_KIND_GATE_UP = 0, MNW_KIND_DOWN = 1, MNW_KIND_GATE = 2, MNW_KIND_UP = 3 };

typedef struct mnw_moe_layer mnw_moe_layer;

/* Human-readable name of a status code (static storage). */
const char* mnw_status_string(int status);

/* Describe an expert blob.  `header_host` is a host copy of the blob's first
 * 256 bytes; `blob_dev` the whole blob in device memory (borrowed, not
 * copied; it must outlive the layer).  Validates magic, version, CRC and the
 * section sizes against `blob_bytes`.  On success *out is a host object
 * released by mnw_moe_layer_destroy(). */
int mnw_moe_layer_init(const void* header_host, const void* blob_dev, size_t blob_bytes,
                       mnw_moe_layer** out);
void mnw_moe_layer_destroy(mnw_moe_layer* layer);
/* Shape of a layer: any output pointer may be NULL. */
int mnw_moe_layer_info(const mnw_moe_layer* layer, int* wfmt, int* E, int* H, int* I);

/* a1 -- token permutation: grouping the assignments by expert on the GPU
 * ("coder543/minnow" README, section "Quantization").
 * ids: device int32 [T*k], assignment a = t*k + j goes to expert ids[a].
 * Writes (device): expert_offsets int32 [E+1] (exclusive prefix of the
 * per-expert counts; expert_offsets[E] = number of valid assignments),
 * sorted_assign int32 [T*k] (sorted_assign[p] = a; slots past the valid count
 * hold -1), assign_pos int32 [T*k] (inverse map; -1 for a dropped id).
 * Positions are stable: within an expert, assignments keep increasing a.
 * If x (device bf16 [T, H]) and x_perm (device bf16 [T*k, H]) are both
 * non-NULL, also gathers x_perm[p] = x[sorted_assign[p] / k] (zeros where
 * sorted_assign[p] is -1).  An id outside [0, E) sets MNW_DEVERR_BAD_EXPERT_ID
 * in *err (device, may be NULL) and is dropped.  Limits: 1 <= k <= 32,
 * 1 <= E <= 1024, T*k <= 2^24.  T = 0 is a no-op. */
int mnw_moe_permute(const int32_t* ids, int T, int k, int E, int32_t* expert_offsets,
                    int32_t* sorted_assign, int32_t* assign_pos, const void* x, int H,
                    void* x_perm, uint32_t* err, mnw_stream stream);
/* The same permutation computed on the host, for a host-routing comparison
 * path ("coder543/minnow" README, "Quantization": --host-routing): ids,
 * expert_offsets, sorted_assign and assign_pos are HOST arrays with the
 * layouts above, and the results are identical to mnw_moe_permute's.
 * *dropped (may be NULL) receives the number of ids outside [0, E).  Needs
 * no GPU.  Same limits as mnw_moe_permute. */
int mnw_moe_permute_host(const int32_t* ids, int T, int k, int E, int32_t* expert_offsets,
                         int32_t* sorted_assign, int32_t* assign_pos, uint32_t* dropped);

/* GPU routing fused with the permutation (the step before a1 on the decode
 * path): the "coder543/minnow" README, section "Quantization", routes the
 * 32-token decode blocks on the GPU; the "LLaDA2.2-flash-minnow" model card,
 * "Checkpoints and precision", keeps routers in their source floating point.
 * The pages give no formula; the rule used here:
 *   logits[t, e] = x[t] . w_router[e]   (BF16 inputs, FP32 accumulation in a
 *                                        fixed order: reproducible bits)
 *   ids[t, 0..k) = the k largest logits of row t, largest first, the lower
 *                  expert index first among equal logits (NaN ranks last)
 *   w[t, j]      = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k chosen (FP32)
 * then expert_offsets, sorted_assign and assign_pos exactly as
 * mnw_moe_permute() gives for those ids.
 * x: device bf16 [T, H]; w_router: device bf16 [E, H]; ids: device int32
 * [T, k]; w: device f32 [T, k]; the permutation outputs as mnw_moe_permute.
 * scratch: device, 256-byte aligned, >= mnw_moe_route_scratch_size(T, E)
 * bytes.  It starts with arrival counters that must be zero before the first
 * call (a zero-filled buffer) and that every completed call leaves at zero;
 * the rest receives the logits [T, E] (f32, row-major).  Calls sharing one
 * scratch must not overlap.  err (device, nullable) as for mnw_moe_permute.
 * One kernel launch when T*k <= 4096 (the permutation runs in its last CTA);
 * larger batches add the permutation's own launches.  Limits: H % 128 == 0,
 * 1 <= k <= min(E, 32), E <= 1024.  T = 0 is a no-op. */
size_t mnw_moe_route_scratch_size(int T, int E);
int mnw_moe_route(const void* x, const void* w_router, int T, int H, int E, int k, int32_t* ids, float* w,
                  int32_t* expert_offsets, int32_t* sorted_assign, int32_t* assign_pos, void* scratch,
                  size_t scratch_bytes, uint32_t* err, mnw_stream stream);

/* a2 -- dynamic activation quantisation of R rows of K BF16 values.
 * Row r reads x[src] with src = r, or, when row_index (device int32 [R]) is
 * non-NULL, src = row_index[r] / index_div (a negative row_index gives a
 * zero row).  act = MNW_ACT_INT8_G128 ("LLaDA2.2-flash-minnow" model card,
 * W8A8 paragraph): per 128 values, scale = amax / 127 (FP32),
 * code = clamp(rne(x / scale), -127, 127); codes int8 [R, K], scales f32
 * [R, K/128]; row_outer unused.  act = MNW_ACT_NVFP4_G16 (model card, NVFP4
 * row): outer = amax_row / 2688; per 16 values sb = e4m3_rn_satfinite(
 * (amax_block / outer) / 6), code = e2m1_rn_satfinite(x / (sb * outer));
 * codes u8 [R, K/2] (even element in the low nibble), scales E4M3 u8
 * [R, K/16], row_outer f32 [R].  Every step is one IEEE binary32 operation
 * with round-to-nearest-even; the results are bit-exact.  K must be a
 * multiple of 128 (INT8) or 16 (NVFP4).
 * act = MNW_ACT_F16_ROWS (an exact re-encoding, not a quantiser of the
 * pages): e = clamp(floor(log2 amax_row) - 14, -110, 113) (-110 for a zero
 * row), row_outer = 2^e, codes fp16 [R, K] = fp16_rn(x * 2^-e); scales
 * unused (may be NULL); a negative row_index gives codes 0 and row_outer 1.
 * Every BF16 value of a row no more than 2^28 below its largest magnitude
 * is kept exactly.  K must be a multiple of 8. */
int mnw_moe_quantize_act(int act, const void* x, int R, int K, const int32_t* row_index,
                         int index_div, void* codes, void* scales, float* row_outer,
                         mnw_stream stream);

/* a3/a4/a6 -- grouped expert GEMMs.  Rows [expert_offsets[e],
 * expert_offsets[e+1]) of the activation operand belong to expert e
 * (expert_offsets: device int32 [E+1], as written by mnw_moe_permute).
 * kind = MNW_KIND_GATE_UP: K = H, out (device bf16 [P, I]) =
 *   bf16(SiLU(a . Wg^T) * (a . Wu^T)), the gate/up/SiLU fusion of the minnow
 *   README, "Quantization".
 * kind = MNW_KIND_DOWN: K = I, out (device bf16 [P, H]) = bf16(a . Wd^T).
 * Accumulation is FP32 on the tensor cores.
 *
 * bf16 / w8a16 / w4a16: a is device bf16 [P, K]; the weights (BF16, INT8 or
 * INT4 with FP16 group scales) are dequantised on chip on their way into the
 * BF16 tensor cores, with no expanded copy in memory ("LLaDA2.2-flash-minnow"
 * model card, paragraph after the precision table).  INT codes enter as exact
 * BF16 integers; each 128-wide group's dot product is scaled by its FP16
 * scale and summed in FP32. */
int mnw_moe_grouped_gemm_bf16(const mnw_moe_layer* layer, int kind, const void* a,
                              const int32_t* expert_offsets, int P, void* out, uint32_t* err,
                              mnw_stream stream);
int mnw_moe_grouped_gemm_w8a16(const mnw_moe_layer* layer, int kind, const void* a,
                               const int32_t* expert_offsets, int P, void* out, uint32_t* err,
                               mnw_stream stream);
int mnw_moe_grouped_gemm_w4a16(const mnw_moe_layer* layer, int kind, const void* a,
                               const int32_t* expert_offsets, int P, void* out, uint32_t* err,
                               mnw_stream stream);
/* w8a16_f16rows / w4a16_f16rows: the grouped GEMMs of the W8A16/W4A16 modes
 * on FP16 tensor cores.  a: device fp16 [P, K] and row_outer device f32 [P]
 * from mnw_moe_quantize_act(MNW_ACT_F16_ROWS); each weight enters as
 * fp16_rn(q * s) (its code times its FP16 group scale, one rounding), one
 * FP32 accumulator spans all of K, and the row factor f multiplies each dot
 * product: GATE_UP out = bf16(SiLU(f * (a . Wg^T)) * (f * (a . Wu^T))), DOWN
 * out = bf16(f * (a . Wd^T)).  MNW_E_UNSUPPORTED when some q * s of the
 * matrices used would leave FP16's normal range (a scale above 65504 / qmax,
 * qmax = 127 or 8, or a non-zero scale below 2^-14); mnw_moe_forward then
 * keeps the BF16 form for that GEMM.  A call with P = 0 launches nothing and
 * only reports that: MNW_OK if the layer admits the form for `kind`,
 * MNW_E_UNSUPPORTED if not.  Kernel choice as for the other INT
 * entries: below 32 tokens per expert on average the warp-MMA kernel, where
 * the codes stay exact FP16 integers and each group's FP32 dot product is
 * scaled by s afterwards (no fp16(q * s) rounding there). */
int mnw_moe_grouped_gemm_w8a16_f16rows(const mnw_moe_layer* layer, int kind, const void* a,
                                       const float* row_outer, const int32_t* expert_offsets, int P,
                                       void* out, uint32_t* err, mnw_stream stream);
int mnw_moe_grouped_gemm_w4a16_f16rows(const mnw_moe_layer* layer, int kind, const void* a,
                                       const float* row_outer, const int32_t* expert_offsets, int P,
                                       void* out, uint32_t* err, mnw_stream stream);
/* w8a8 / w4a8 (model card, W8A8/W4A8 paragraph): a_codes device int8 [P, K]
 * and a_scales device f32 [P, K/128] from mnw_moe_quantize_act(INT8_G128).
 * For every 128-wide group g the exact integer dot product D_g of the codes is
 * formed, then out accumulates (s_w * s_a) * D_g in FP32.  group_dots (device
 * int32, may be NULL) receives every D_g, layout [P][C][K/128] with
 * C = 2*I (gate columns, then up columns) or H: a test hook. */
int mnw_moe_grouped_gemm_w8a8(const mnw_moe_layer* layer, int kind, const int8_t* a_codes,
                              const float* a_scales, const int32_t* expert_offsets, int P,
                              void* out, int32_t* group_dots, uint32_t* err, mnw_stream stream);
int mnw_moe_grouped_gemm_w4a8(const mnw_moe_layer* layer, int kind, const int8_t* a_codes,
                              const float* a_scales, const int32_t* expert_offsets, int P,
                              void* out, int32_t* group_dots, uint32_t* err, mnw_stream stream);
/* nvfp4 (model card, NVFP4 row): a_codes device u8 [P, K/2], a_sf device
 * E4M3 u8 [P, K/16], a_outer device f32 [P] from
 * mnw_moe_quantize_act(NVFP4_G16).  out = sum of block-scaled products times
 * outer_w[e] * a_outer[p]. */
int mnw_moe_grouped_gemm_nvfp4(const mnw_moe_layer* layer, int kind, const uint8_t* a_codes,
                               const uint8_t* a_sf, const float* a_outer,
                               const int32_t* expert_offsets, int P, void* out, uint32_t* err,
                               mnw_stream stream);

/* The activation step of the unfused comparison path ("coder543/minnow"
 * README, "Quantization": --unfused-activation): h[i] = bf16(SiLU(g[i]) *
 * u[i]), SiLU(g) = g / (1 + e^-g), in FP32 from BF16 g and u (device bf16
 * arrays of n values, n % 8 == 0; h device bf16 [n]).  The fused GEMMs
 * evaluate the same expression on the FP32 dot products instead of their BF16
 * roundings. */
int mnw_moe_silu_mul(const void* g, const void* u, size_t n, void* h, mnw_stream stream);

/* a5 -- combine: out[t] = bf16(sum_j w[t, j] * y[assign_pos[t*k + j]]) with
 * FP32 accumulation in ascending j; assignments with assign_pos < 0 are
 * skipped.  y: device bf16 [P, H]; assign_pos: device int32 [T*k];
 * w: device f32 [T, k]; out: device bf16 [T, H].  H % 8 == 0. */
int mnw_moe_combine(const void* y, const int32_t* assign_pos, const float* w, int T, int k,
                    int H, void* out, mnw_stream stream);

/* The whole layer: permute -> (quantise x) -> gate/up/SiLU -> (quantise h)
 * -> down -> combine, all on `stream`, with every intermediate in `ws`
 * (device, at least mnw_moe_workspace_size() bytes, 256-byte aligned).  act
 * must suit the weight format: BF16 for BF16/INT8/INT4 weights, INT8_G128
 * for INT8/INT4 weights, NVFP4_G16 for NVFP4 weights.  x: device bf16
 * [T, H]; ids: device int32 [T, k]; w: device f32 [T, k]; out: device bf16
 * [T, H].  The device error word is the first 4 bytes of ws
 * (mnw_moe_workspace_error_word); it is cleared by this call. */
size_t mnw_moe_workspace_size(const mnw_moe_layer* layer, int act, int T, int k);
int mnw_moe_forward(const mnw_moe_layer* layer, int act, const void* x, const int32_t* ids,
                    const float* w, int T, int k, void* out, void* ws, size_t ws_bytes,
                    mnw_stream stream);
uint32_t* mnw_moe_workspace_error_word(void* ws);

/* The whole layer with GPU routing: mnw_moe_route() on x and w_router (device
 * bf16 [E, H]), then the layer exactly as mnw_moe_forward() with those ids and
 * weights (the router's launch already holds the permutation).  ids_out
 * (device int32 [T, k]) and w_out (device f32 [T, k]) receive the router's
 * choices.  ws: >= mnw_moe_workspace_size_routed() bytes; the router's
 * counters live in it and are cleared by every call. */
size_t mnw_moe_workspace_size_routed(const mnw_moe_layer* layer, int act, int T, int k);
/* Host routing, process-wide (the "coder543/minnow" README, "Quantization":
 * --host-routing, a comparison path; default 0): mnw_moe_forward_routed then
 * computes the logits on the GPU, copies them to the host, picks the top-k and
 * the softmax weights (same rule, FP32 host arithmetic) and the permutation
 * (as mnw_moe_permute_host) on the host, and copies ids, weights and the
 * permutation back before running the layer.  The call then synchronises
 * `stream` twice and uses host memory of its own (T*E floats and the routing
 * arrays) for the duration of the call.  Not synchronised with calls in flight
 * on other threads. */
int mnw_moe_set_host_routing(int on);
int mnw_moe_forward_routed(const mnw_moe_layer* layer, int act, const void* x, const void* w_router, int T,
                           int k, int32_t* ids_out, float* w_out, void* out, void* ws, size_t ws_bytes,
                           mnw_stream stream);

/* The whole layer from and to HOST buffers: copies x into ws, runs
 * mnw_moe_forward, and synchronises `stream`.  ids, w and out are used in
 * place when they are page-locked memory mapped into the device's address
 * space (e.g. cudaHostAlloc on a unified-addressing system; the kernels then
 * read ids and w and write out over the host link), otherwise they are
 * staged through ws with copies on `stream`.  ws must hold
 * mnw_moe_workspace_size_host() bytes.  Returns MNW_E_CUDA if the device
 * error word is non-zero afterwards. */
size_t mnw_moe_workspace_size_host(const mnw_moe_layer* layer, int act, int T, int k);
int mnw_moe_forward_host(const mnw_moe_layer* layer, int act, const void* x_host,
                         const int32_t* ids_host, const float* w_host, int T, int k,
                         void* out_host, void* ws, size_t ws_bytes, mnw_stream stream);

/* Number of kernels this library has enqueued since it was loaded (every
 * successful launch, all threads and streams; a host-side count). */
uint64_t mnw_moe_launch_count(void);

/* Grouped-GEMM kernel selection, process-wide (a tuning and testing knob;
 * results agree to FP32 rounding order either way).  Three kernels:
 *  - warp-level MMA (operands dequantised straight into registers): INT8/INT4
 *    weights with BF16, FP16-row or INT8 activations;
 *  - tcgen05 row tiles (tokens as M = 128, 256 weight rows as N, both from
 *    shared memory): FP16 rows on INT8/INT4 weights, BF16 on BF16 weights;
 *  - tcgen05 weight tiles (128 weight rows as M, the tokens of one expert as
 *    N): every format and mode.
 * MNW_PATH_AUTO: INT8/INT4 weights with fewer than 32 tokens per expert on
 * average (P / E) take the warp kernel, otherwise the row-tile kernel where it
 * applies and the weight-tile kernel elsewhere.  MNW_PATH_TCGEN05 forces the
 * weight-tile kernel, MNW_PATH_WARP_MMA the warp kernel where it applies,
 * MNW_PATH_ROWS the row-tile kernel where it applies (the weight-tile kernel
 * elsewhere).  Not synchronised with calls in flight on other threads. */
enum mnw_path { MNW_PATH_AUTO = 0, MNW_PATH_TCGEN05 = 1, MNW_PATH_WARP_MMA = 2, MNW_PATH_ROWS = 3 };
int mnw_moe_set_gemm_path(int path);
/* The forward's gate/up step, process-wide: 1 (default) fused -- SiLU(g) * u
 * in the GEMM epilogue; 0 -- the unfused comparison path: gate and up as two
 * single-matrix GEMMs (BF16 g and u in the workspace), then
 * mnw_moe_silu_mul().  Not synchronised with calls in flight on other
 * threads. */
int mnw_moe_set_fused_activation(int fused);

/* The whole layer with no device allocation and no caller workspace (the
 * pages have no counterpart; this is an integration convenience).  For
 * callers that cannot allocate device memory -- e.g. a plugin in a process
 * whose GPU memory is owned up front by another allocator with no hook for
 * plugins, or a latency-critical path that must not pay cudaMalloc's implicit
 * synchronisation.  Same kernels and results as mnw_moe_forward(), with the
 * intermediates in one fixed array of MNW_STATIC_WS_BYTES compiled into the
 * library; every GPU that loads the library holds that array until exit.
 *  - Requests whose mnw_moe_workspace_size() exceeds MNW_STATIC_WS_BYTES
 *    return MNW_E_WORKSPACE_TOO_SMALL before anything is enqueued.
 *  - The first call on each device looks up the array's device address (a
 *    CUDA runtime query, no allocation); make that first call before any
 *    stream capture on that device.
 *  - All calls share the array: calls that overlap on the GPU race and corrupt
 *    each other's results.  Serialise them (one stream).
 *  - err (device, may be NULL) receives this call's device error word
 *    (MNW_DEVERR_*), written on `stream` by every call (0 for T = 0).
 *  - The array's address is cached per device for the life of the process;
 *    do not use the library after cudaDeviceReset().
 * x, ids, w, out are as for mnw_moe_forward(). */
#define MNW_STATIC_WS_BYTES (32u * 1024u * 1024u)
int mnw_moe_forward_static(const mnw_moe_layer* layer, int act, const void* x, const int32_t* ids,
                           const float* w, int T, int k, void* out, uint32_t* err, mnw_stream stream);

/* Self-test of the failure detection every kernel of this library relies on
 * (the pages describe no such call; it exists so that the bounded waits can be
 * tested on a GPU without a fault).  Launches one CTA of two warps on
 * `stream`; each waits on a shared-memory barrier phase that nothing
 * completes.  The first gives up after `limit_us` microseconds (1 .. 10^6),
 * ORs MNW_DEVERR_TIMEOUT into the device word *err and raises the CTA's abort
 * flag; the second waits with the library's own limit (2 s) and must leave
 * through the abort flag instead, in which case 1 is OR-ed into the device
 * word *left_early.  The kernel returns normally and the context stays
 * usable.  Both words are caller-owned device memory, zeroed beforehand.
 * Returns MNW_E_INVALID_ARG for null pointers or a limit out of range. */
int mnw_moe_selftest_wait_timeout(uint32_t limit_us, uint32_t* err, uint32_t* left_early, mnw_stream stream);
/* Self-test of the wait on a token-tile counter that a dependent launch uses
 * (the down launch behind the gate/up launch of a forward): one thread waits
 * up to limit_us (1 us .. 1 s) for *counter (device u32) >= need.  If the
 * counter stays below, it ORs MNW_DEVERR_TIMEOUT into *err (device u32) and
 * returns; no fault, the context stays usable. */
int mnw_moe_selftest_counter_timeout(uint32_t limit_us, const uint32_t* counter, uint32_t need, uint32_t* err,
                                     mnw_stream stream);

/* ---- block attention for prompt prefill (the second workload) ----
 * "coder543/minnow" README, "Quantization": Block FlashAttention serves
 * long-prompt prefill with the attention scores kept on chip.  For every
 * token t of sequence b and query head h (kv head g = h / (Hq / Hkv)):
 *   out[b,t,h,:] = sum_j softmax_j(scale * q[b,t,h,:] . k[b,j,g,:]) v[b,j,g,:]
 * over the allowed keys j: j / blk <= t / blk (block-causal with blocks of
 * blk tokens; blk = 1 is causal, blk >= T bidirectional).  q and out are
 * [B, T, Hq, d] BF16, k and v [B, T, Hkv, d] BF16, all contiguous, 16-byte
 * aligned device memory; d must be 128.  Scores and the softmax are FP32,
 * the probabilities enter the second product as BF16 (FP32 accumulation),
 * out is rounded to BF16.  ws (device, caller-owned, at least
 * mnw_attn_workspace_size bytes, 256-byte aligned) holds a transposed copy
 * of v.  Returns MNW_E_INVALID_ARG (null or misaligned pointers, Hq not a
 * multiple of Hkv, blk < 1, scale not positive and finite),
 * MNW_E_UNSUPPORTED (d != 128), MNW_E_WORKSPACE_TOO_SMALL; B or T = 0 is a
 * no-op.  Device-side timeouts are OR-ed into *err (device u32, nullable). */
size_t mnw_attn_workspace_size(int B, int T, int Hkv, int d);
int mnw_attn_prefill(const void* q, const void* k, const void* v, int B, int T, int Hq, int Hkv, int d, int blk,
                     float scale, void* out, void* ws, size_t ws_bytes, uint32_t* err, mnw_stream stream);

/* Synchronise `stream`, then copy the device error word to *out_host. */
int mnw_moe_read_error(const uint32_t* err, uint32_t* out_host, mnw_stream stream);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif
#ifdef __cplusplus
}
#endif
#endif
