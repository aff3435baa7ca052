/*
 * moe_oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU restatement of the routed-expert MoE
 * layer, written from the format and mode descriptions of:
 *   [minnow]  "coder543/minnow" README, sections "Quantization" and
 *             "Development and performance";
 *   [card]    "LLaDA2.2-flash-minnow" model card, section "Checkpoints and
 *             precision" (its precision table and the paragraphs after it).
 * Accumulation is FP64; the dynamic activation quantisers use IEEE binary32
 * operations with round-to-nearest-even because their scales are FP32
 * ([card] W8A8 paragraph; NVFP4 row of the precision table).
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library.  It shares no code with the CUDA path.
 *
 * Parity status: every function here is pinned by a "not gpu" test
 * (tests/test_oracle_*.py) except where its comment says "parity unpinned".
 */
#ifndef MNW_MOE_ORACLE_H
#define MNW_MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight formats of the expert blob ([card] precision table). */
enum { MNWO_FMT_BF16 = 0, MNWO_FMT_INT8_G128 = 1, MNWO_FMT_INT4_G128 = 2, MNWO_FMT_NVFP4_G16 = 3 };
/* Activation modes: BF16 (A16), dynamic INT8 per 128 (A8), dynamic NVFP4 (A4),
 * and FP16 rows with a power-of-two row factor (an exact re-encoding of BF16
 * rows for FP16 tensor cores; not a mode of the pages, see mnwo_encode_f16_rows). */
enum { MNWO_ACT_BF16 = 0, MNWO_ACT_INT8_G128 = 1, MNWO_ACT_NVFP4_G16 = 2, MNWO_ACT_F16_ROWS = 3 };
/* Grouped GEMM kinds: the fused gate/up/SiLU, down, and the gate or up
 * matrix alone (the unfused-activation comparison path of [minnow]
 * "Quantization": the activation then runs as its own step, mnwo_silu_mul). */
enum { MNWO_KIND_GATE_UP = 0, MNWO_KIND_DOWN = 1, MNWO_KIND_GATE = 2, MNWO_KIND_UP = 3 };
/* Matrices of one expert. */
enum { MNWO_GATE = 0, MNWO_UP = 1, MNWO_DOWN = 2 };

/* Return codes. */
enum { MNWO_OK = 0, MNWO_E_ARG = 1, MNWO_E_BLOB = 2, MNWO_E_NONFINITE = 3, MNWO_E_MODE = 4 };

/* ---- scalar decoders (closed forms of each format) ---- */
double mnwo_bf16_to_double(uint16_t bits);
int    mnwo_fp16_to_double(uint16_t bits, double* out);      /* rejects Inf/NaN */
int    mnwo_int4_value(uint8_t nibble);                      /* two's complement, [-8, 7] */
int    mnwo_int8_value(uint8_t byte);                        /* two's complement */
double mnwo_e2m1_to_double(uint8_t nibble);                  /* s|e1e0|m */
int    mnwo_e4m3_to_double(uint8_t byte, double* out);       /* OCP E4M3FN; rejects NaN */

/* ---- scalar encoders: round to nearest, ties to even ---- */
uint16_t mnwo_bf16_from_double(double v);                    /* overflow -> Inf */
uint16_t mnwo_fp16_from_double(double v);                    /* overflow -> Inf */
uint8_t  mnwo_e4m3_rn_satfinite(float v);                    /* saturates at +-448 */
uint8_t  mnwo_e2m1_rn_satfinite(float v);                    /* saturates at +-6   */

/* ---- dynamic activation quantisers (rows of K values, BF16 in) ---- */
/* INT8, one FP32 scale per 128 consecutive values of a row ([card] W8A8). */
int mnwo_quant_int8_g128(const uint16_t* x, int R, int K, int8_t* codes, float* scales);
/* NVFP4: E2M1 codes (two per byte, low nibble = even index), E4M3 scale per 16,
 * FP32 outer scale per row ([card] NVFP4 row, activation column). */
int mnwo_quant_nvfp4_g16(const uint16_t* x, int R, int K, uint8_t* codes, uint8_t* sf, float* outer);

/* FP16 rows: e = clamp(floor(log2 amax_row) - 14, -110, 113) (e = -110 for an
 * all-zero row), factor = 2^e, code = fp16_rn(x * 2^-e).  The row's largest
 * magnitude lands in [2^14, 2^15) (unless clamped); every value at most 2^28
 * below it is kept exactly (BF16's 8 significant bits fit FP16's 11).
 * MNWO_E_NONFINITE for a row holding Inf or NaN. */
int mnwo_encode_f16_rows(const uint16_t* x, int R, int K, uint16_t* codes, float* factor);

/* ---- router (the step before the permutation on the GPU routing path) ----
 * [minnow] "Quantization": GPU routing for 32-token decode blocks; [card]:
 * routers keep their source floating-point (BF16) weights.  Reading of the
 * pages (they give no formula): logits[t, e] = sum_h x[t, h] * wr[e, h]
 * (FP64 here); ids[t, 0..k) = the k largest logits of row t, largest first,
 * the lower expert index first among equal logits; w[t, j] = softmax of the k
 * chosen logits, exp(l_j - l_max) / sum_i exp(l_i - l_max) in FP64, stored
 * as float.  x: [T, H] BF16 bits; wr: [E, H] BF16 bits; logits (nullable):
 * [T, E] FP64.  Returns MNWO_E_ARG for k outside [1, E]. */
int mnwo_route(const uint16_t* x, const uint16_t* wr, int T, int H, int E, int k, int32_t* ids, float* w,
               double* logits);

/* ---- token permutation into expert-sorted order ---- */
/* Returns the number of dropped (out-of-range) ids, or -1 on bad arguments. */
int mnwo_permute(const int32_t* ids, int T, int k, int E,
                 int32_t* expert_offsets, int32_t* sorted_assign, int32_t* assign_pos);

/* ---- expert-weight blob ---- */
typedef struct {
  uint32_t wfmt, E, H, I, group;
  uint64_t expert_stride, data_offset, total_bytes;
  uint64_t codes_off[3], scales_off[3], outer_off[3];
} mnwo_blob_info;

int mnwo_blob_parse(const uint8_t* blob, size_t bytes, mnwo_blob_info* info);
/* Decoded value of weight (n, k) of matrix m (gate/up [I,H], down [H,I]) of expert e. */
int mnwo_weight(const uint8_t* blob, const mnwo_blob_info* info, int e, int m, int n, int k, double* out);

/* ---- grouped GEMM references, one per ABI call ----
 * Rows [offsets[e], offsets[e+1]) of `a` belong to expert e.
 * kind GATE_UP: out[p, n] = bf16(SiLU(g) * u), out is [P, I].
 * kind DOWN:    out[p, n] = bf16(a_p . Wd[n]), out is [P, H]. */
int mnwo_gemm_a16(const uint8_t* blob, size_t bytes, int kind, const uint16_t* a,
                  const int32_t* offsets, int P, uint16_t* out);
/* A8: INT32 group dot products, scaled and summed in FP64.  `dots` (nullable)
 * receives every group dot product, layout [P][Ncols][K/128] with
 * Ncols = 2I (gate columns then up columns) or H. */
int mnwo_gemm_a8(const uint8_t* blob, size_t bytes, int kind, const int8_t* a_codes,
                 const float* a_scales, const int32_t* offsets, int P, uint16_t* out, int32_t* dots);
int mnwo_gemm_a4(const uint8_t* blob, size_t bytes, int kind, const uint8_t* a_codes,
                 const uint8_t* a_sf, const float* a_outer, const int32_t* offsets, int P,
                 uint16_t* out);
/* FP16 rows (INT8/INT4 weights): dot = factor[p] * sum_k fp16(a[p,k]) * w[n,k],
 * the weights decoded exactly as in mnwo_gemm_a16. */
int mnwo_gemm_f16rows(const uint8_t* blob, size_t bytes, int kind, const uint16_t* a,
                      const float* factor, const int32_t* offsets, int P, uint16_t* out);

/* ---- the unfused activation: out = bf16(SiLU(g) * u), FP64 from BF16 g, u ---- */
void mnwo_silu_mul(const uint16_t* g, const uint16_t* u, size_t n, uint16_t* out);

/* ---- combine ---- */
void mnwo_combine(const uint16_t* y, const int32_t* assign_pos, const float* w, int T, int k,
                  int H, uint16_t* out);

/* ---- whole layer, token by token (no permutation needed) ----
 * `rows` (nullable) selects which tokens to compute; out is [nrows, H]. */
int mnwo_moe_forward(const uint8_t* blob, size_t bytes, int act, const uint16_t* x,
                     const int32_t* ids, const float* w, int T, int k,
                     const int32_t* rows, int nrows, uint16_t* out);

/* ---- block attention for prefill (the second workload) ----
 * [minnow] "Quantization" (Block FlashAttention keeps the prompt's attention
 * scores on chip; what it computes is plain attention): for each selected
 * token t of sequence b and query head h, with kv head g = h / (Hq / Hkv),
 * out = softmax_j(scale * q . k_j) weighted sum of v_j over the allowed keys
 * j: j < T and j / blk <= t / blk (block-causal; blk = 1 causal, blk >= T
 * bidirectional).  FP64 from BF16 q [B,T,Hq,d], k and v [B,T,Hkv,d]; rows
 * (nullable) lists flat token indices b*T + t; out is [nrows, Hq, d] FP64. */
int mnwo_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int T, int Hq, int Hkv,
                   int d, int blk, double scale, const int32_t* rows, int nrows, double* out);

#ifdef __cplusplus
}
#endif
#endif
