/*
 * CPU oracle for the MXFP4 latent-MoE layer. TEST INFRASTRUCTURE ONLY.
 *
 * This is a plain, slow, fp64 restatement of what the layer computes. Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or constant with the CUDA library, and the
 * CUDA library never calls it.
 *
 * What the layer is (sources are the pages' titles and sections):
 *  - "Kimi K3.1 Pro on AMD Instinct GPUs", section "Kimi K3.1 Pro at a glance":
 *    896 routed experts, 16 active per token, sigmoid routing, expert
 *    intermediate 3,072 inside a 3,584-wide latent, SiTU-GLU activation,
 *    routed experts stored in MXFP4 with one E8M0 scale per 32 values.
 *  - same page, "Serving with ATOM / What we optimized", paragraph "The MXFP4
 *    latent MoE on FlyDSL": a grouped-MoE kernel with MXFP4 weights and an FP8
 *    second stage.
 *  - "Day 0 Kimi-K3 Inference Deployment with ATOM on AMD Instinct MI355X
 *    GPUs", "Model Architecture" table (896 experts, top-16, latent 3584,
 *    intermediate 3072) and "HBM Usage Under TP8" (w1/w2/w3 expert matrices).
 *
 * Readings taken where the pages are silent (each is listed with its reason in
 * the design notes of the repository):
 *  - SiTU-GLU is undefined on the pages; the stand-in is SwiGLU:
 *    h = silu(gate) * up, silu(g) = g * sigmoid(g).
 *  - w1 = gate, w3 = up, w2 = down; w13 is stored [E][2I][d] with the I gate
 *    rows first, then the I up rows.
 *  - The 32-value scale blocks run along the reduction (input) dimension.
 *  - Selection is on the logits (sigmoid is monotone); ties go to the lower
 *    expert id; weights are sigmoid(l_j) / sum of the k selected sigmoids.
 *  - Activations of both stages are MXFP8: E4M3 elements, one E8M0 scale per
 *    32, shared exponent floor(log2(amax)) - 8 (the OCP MX rule with emax of
 *    E4M3 = 8), elements rounded to nearest-even with saturation to +-448,
 *    scale code clamped to [0, 254].
 *  - The stage-1 output h is computed in fp64, rounded to fp32, then quantised.
 *
 * Packing: E2M1 codes two per byte, the even element in the low nibble.
 * Scales are canonical row-major [rows][K/32] bytes. bf16 values travel as
 * their 16-bit patterns.
 *
 * Pins: tests/test_oracle_*.py check every function here against facts that do
 * not come from this file (OCP value lists, torch's float8 casts, brute-force
 * sorts, a dense numpy restatement of the layer, closed forms, invariants).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element decodes by table built from the format definitions (OCP MX v1.0). */
double orc_e2m1_value(uint8_t code);   /* low nibble used */
double orc_e4m3_value(uint8_t code);   /* 0x7F and 0xFF are NaN */
double orc_e8m0_value(uint8_t code);   /* 2^(code-127); 0xFF is NaN */

/* Round-to-nearest-even of a real number to E4M3 with saturation to +-448.
 * The sign is kept for zero results. Input must not be NaN. */
uint8_t orc_e4m3_encode_rne_sat(double v);

/* The scalar MX rule on one block of 32 fp32 values -> 32 E4M3 codes and one
 * E8M0 scale code. */
void orc_mx_quant_block(const float* v32, uint8_t* codes32, uint8_t* scale);

/* MX rule over a row-major [rows][K] fp32 matrix (K % 32 == 0).
 * codes [rows][K], scales [rows][K/32]. */
void orc_mx_quant_rows(const float* v, int64_t rows, int64_t K,
                       uint8_t* codes, uint8_t* scales);

/* Same, on bf16 bit patterns [rows][K]. */
void orc_mx_quant_rows_bf16(const uint16_t* x, int64_t rows, int64_t K,
                            uint8_t* codes, uint8_t* scales);

/* Sigmoid top-k routing of T rows of E logits.
 * ids [T][k] in order (logit descending, id ascending); w [T][k] fp32. */
void orc_route_topk(const float* logits, int64_t T, int32_t E, int32_t k,
                    int32_t* ids, float* w);

/* Grouping of the T*k slots by expert.
 * counts [E]; offsets [E+1], offsets[e+1] = offsets[e] + ceil(counts[e]/pad_m)*pad_m;
 * slot_to_row [T*k]: rows of one expert ordered by ascending token;
 * row_to_slot [rows_capacity]: slot of each row, -1 on padding rows, untouched
 * past offsets[E]. Returns 0, or -1 when an id is out of range, an id repeats
 * within a token, or offsets[E] > rows_capacity. */
int32_t orc_permute(const int32_t* ids, int64_t T, int32_t E, int32_t k, int32_t pad_m,
                    int32_t* counts, int32_t* offsets, int32_t* slot_to_row,
                    int32_t* row_to_slot, int64_t rows_capacity);

/* Stage 1 of one expert on one activation row, in fp64:
 * g = Xd * W1d^T, u = Xd * W3d^T, h = silu(g) * u.
 * xq [d] E4M3 codes, xs [d/32]; w13_e [2I][d/2] packed E2M1, w13s_e [2I][d/32].
 * h [I] fp64 (before the fp32 rounding and requantisation). */
void orc_expert_stage1(const uint8_t* xq, const uint8_t* xs, int32_t d, int32_t I,
                       const uint8_t* w13_e, const uint8_t* w13s_e, double* h);

/* Stage 2 of one expert on one row: y = Hd * W2d^T in fp64.
 * hq [I] E4M3 codes, hs [I/32]; w2_e [d][I/2] packed E2M1, w2s_e [d][I/32]. */
void orc_expert_stage2(const uint8_t* hq, const uint8_t* hs, int32_t I, int32_t d,
                       const uint8_t* w2_e, const uint8_t* w2s_e, double* y);

/* ---- A4W4 stage 1 (MXFP4 activations) -------------------------------------
 * The pages' stage-1 kernel is selected by an environment switch named A4W4
 * ("Appendix: environment variables" of "Kimi K3.1 Pro on AMD Instinct GPUs",
 * next to the FP8 second-stage switch): 4-bit activations and 4-bit weights.
 * Reading: the stage-1 activations are MXFP4 (E2M1 elements, one E8M0 scale
 * per 32, shared exponent floor(log2(amax)) - 2, the OCP MX rule with emax of
 * E2M1 = 2), elements rounded to nearest-even with saturation to +-6; stage 2
 * stays MXFP8. */

/* Round-to-nearest-even of a real number to E2M1 with saturation to +-6. The
 * sign is kept for zero results (code 0x8 for -0). Input must not be NaN. */
uint8_t orc_e2m1_encode_rne_sat(double v);

/* The MX rule for MXFP4 on one block of 32 fp32 values -> 16 bytes of packed
 * E2M1 codes (even element in the low nibble) and one E8M0 scale code. */
void orc_mxfp4_quant_block(const float* v32, uint8_t* packed16, uint8_t* scale);

/* MXFP4 over a row-major [rows][K] matrix of fp32 values or of bf16 bit
 * patterns: packed codes [rows][K/2], scales [rows][K/32]. */
void orc_mxfp4_quant_rows(const float* v, int64_t rows, int64_t K,
                          uint8_t* packed, uint8_t* scales);
void orc_mxfp4_quant_rows_bf16(const uint16_t* x, int64_t rows, int64_t K,
                               uint8_t* packed, uint8_t* scales);

/* Stage 1 of one expert on one MXFP4 activation row, in fp64: as
 * orc_expert_stage1 with xq [d/2] packed E2M1 codes and xs [d/32]. */
void orc_expert_stage1_a4(const uint8_t* xq, const uint8_t* xs, int32_t d, int32_t I,
                          const uint8_t* w13_e, const uint8_t* w13s_e, double* h);

/* The whole layer with MXFP4 stage-1 activations (same arguments and
 * outputs as orc_moe_forward). */
void orc_moe_forward_a4w4(const uint16_t* x, const float* logits, int64_t n,
                          int32_t d, int32_t E, int32_t k, int32_t I,
                          const uint8_t* w13, const uint8_t* w13s,
                          const uint8_t* w2, const uint8_t* w2s,
                          uint16_t* y, int32_t* ids, float* w, double* y64,
                          int32_t threads);

/* ---- Neighbouring BF16 steps ------------------------------------------------
 * The pages run the router GEMM producing the logits, the latent down/up
 * projections (7,168 <-> 3,584) and two shared experts in BF16 next to the
 * routed experts ("Kimi K3.1 Pro at a glance" and "The MXFP4 latent MoE on
 * FlyDSL" of "Kimi K3.1 Pro on AMD Instinct GPUs"; "HBM Usage Under TP8" of
 * "Day 0 Kimi-K3 Inference Deployment with ATOM on AMD Instinct MI355X
 * GPUs"). Each is a dense product of bf16 operands. */

/* C[M][N] = A[M][K] . B[N][K]^T in fp64 from bf16 bit patterns. */
void orc_gemm_bf16(const uint16_t* a, const uint16_t* b, int64_t M, int64_t N, int64_t K,
                   double* c);

/* The gated MLP step of a shared expert: B holds 2*Nh rows, gate rows first
 * then up rows; h[M][Nh] = silu(g) * u with g = A . Bgate^T, u = A . Bup^T,
 * all in fp64. */
void orc_gemm_bf16_swiglu(const uint16_t* a, const uint16_t* b, int64_t M, int64_t Nh,
                          int64_t K, double* h);

/* Round a real number to the nearest bf16 (ties to even), returning its bits. */
uint16_t orc_bf16_rne(double v);

/* orc_bf16_rne over n values (a block's bf16 intermediates and output). */
void orc_bf16_rne_n(const double* v, int64_t n, uint16_t* out);

/* The whole layer for n independent tokens.
 * x [n][d] bf16 bits, logits [n][E] fp32, weights for all E experts:
 * w13 [E][2I][d/2], w13s [E][2I][d/32], w2 [E][d][I/2], w2s [E][d][I/32].
 * Outputs: y [n][d] bf16 bits; optional ids [n][k], w [n][k]; optional
 * y64 [n][d] (the fp64 sum before the bf16 rounding).
 * threads <= 0 means one per hardware thread. */
void orc_moe_forward(const uint16_t* x, const float* logits, int64_t n,
                     int32_t d, int32_t E, int32_t k, int32_t I,
                     const uint8_t* w13, const uint8_t* w13s,
                     const uint8_t* w2, const uint8_t* w2s,
                     uint16_t* y, int32_t* ids, float* w, double* y64,
                     int32_t threads);

/* Bytes of one expert in MXFP4 (three matrices of I x d, packed values and
 * scales): 3 * d * I * (1/2 + 1/32). */
int64_t orc_expert_bytes(int32_t d, int32_t I);

#ifdef __cplusplus
}
#endif

#endif
