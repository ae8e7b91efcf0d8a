/*
 * moe.h -- C-ABI of libmoe.so, the GB300 (sm_103a) MXFP4 latent-MoE layer.
 *
 * The layer (sources are page titles and sections):
 *   "Kimi K3.1 Pro on AMD Instinct GPUs", "Kimi K3.1 Pro at a glance":
 *     896 routed experts, 16 active per token, sigmoid routing, expert
 *     intermediate 3,072 in a 3,584-wide latent, SiTU-GLU activation,
 *     routed experts in MXFP4 with one E8M0 scale per 32 values.
 *   same page, "Serving with ATOM / What we optimized", "The MXFP4 latent MoE
 *     on FlyDSL": a grouped-MoE kernel, MXFP4 weights, FP8 second stage.
 *   "Day 0 Kimi-K3 Inference Deployment with ATOM on AMD Instinct MI355X
 *     GPUs", "Model Architecture" table and "HBM Usage Under TP8" (w1/w2/w3).
 *
 * Readings where the pages are silent: SwiGLU stands in for the undefined
 * SiTU-GLU (h = silu(gate) * up); w1 = gate, w3 = up, w2 = down; scale blocks
 * of 32 run along the reduction dimension; activations of both stages are
 * MXFP8 (E4M3 + one E8M0 per 32, OCP MX rule, round-to-nearest-even with
 * saturation to +-448); selection on the logits with ties to the lower id,
 * weights = sigmoid(l_j) / sum of the k selected sigmoids.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller, unless stated. The
 *    library never allocates or frees device memory and never synchronises,
 *    except moe_check_device_status.
 *  - Work is enqueued on `stream` in order; the host returns without waiting.
 *    Most kernels use programmatic dependent launch: one may start while the
 *    previous kernel of this library in the stream is still running (after
 *    any other kernel it starts only once that one has finished), and it
 *    waits for its predecessor (griddepcontrol.wait) before touching memory
 *    that kernel or the caller may use, so stream order holds as usual.
 *  - Arguments are validated on the host before any launch. A failed check
 *    returns a non-zero moe_status and enqueues nothing.
 *  - Launch failures return MOE_ERR_CUDA. Problems found on the device (a
 *    bounded wait that ran out, an expert id out of range) are recorded in the
 *    4-byte status word at the start of the workspace `ws`; read it with
 *    moe_check_device_status. The GPU never traps.
 *  - bf16 tensors are passed as uint16_t bit patterns.
 *  - All work runs on the CUDA device current in the calling thread.
 *  - Thread-safe as long as concurrent calls use distinct workspaces.
 *
 * Shapes (checked; anything else is MOE_ERR_UNSUPPORTED):
 *   1 <= E <= 1024, 0 <= k <= min(E, 32), T >= 0, T*k < 2^31,
 *   d % 128 == 0 and I % 128 == 0 (both >= 128),
 *   moe_permute takes any power of two 1..1024 as pad_m.
 *
 * Two kernel families run the grouped GEMMs (moe_gemm_kernel):
 *   MOE_GEMM_TOKEN_TILES   tokens are the MMA's M side (128-row tiles),
 *                          weights the N side; for many tokens per expert.
 *                          An expert with an even number of tiles, or with
 *                          at least 8 (more than 896 tokens), runs its full
 *                          pairs of tiles as one 256-row MMA over a pair of
 *                          SMs, in a launch before the one for the other
 *                          tiles; the results are those of one tile at a
 *                          time. Groups padded
 *                          to 128 rows; activation scales in the TILED
 *                          layout.
 *   MOE_GEMM_WEIGHT_TILES  weights are the M side (128 weight rows per MMA),
 *                          an expert's tokens the N side in chunks of 32, or
 *                          of 64 when rows_capacity exceeds 55 rows per
 *                          expert (more than ~24 routed rows per expert); for
 *                          a few tokens per expert (decode), where streaming
 *                          the weights from HBM is the bound. Groups padded to
 *                          32 rows; activation scales in the GROUP32 layout.
 *   MOE_GEMM_PAIR_TILES    weights are the M side of an MMA spread over a pair
 *                          of SMs (2-CTA clusters, 256 weight rows per MMA),
 *                          an expert's tokens the N side in chunks of 128
 *                          (stage 1) or 256 (stage 2), the last chunk as wide
 *                          as its tokens rounded up to 16; for many tokens per
 *                          expert (prefill). Groups padded to 128 rows;
 *                          activation scales TILED (as token tiles). Needs
 *                          d % 256 == 0 and I % 256 == 0.
 *
 * Data layouts:
 *   x, y        bf16 [T][d] row-major.
 *   logits      fp32 [T][E].
 *   topk_ids    int32 [T][k], topk_w fp32 [T][k]; slot s = t*k + j.
 *   Weights     canonical: w13 u8 [E][2I][d/2]: rows 0..I-1 gate (w1),
 *               I..2I-1 up (w3); w2 u8 [E][d][I/2]; two E2M1 codes per byte,
 *               even element in the low nibble; scales u8 [rows][K/32] (one
 *               E8M0 code per 32 consecutive inputs). The GEMMs take the codes
 *               in the BOXED layout (moe_prepack_weights) and the scales in the
 *               TILED layout (moe_prepack_scales), both made once at load.
 *   BOXED code layout of a matrix of R rows x K inputs (R, K multiples of
 *   128): contiguous 8 KB boxes of 128 rows x 128 inputs (64 bytes per row),
 *   box (r/128, c/128) at index (r/128)*(K/128) + c/128; the byte of element
 *   (r, c) is box*8192 + (r%128)*64 + (c%128)/2. Every tensor-memory-access
 *   load of a weight box is then one contiguous 8 KB read.
 *   Activations xq u8 [rows][d] and hq u8 [rows][I] E4M3 codes; their scales
 *               in the TILED layout.
 *   TILED scale layout of an operand with R rows and K inputs per row (R
 *   rounded up to 128, K % 128 == 0): the scale of row r, 32-block b is byte
 *     ((r/128)*(K/128) + b/4)*512 + (r%32)*16 + ((r/32)%4)*4 + b%4,
 *   i.e. one 512-byte atom per 128 rows x 128 inputs, in the order the
 *   tensor-core scale-factor copy reads it.
 *   GROUP32 scale layout (activations of the weight-tile GEMMs): one 512-byte
 *   block per 32 rows x 128 inputs; the scale of row r, 32-block b is byte
 *     ((r/32)*(K/128) + b/4)*512 + (r%32)*16 + b%4,
 *   the other 12 bytes of each 16 unused (rows * K / 8 bytes in all).
 *   Grouped rows: rows [offsets[e], offsets[e+1]) belong to expert e, the
 *   first counts[e] of them hold its tokens in ascending token order, the rest
 *   are padding (row_to_slot == -1, contents unspecified, never read back).
 */
#ifndef MXFP4_LATENT_MOE_H
#define MXFP4_LATENT_MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARGUMENT = 1,    /* null pointer, negative size, bad alignment */
  MOE_ERR_UNSUPPORTED = 2,         /* shape outside the supported set */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes or rows_capacity below what the call needs */
  MOE_ERR_CUDA = 4,                /* a CUDA runtime/driver call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 5,      /* device status: a bounded wait ran out */
  MOE_ERR_DEVICE_BAD_INPUT = 6     /* device status: expert id out of range or repeated */
} moe_status;

typedef enum {
  MOE_SCALES_TILED128 = 0,   /* activation scales for the token-tile GEMMs */
  MOE_SCALES_GROUP32 = 1     /* activation scales for the weight-tile GEMMs */
} moe_scale_layout;

typedef enum {
  MOE_GEMM_AUTO = 0,         /* moe_forward only: see moe_default_kernel */
  MOE_GEMM_TOKEN_TILES = 1,  /* tokens on the MMA's M side */
  MOE_GEMM_WEIGHT_TILES = 2, /* weights on the MMA's M side, tokens as N */
  MOE_GEMM_PAIR_TILES = 3    /* weights on M across a pair of SMs, tokens as N */
} moe_gemm_kernel;

typedef struct {
  int32_t T; /* tokens */
  int32_t d; /* latent width (3584) */
  int32_t E; /* routed experts (896) */
  int32_t k; /* experts per token (16) */
  int32_t I; /* expert intermediate width (3072) */
} moe_dims;

typedef struct {
  const uint8_t* w13;    /* BOXED codes of w13 viewed as [E*2I][d] (moe_prepack_weights) */
  const uint8_t* w13_sf; /* TILED scales of w13 viewed as [E*2I][d] (moe_prepack_scales) */
  const uint8_t* w2;     /* BOXED codes of w2 viewed as [E*d][I] */
  const uint8_t* w2_sf;  /* TILED scales of w2 viewed as [E*d][I] */
} moe_weights;

/* Bytes of the device status word region at the start of every workspace. */
#define MOE_STATUS_BYTES 256

/* Short English text of a status code. Never NULL; static storage. */
const char* moe_status_string(moe_status s);

/* Version of this ABI (incremented on incompatible change). */
int32_t moe_abi_version(void);

/* Bytes of a TILED scale array for `rows` rows of K inputs (rows rounded up
 * to a multiple of 128). Returns 0 for unsupported K. */
size_t moe_tiled_scale_bytes(int64_t rows, int32_t K);

/* The GEMM kernels moe_forward uses for MOE_GEMM_AUTO: MOE_GEMM_WEIGHT_TILES
 * while the experts average at most 56 routed rows (T*k <= 56*E), else
 * MOE_GEMM_TOKEN_TILES. On GB300 at the full layer dims the weight tiles
 * stream the weights at 80-94% of HBM bandwidth up to T = 3072 tokens (32-
 * then 64-token chunks), while the token tiles are bound by their 128-row
 * tensor work there and win from T = 3584. Returns -1 for an unsupported
 * shape. */
int32_t moe_default_kernel(int32_t T, int32_t E, int32_t k);

/* Bytes of an activation scale array for `rows` rows of K inputs in the given
 * moe_scale_layout (rows rounded up to 128 or 32). 0 for unsupported K or
 * layout. */
size_t moe_activation_scale_bytes(int64_t rows, int32_t K, int32_t scale_layout);

/* Rows a grouped activation buffer needs for T tokens, k experts each, E
 * experts and padding pad_m: T*k + min(E, T*k)*(pad_m-1), rounded up to 128. */
int64_t moe_rows_capacity(int32_t T, int32_t E, int32_t k, int32_t pad_m);

/* Canonical scales [rows][K/32] -> TILED layout (moe_tiled_scale_bytes bytes).
 * One-time weight preparation; the bytes are permuted, not changed. Rows past
 * `rows` in the last 128-row atom are written as 0. src and dst must not
 * overlap; dst 16-byte aligned. */
moe_status moe_prepack_scales(const uint8_t* src, int64_t rows, int32_t K, uint8_t* dst,
                              cudaStream_t stream);

/* Canonical packed E2M1 codes [rows][K/2] -> BOXED layout (rows*K/2 bytes).
 * One-time weight preparation; bytes are moved, not changed. rows % 128 == 0;
 * src 16-byte and dst 32-byte aligned; no overlap. */
moe_status moe_prepack_weights(const uint8_t* src, int64_t rows, int32_t K, uint8_t* dst,
                               cudaStream_t stream);

/* Sigmoid top-k routing ("Kimi K3.1 Pro at a glance", Experts row: "896
 * routed (top-16, sigmoid routing)").
 * For each token t: the k largest logits[t][:], ordered by logit descending
 * and expert id ascending on ties (IEEE compare, -0 == +0);
 * topk_w[t][j] = sigmoid(l_j) / sum_j' sigmoid(l_j') in fp32.
 * logits fp32 [T][E] (finite); outputs int32 [T][k] and fp32 [T][k]. */
moe_status moe_route_topk(const float* logits, int32_t T, int32_t E, int32_t k,
                          int32_t* topk_ids, float* topk_w, cudaStream_t stream);

/* Workspace bytes moe_permute needs (status word + per-chunk histograms). */
size_t moe_permute_workspace_size(int32_t T, int32_t E);

/* Expert grouping for the grouped-MoE kernel ("The MXFP4 latent MoE on
 * FlyDSL"): histogram, exclusive scan of padded counts, stable scatter.
 * counts [E]; offsets [E+1] with offsets[e+1] = offsets[e] +
 * ceil(counts[e]/pad_m)*pad_m; slot_to_row [T*k]; row_to_slot [rows_capacity]
 * (slot of each grouped row; -1 on every row of [0, rows_capacity) that holds
 * no slot, padding rows included).
 * Within an expert, rows follow ascending token order: the result is unique
 * and does not depend on scheduling. rows_capacity must be at least
 * moe_rows_capacity(T, E, k, pad_m) (checked on the host). An id out of range
 * or repeated within a token sets MOE_ERR_DEVICE_BAD_INPUT in the status word
 * and leaves the outputs unspecified. */
moe_status moe_permute(const int32_t* topk_ids, int32_t T, int32_t E, int32_t k, int32_t pad_m,
                       int32_t* counts, int32_t* offsets, int32_t* slot_to_row,
                       int32_t* row_to_slot, int64_t rows_capacity, void* ws, size_t ws_bytes,
                       cudaStream_t stream);

/* Allocation-free variant of moe_permute. The pages have no counterpart: it
 * exists for callers that cannot hand the library device memory for a
 * workspace -- a host framework that owns every device allocation through its
 * own pool and forbids libraries to allocate, or a latency-critical caller that
 * must not call cudaMalloc on its serving path (it may synchronise the whole
 * device). Same arguments, results and rules as moe_permute, without ws:
 *  - The per-chunk histograms live in a fixed 1 MiB device array inside
 *    libmoe.so, held by every GPU that loads the library until the process
 *    exits. Calls need ceil(T/256) * E * 4 <= 1 MiB (T <= 74,752 at E = 896);
 *    larger calls return MOE_ERR_WORKSPACE_TOO_SMALL and enqueue nothing.
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress) and caches it; make that
 *    first call before any stream capture. Nothing here calls cudaMalloc,
 *    cudaFree or any other allocating routine.
 *  - All calls share the array and it keeps the previous call's contents;
 *    every byte a call reads it has written first, so no clearing is needed.
 *    Calls that overlap on the GPU (other streams, other host threads) race
 *    on it: serialise them.
 *  - status: optional device int32 (NULL = none) that receives
 *    MOE_ERR_DEVICE_BAD_INPUT for an id out of range or repeated within a
 *    token (first error wins; the caller clears it). */
moe_status moe_permute_noalloc(const int32_t* topk_ids, int32_t T, int32_t E, int32_t k,
                               int32_t pad_m, int32_t* counts, int32_t* offsets,
                               int32_t* slot_to_row, int32_t* row_to_slot, int64_t rows_capacity,
                               int32_t* status, cudaStream_t stream);

/* MXFP8 quantisation of the stage-1 activations (OCP MX rule, E4M3 + E8M0
 * per 32 consecutive values of a row): per block, scale code
 * c = clamp(floor(log2(amax)) - 8 + 127, 0, 254) (0 for an all-zero block),
 * element codes = E4M3 round-to-nearest-even of x * 2^(127-c) saturated to
 * +-448, the sign kept on zero results.
 * x bf16 [T][d]. With slot_to_row == NULL the output rows are the tokens
 * (row t); otherwise token t is written to every row slot_to_row[t*k + j],
 * j < k. codes u8 [rows_capacity][d]; scales in scale_layout (moe_scale_layout:
 * TILED for the token-tile GEMMs, GROUP32 for the weight-tile GEMMs) for
 * (rows_capacity, d). rows_capacity % 128 == 0. */
moe_status moe_quant_mxfp8(const uint16_t* x, int32_t T, int32_t d, const int32_t* slot_to_row,
                           int32_t k, uint8_t* codes, uint8_t* scales, int32_t scale_layout,
                           int64_t rows_capacity, cudaStream_t stream);

/* Stage 1 grouped GEMM on tcgen05 block-scaled tensor cores
 * (kind::mxf8f6f4, MXFP8 activations x MXFP4 weights, fp32 accumulation)
 * with the GLU and the FP8 second-stage quantisation fused in the epilogue
 * ("The MXFP4 latent MoE on FlyDSL"; expert shapes from the Experts row).
 * For each expert e and each of its grouped rows r:
 *   g = X[r] . W1[e]^T, u = X[r] . W3[e]^T  (dequantised operands, fp32 sums)
 *   h = silu(g) * u (fp32), then MXFP8 as in moe_quant_mxfp8
 *   -> hq [r][I] codes and hs scales for (rows_capacity, I).
 * kernel: MOE_GEMM_TOKEN_TILES (xs and hs TILED, groups padded to 128) or
 * MOE_GEMM_WEIGHT_TILES (xs and hs GROUP32, groups padded to 32).
 * counts int32 [E] and offsets int32 [E+1] are read on the device and must
 * come from moe_permute with that padding: every group a multiple of it
 * holding counts[e] tokens, offsets[0] == 0, offsets[E] <= rows_capacity.
 * Offsets or counts that break this are refused on the device
 * (MOE_ERR_DEVICE_BAD_INPUT in the status word, nothing written).
 * Only rows that hold tokens are written: padding rows of a group (and their
 * scales) are left untouched.
 * ws: at least MOE_STATUS_BYTES; the status word records timeouts.
 * w13: BOXED codes (moe_prepack_weights of the [E*2I][d] matrix), w13_sf:
 * TILED scales (moe_prepack_scales). xq, hq 16-byte aligned; w13 32-byte
 * aligned; scale arrays 16-byte aligned. */
moe_status moe_grouped_gemm_w13_glu(const uint8_t* xq, const uint8_t* xs, const int32_t* counts,
                                    const int32_t* offsets, int32_t E, int32_t d, int32_t I,
                                    int32_t kernel, const uint8_t* w13, const uint8_t* w13_sf,
                                    uint8_t* hq, uint8_t* hs, int64_t rows_capacity, void* ws,
                                    size_t ws_bytes, cudaStream_t stream);

/* Stage 2 grouped GEMM (the down projection w2, 3,072 -> 3,584 in the pages'
 * layer): Yp[r] = H[r] . W2[e]^T with MXFP8 H and MXFP4 W2 on tcgen05
 * block-scaled tensor cores, fp32 accumulation, rounded to bf16.
 * yp bf16 [rows_capacity][d], 16-byte aligned; w2 BOXED codes of the
 * [E*d][I] matrix and w2_sf its TILED scales; hq, hs, counts, offsets and
 * kernel as produced for / by the stage-1 call. Padding rows of yp are left
 * untouched. */
moe_status moe_grouped_gemm_w2(const uint8_t* hq, const uint8_t* hs, const int32_t* counts,
                               const int32_t* offsets, int32_t E, int32_t I, int32_t d,
                               int32_t kernel, const uint8_t* w2, const uint8_t* w2_sf,
                               uint16_t* yp, int64_t rows_capacity, void* ws, size_t ws_bytes,
                               cudaStream_t stream);

/* Routing-weighted combine: y[t] = bf16_rne(sum_{j=0..k-1} topk_w[t][j] *
 * Yp[slot_to_row[t*k+j]]) with fp32 accumulation in j order. k == 0 gives
 * y = 0. yp, y 16-byte aligned. */
moe_status moe_unpermute_combine(const uint16_t* yp, const int32_t* slot_to_row,
                                 const float* topk_w, int32_t T, int32_t k, int32_t d,
                                 uint16_t* y, cudaStream_t stream);

/* Workspace bytes moe_forward and moe_forward_a4w4 need for these dims. */
moe_status moe_workspace_size(const moe_dims* dims, size_t* bytes);

/* The whole layer: route -> permute -> quantise -> stage-1 GEMM + GLU +
 * requant -> stage-2 GEMM -> combine, all on `stream` with no host
 * synchronisation. Clears the status word at its start. kernel selects the
 * grouped-GEMM family (moe_gemm_kernel; MOE_GEMM_AUTO = moe_default_kernel).
 * x bf16 [T][d], logits fp32 [T][E], weights as in moe_weights, y bf16 [T][d].
 * topk_ids_out / topk_w_out may be NULL; if given they receive the routing.
 * ws: moe_workspace_size bytes, 256-byte aligned. */
moe_status moe_forward(const moe_dims* dims, int32_t kernel, const uint16_t* x,
                       const float* logits, const moe_weights* weights, uint16_t* y,
                       int32_t* topk_ids_out, float* topk_w_out, void* ws, size_t ws_bytes,
                       cudaStream_t stream);

/* ---- A4W4 stage 1 ---------------------------------------------------------
 * The pages select their stage-1 MoE kernel with a switch named A4W4 next to
 * the FP8 second-stage switch ("Appendix: environment variables" of "Kimi
 * K3.1 Pro on AMD Instinct GPUs"): 4-bit activations with the 4-bit weights.
 * These entry points run stage 1 with MXFP4 activations (E2M1 elements, one
 * E8M0 scale per 32, shared exponent floor(log2(amax)) - 2, elements rounded
 * to nearest even and saturated to +-6; -0 kept) on kind::mxf4 tensor cores;
 * stage 2 is unchanged (MXFP8 h, the FP8 second stage). */

/* MXFP4 quantisation of bf16 activations, otherwise as moe_quant_mxfp8:
 * codes packed [rows_capacity][d/2] (even element in the low nibble of each
 * byte, 4-byte aligned), scales in scale_layout for (rows_capacity, d). */
moe_status moe_quant_mxfp4(const uint16_t* x, int32_t T, int32_t d, const int32_t* slot_to_row,
                           int32_t k, uint8_t* codes, uint8_t* scales, int32_t scale_layout,
                           int64_t rows_capacity, cudaStream_t stream);

/* Stage 1 with MXFP4 activations (token tiles: groups padded to 128, xs
 * TILED): g, u, h as in moe_grouped_gemm_w13_glu with X decoded from E2M1;
 * h -> MXFP8 codes hq and scales hs in hs_layout (TILED for the token-tile
 * stage 2, GROUP32 for the weight-tile stage 2). xq packed [rows_capacity][d/2];
 * d % 256 == 0 (MOE_ERR_UNSUPPORTED otherwise). w13 and w13_sf, counts,
 * offsets, alignment, padding rows and errors as moe_grouped_gemm_w13_glu. */
moe_status moe_grouped_gemm_w13_glu_a4w4(const uint8_t* xq, const uint8_t* xs,
                                         const int32_t* counts, const int32_t* offsets, int32_t E,
                                         int32_t d, int32_t I, int32_t hs_layout,
                                         const uint8_t* w13, const uint8_t* w13_sf, uint8_t* hq,
                                         uint8_t* hs, int64_t rows_capacity, void* ws,
                                         size_t ws_bytes, cudaStream_t stream);

/* The whole layer with MXFP4 stage-1 activations: route -> permute (groups
 * of 128) -> MXFP4 quantise -> A4W4 stage 1 + GLU + MXFP8 requant -> stage 2
 * -> combine. kernel selects the stage-2 family (MOE_GEMM_AUTO =
 * moe_default_kernel); stage 1 always runs on token tiles. d % 256 == 0.
 * Other arguments as moe_forward. */
moe_status moe_forward_a4w4(const moe_dims* dims, int32_t kernel, const uint16_t* x,
                            const float* logits, const moe_weights* weights, uint16_t* y,
                            int32_t* topk_ids_out, float* topk_w_out, void* ws, size_t ws_bytes,
                            cudaStream_t stream);

/* ---- Neighbouring BF16 steps ------------------------------------------------
 * The pages' layer runs its router GEMM, the latent down/up projections
 * (7,168 <-> 3,584) and two shared experts in BF16 beside the MXFP4 routed
 * experts ("Kimi K3.1 Pro at a glance" and "The MXFP4 latent MoE on FlyDSL"
 * of "Kimi K3.1 Pro on AMD Instinct GPUs"; "HBM Usage Under TP8" of "Day 0
 * Kimi-K3 Inference Deployment with ATOM on AMD Instinct MI355X GPUs"). They
 * are dense products C = A . B^T of bf16 operands with fp32 accumulation on
 * tcgen05 tensor cores (kind::f16). */
typedef enum {
  MOE_EPI_F32 = 0,          /* C fp32 [M][N] (router logits) */
  MOE_EPI_BF16 = 1,         /* C bf16 [M][N], round to nearest even */
  MOE_EPI_SWIGLU_BF16 = 2   /* B = N/2 gate rows then N/2 up rows; C = h bf16 [M][N/2],
                               h = silu(A . Bgate^T) * (A . Bup^T) (a shared expert's
                               gated MLP step); N % 256 == 0 */
} moe_gemm_epilogue;

/* C = A . B^T: a bf16 [M][K], b bf16 [N][K] (both K-major, 16-byte aligned),
 * c [M][N] (or [M][N/2] for MOE_EPI_SWIGLU_BF16), 16-byte aligned.
 * K % 64 == 0, N % 8 == 0 (MOE_ERR_UNSUPPORTED otherwise); any M.
 * ws (16-byte aligned): moe_gemm_bf16_workspace_size bytes; its status word
 * records device timeouts, and calls with few output tiles (small M) split K
 * over the SMs and keep fp32 partial sums there, added in a fixed order, so
 * the result does not depend on the split. */
moe_status moe_gemm_bf16(const uint16_t* a, const uint16_t* b, int64_t M, int32_t N, int32_t K,
                         int32_t epilogue, void* c, void* ws, size_t ws_bytes,
                         cudaStream_t stream);

/* Workspace bytes of moe_gemm_bf16 for this shape (0 for an unsupported one). */
size_t moe_gemm_bf16_workspace_size(int64_t M, int32_t N, int32_t K, int32_t epilogue);

/* The router GEMM: logits fp32 [T][E] = x bf16 [T][d_in] . w_router bf16
 * [E][d_in]^T, the input of moe_route_topk / moe_forward. d_in % 64 == 0,
 * E % 8 == 0, E <= 1024; ws: moe_gemm_bf16_workspace_size(T, E, d_in,
 * MOE_EPI_F32) bytes. */
moe_status moe_router_logits(const uint16_t* x, const uint16_t* w_router, int32_t T,
                             int32_t d_in, int32_t E, float* logits, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* C = [A1 | A2] . B^T: moe_gemm_bf16 with A given in two parts along K,
 * a1 bf16 [M][K1] and a2 bf16 [M][K2] (each K-major, 16-byte aligned), b bf16
 * [N][K1 + K2]; c, epilogue, ws and the split of K as moe_gemm_bf16 with
 * K = K1 + K2 (moe_gemm_bf16_workspace_size(M, N, K1 + K2, epilogue)).
 * K1 >= 64, K1 % 64 == 0, K2 % 64 == 0 (K2 = 0 is moe_gemm_bf16); a2 may be
 * NULL when K2 == 0. The composed block's output GEMM reads the routed
 * experts' latent output and the shared experts' h this way, without copying
 * them side by side. */
moe_status moe_gemm_bf16_cat(const uint16_t* a1, int32_t K1, const uint16_t* a2, int32_t K2,
                             const uint16_t* b, int64_t M, int32_t N, int32_t epilogue, void* c,
                             void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---- The composed latent-MoE block -----------------------------------------
 * "Kimi K3.1 Pro at a glance": 896 routed experts (top-16, sigmoid routing)
 * plus two shared experts; the routed experts work in a 3,584-wide latent,
 * half the 7,168-wide hidden size; shared experts, latent up/down projections
 * and router are BF16. "The MXFP4 latent MoE on FlyDSL": the two shared
 * experts run on a second stream, concurrently with the routed experts. "Day
 * 0 Kimi-K3 ...", "Kimi-K3 Architecture and Weights": Stable LatentMoE first
 * projects the hidden state down to the latent.
 *
 * For hidden states h bf16 [T][hidden]:
 *   x      = bf16(h . w_down^T)                      [T][d]     latent down
 *   logits = h . w_router^T (fp32)                    [T][E]     router
 *   y_lat  = moe_forward(x, logits)                   [T][d]     routed experts
 *   hs     = bf16(silu(h . G^T) * (h . U^T))          [T][shared_I]
 *   out    = bf16([y_lat | hs] . w_out^T)             [T][hidden]
 * (fp32 accumulation in every product). Readings where the pages are silent:
 * the router reads the hidden state; each shared expert is a SwiGLU MLP
 * hidden -> 3,072 -> hidden, and the two are stored as one gated MLP of
 * intermediate width shared_I = 6,144 (the sum of two gated MLPs is one gated
 * MLP over their concatenated intermediate rows); the block's output is the
 * latent up projection of y_lat plus the shared experts' output. */
typedef struct {
  int32_t T;        /* tokens */
  int32_t hidden;   /* hidden width (7168); % 64 */
  int32_t d;        /* latent width (3584) */
  int32_t E;        /* routed experts (896); % 8 */
  int32_t k;        /* experts per token (16) */
  int32_t I;        /* routed expert intermediate width (3072) */
  int32_t shared_I; /* intermediate width of all shared experts together (2 x 3072); % 128 */
} moe_block_dims;

typedef struct {
  const uint16_t* w_down;     /* bf16 [d][hidden] latent down projection */
  const uint16_t* w_router;   /* bf16 [E][hidden] */
  const uint16_t* w_shared13; /* bf16 [2*shared_I][hidden]: the shared experts' gate rows
                                 (expert 0 then expert 1), then their up rows, same order */
  const uint16_t* w_out;      /* bf16 [hidden][d + shared_I]: columns 0..d-1 the latent up
                                 projection, columns d.. the shared experts' down
                                 projections (expert 0 then expert 1) */
  moe_weights routed;         /* the routed experts, as for moe_forward */
} moe_block_weights;

/* Workspace bytes of moe_block_forward for these dims. The routed-layer
 * shape rules of moe_workspace_size apply, plus hidden % 64 == 0, E % 8 == 0
 * and shared_I % 128 == 0 (MOE_ERR_UNSUPPORTED otherwise). */
moe_status moe_block_workspace_size(const moe_block_dims* dims, size_t* bytes);

/* The block on `stream`, with the shared experts on `shared_stream`
 * concurrently with the latent down projection, the router and the routed
 * experts (fork and join by CUDA events; with shared_stream == stream
 * everything runs in order on `stream`). Work that precedes the call on
 * `stream` is complete before either stream reads h; when the call returns
 * to the host, all its work is enqueued on `stream` (the join), so later
 * work on `stream` sees `out`. kernel: the routed experts' GEMM family as in
 * moe_forward. h, out 16-byte aligned; ws moe_block_workspace_size bytes,
 * 256-byte aligned, status word at its start (moe_check_device_status);
 * weights 16-byte aligned (routed weights as moe_forward). The fork and join
 * events are created on the first call in each host thread for each device
 * and kept; make that first call before any stream capture. Concurrent calls
 * need distinct workspaces. */
moe_status moe_block_forward(const moe_block_dims* dims, int32_t kernel, const uint16_t* h,
                             const moe_block_weights* weights, uint16_t* out, void* ws,
                             size_t ws_bytes, cudaStream_t stream, cudaStream_t shared_stream);

/* Synchronises `stream`, then returns the status recorded in the workspace's
 * status word (MOE_OK if none). */
moe_status moe_check_device_status(const void* ws, cudaStream_t stream);

/* Enqueues a reset of the status word to MOE_OK. */
moe_status moe_clear_device_status(void* ws, cudaStream_t stream);

/* Self-test of the bounded device wait used by the GEMM pipelines: one CTA
 * waits on a shared-memory barrier that nothing signals, gives up after
 * `limit_us` microseconds and records MOE_ERR_DEVICE_TIMEOUT in the status
 * word. Never hangs or traps; the context stays usable. */
moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us,
                                     cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif
