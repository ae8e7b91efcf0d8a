// Launchers of the libmoe kernels (host side, C++ linkage, not exported).
// Arguments are validated by the C-ABI layer (api.cu) before they get here.
#pragma once

#include <climits>

#include "common.cuh"

namespace moe {

// Shape limits of every routing and grouping entry point: E experts (one
// thread per expert in the grouping scans and in the GEMMs' tile prefix) and
// k selected experts per token (one lane per selected expert in routing).
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;

inline moe_status check_routing_shape(int32_t T, int32_t E, int32_t k) {
  if (T < 0 || E < 0 || k < 0) return MOE_ERR_INVALID_ARGUMENT;
  if (E < 1 || E > kMaxExperts || k > kMaxTopK || k > E) return MOE_ERR_UNSUPPORTED;
  if (int64_t(T) * k >= int64_t(INT32_MAX)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// v is a power of two in [lo, hi].
inline bool pow2_in(int32_t v, int32_t lo, int32_t hi) {
  return v >= lo && v <= hi && (v & (v - 1)) == 0;
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int* ids, float* w,
                              cudaStream_t st);

size_t permute_scratch_bytes(int T, int E);
cudaError_t launch_permute(const int* ids, int T, int E, int k, int pad_m, int* counts,
                           int* offsets, int* slot_to_row, int* row_to_slot,
                           int64_t rows_capacity, int* hist, int* status, cudaStream_t st);

cudaError_t launch_quant_mxfp8(const uint16_t* x, int T, int d, const int* slot_to_row, int k,
                               uint8_t* codes, uint8_t* scales, int layout, cudaStream_t st);
cudaError_t launch_quant_mxfp4(const uint16_t* x, int T, int d, const int* slot_to_row, int k,
                               uint8_t* codes, uint8_t* scales, int layout, cudaStream_t st);
cudaError_t launch_prepack_scales(const uint8_t* src, int64_t rows, int K, uint8_t* dst,
                                  cudaStream_t st);
cudaError_t launch_prepack_weights(const uint8_t* src, int64_t rows, int K, uint8_t* dst,
                                   cudaStream_t st);

cudaError_t launch_gemm_w13_glu(const uint8_t* xq, const uint8_t* xs, const int* counts,
                                const int* offsets, int E, int d, int I, const uint8_t* w13,
                                const uint8_t* w13_sf, uint8_t* hq, uint8_t* hs,
                                int64_t rows_capacity, int* status, cudaStream_t st);
// A4W4 stage 1 (token tiles only): MXFP4 activations xq [rows][d/2] with
// TILED scales, hs written in hs_layout (TILED or GROUP32).
cudaError_t launch_gemm_w13_glu_a4w4(const uint8_t* xq, const uint8_t* xs, const int* counts,
                                     const int* offsets, int E, int d, int I, const uint8_t* w13,
                                     const uint8_t* w13_sf, uint8_t* hq, uint8_t* hs,
                                     int hs_layout, int64_t rows_capacity, int* status,
                                     cudaStream_t st);
// The full 256-row pairs of each expert's m-tiles over CTA pairs
// (gemm_token_pair.cu); the launch_gemm_* entry points run these first.
cudaError_t launch_token_pairs_w13_glu(const uint8_t* xq, const uint8_t* xs, const int* counts,
                                       const int* offsets, int E, int d, int I, const uint8_t* w13,
                                       const uint8_t* w13_sf, uint8_t* hq, uint8_t* hs,
                                       int64_t rows_capacity, int* status, cudaStream_t st);
cudaError_t launch_token_pairs_w13_glu_a4w4(const uint8_t* xq, const uint8_t* xs,
                                            const int* counts, const int* offsets, int E, int d,
                                            int I, const uint8_t* w13, const uint8_t* w13_sf,
                                            uint8_t* hq, uint8_t* hs, int hs_layout,
                                            int64_t rows_capacity, int* status, cudaStream_t st);
cudaError_t launch_token_pairs_w2(const uint8_t* hq, const uint8_t* hs, const int* counts,
                                  const int* offsets, int E, int I, int d, const uint8_t* w2,
                                  const uint8_t* w2_sf, uint16_t* yp, int64_t rows_capacity,
                                  int* status, cudaStream_t st);
cudaError_t launch_gemm_w2(const uint8_t* hq, const uint8_t* hs, const int* counts,
                           const int* offsets, int E, int I, int d, const uint8_t* w2,
                           const uint8_t* w2_sf, uint16_t* yp, int64_t rows_capacity, int* status,
                           cudaStream_t st);
// Shared by the grouped GEMMs: 2-D K-major operand tensor map (dim0 = K
// inputs, dim1 = rows, 128-input boxes of box_rows rows, 128-byte swizzle;
// E2M1 operands use TMA's 16U4_ALIGN16B expansion), and the SM count.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();   // cuTensorMapEncodeTiled through the runtime, cached
bool encode_operand(CUtensorMap* map, const void* base, bool e2m1, int K, int64_t rows,
                    int box_rows);
bool encode_boxed_weights(CUtensorMap* map, const void* base, int64_t rows, int K);
bool encode_boxed_weights_packed(CUtensorMap* map, const void* base, int64_t rows, int K);
// A TILED scale array as rows of 128 bytes, boxes of one 512-byte atom.
bool encode_scale_atoms(CUtensorMap* map, const void* base, int64_t bytes);
int sm_count();

cudaError_t launch_gemm_decode_w13_glu(const uint8_t* xq, const uint8_t* xs, const int* counts,
                                       const int* offsets, int E, int d, int I,
                                       const uint8_t* w13, const uint8_t* w13_sf, uint8_t* hq,
                                       uint8_t* hs, int64_t rows_capacity, int* status,
                                       cudaStream_t st);
cudaError_t launch_gemm_decode_w2(const uint8_t* hq, const uint8_t* hs, const int* counts,
                                  const int* offsets, int E, int I, int d, const uint8_t* w2,
                                  const uint8_t* w2_sf, uint16_t* yp, int64_t rows_capacity,
                                  int* status, cudaStream_t st);
// CTA-pair tiles (gemm_pair.cu): weights on M over two SMs, tokens on N;
// groups of 128 rows, TILED activation scales; d % 256 == 0, I % 256 == 0.
cudaError_t launch_gemm_pair_w13_glu(const uint8_t* xq, const uint8_t* xs, const int* counts,
                                     const int* offsets, int E, int d, int I, const uint8_t* w13,
                                     const uint8_t* w13_sf, uint8_t* hq, uint8_t* hs,
                                     int64_t rows_capacity, int* status, cudaStream_t st);
cudaError_t launch_gemm_pair_w2(const uint8_t* hq, const uint8_t* hs, const int* counts,
                                const int* offsets, int E, int I, int d, const uint8_t* w2,
                                const uint8_t* w2_sf, uint16_t* yp, int64_t rows_capacity,
                                int* status, cudaStream_t st);
// Dense BF16 GEMM C = A . B^T (gemm_bf16.cu); epilogues as moe_gemm_epilogue.
enum GemmEpilogue : int { kEpiF32 = 0, kEpiBf16 = 1, kEpiSwiglu = 2 };
int bf16_k_splits(int64_t M, int N, int K, int epilogue);
size_t bf16_partial_bytes(int64_t M, int N, int K, int epilogue);   // 0 without a split
cudaError_t launch_gemm_bf16(const uint16_t* a, const uint16_t* b, int64_t M, int N, int K,
                             int epilogue, void* c, float* partial, int* status, cudaStream_t st);
// The same with A = [A1 | A2] along K (A1 [M][K1], A2 [M][K2], K1 and K2
// multiples of 64; K2 may be 0): C = A1 . B[:, :K1]^T + A2 . B[:, K1:]^T.
cudaError_t launch_gemm_bf16_cat(const uint16_t* a1, int K1, const uint16_t* a2, int K2,
                                 const uint16_t* b, int64_t M, int N, int epilogue, void* c,
                                 float* partial, int* status, cudaStream_t st);
cudaError_t launch_wait_timeout_selftest(int* status, uint32_t limit_us, cudaStream_t st);

// moe_forward / moe_forward_a4w4 with device problems recorded in `status`
// (not cleared here) instead of the workspace's own status word.
moe_status forward_with_status(bool a4w4, const moe_dims* dims, int32_t kernel,
                               const uint16_t* x, const float* logits, const moe_weights* W,
                               uint16_t* y, void* ws, size_t ws_bytes, int* status,
                               cudaStream_t stream);

cudaError_t launch_combine(const uint16_t* yp, const int* slot_to_row, const float* w, int T,
                           int k, int d, uint16_t* y, cudaStream_t st);

}  // namespace moe
