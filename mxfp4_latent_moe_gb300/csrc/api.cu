// C-ABI of libmoe.so: argument validation, workspace layout, launches.
// The contract of every entry point is stated in include/moe.h.
#include <climits>

#include "internal.h"

namespace {

using moe::tiled_sf_offset;

using moe::check_routing_shape;
using moe::pow2_in;
constexpr int kMaxE = moe::kMaxExperts;
constexpr int kMaxK = moe::kMaxTopK;
// Expert groups: multiples of 128 rows for token tiles, of 32 for weight tiles
// (whose activation scales use the GROUP32 layout).
int32_t group_pad(int32_t kernel) { return kernel == MOE_GEMM_WEIGHT_TILES ? 32 : 128; }
int32_t scale_layout(int32_t kernel) {
  return kernel == MOE_GEMM_WEIGHT_TILES ? MOE_SCALES_GROUP32 : MOE_SCALES_TILED128;
}

bool kernel_ok(int32_t kernel) {
  return kernel == MOE_GEMM_TOKEN_TILES || kernel == MOE_GEMM_WEIGHT_TILES ||
         kernel == MOE_GEMM_PAIR_TILES;
}

// The pair tiles cover 256 weight rows per tile: gate/up rows in steps of
// 256 of I (stage 1), output features in steps of 256 of d (stage 2).
bool pair_shape_ok(int32_t d, int32_t I) { return d % 256 == 0 && I % 256 == 0; }

// Stage 1 / stage 2 of a family on the given device pointers.
cudaError_t launch_w13(int32_t kernel, const uint8_t* xq, const uint8_t* xs, const int* counts,
                       const int* offsets, int E, int d, int I, const uint8_t* w13,
                       const uint8_t* w13_sf, uint8_t* hq, uint8_t* hs, int64_t rows_capacity,
                       int* status, cudaStream_t st) {
  if (kernel == MOE_GEMM_WEIGHT_TILES)
    return moe::launch_gemm_decode_w13_glu(xq, xs, counts, offsets, E, d, I, w13, w13_sf, hq, hs,
                                           rows_capacity, status, st);
  if (kernel == MOE_GEMM_PAIR_TILES)
    return moe::launch_gemm_pair_w13_glu(xq, xs, counts, offsets, E, d, I, w13, w13_sf, hq, hs,
                                         rows_capacity, status, st);
  return moe::launch_gemm_w13_glu(xq, xs, counts, offsets, E, d, I, w13, w13_sf, hq, hs,
                                  rows_capacity, status, st);
}

cudaError_t launch_w2(int32_t kernel, const uint8_t* hq, const uint8_t* hs, const int* counts,
                      const int* offsets, int E, int I, int d, const uint8_t* w2,
                      const uint8_t* w2_sf, uint16_t* yp, int64_t rows_capacity, int* status,
                      cudaStream_t st) {
  if (kernel == MOE_GEMM_WEIGHT_TILES)
    return moe::launch_gemm_decode_w2(hq, hs, counts, offsets, E, I, d, w2, w2_sf, yp,
                                      rows_capacity, status, st);
  if (kernel == MOE_GEMM_PAIR_TILES)
    return moe::launch_gemm_pair_w2(hq, hs, counts, offsets, E, I, d, w2, w2_sf, yp,
                                    rows_capacity, status, st);
  return moe::launch_gemm_w2(hq, hs, counts, offsets, E, I, d, w2, w2_sf, yp, rows_capacity,
                             status, st);
}

// The grouped-GEMM kernels moe_forward uses for MOE_GEMM_AUTO. Measured on
// GB300 at full layer size, token tiles stream the weights faster than weight
// tiles at every batch tried (64 and 512 tokens as well as prefill), so AUTO
// picks token tiles for every shape.
// Weight tiles (32- or 64-token chunks on the MMA's N side) while the experts
// average at most 56 routed rows; token tiles (128-token tiles on M) above,
// where two 64-token chunks per expert cost more than the 128-row tiles
// waste on padding (measured at the full dims: weight tiles ahead up to
// T = 3072, token tiles from T = 3584).
int32_t auto_kernel(int32_t T, int32_t E, int32_t k) {
  return int64_t(T) * k <= 56 * int64_t(E) ? MOE_GEMM_WEIGHT_TILES : MOE_GEMM_TOKEN_TILES;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status check_width(int32_t w) {
  if (w < 0) return MOE_ERR_INVALID_ARGUMENT;
  if (w < 128 || w % 128 != 0 || w > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int64_t rows_capacity_of(int32_t T, int32_t E, int32_t k, int32_t pad_m) {
  const int64_t slots = int64_t(T) * k;
  const int64_t rows = slots + (slots < E ? slots : int64_t(E)) * (pad_m - 1);
  return (rows + 127) / 128 * 128;
}

size_t tiled_bytes(int64_t rows, int32_t K) {
  const int64_t rp = (rows + 127) / 128 * 128;
  return size_t(rp) * size_t(K / 32);
}

size_t group32_bytes(int64_t rows, int32_t K) {
  const int64_t rp = (rows + 31) / 32 * 32;
  return size_t(rp) * size_t(K / 8);
}

size_t act_scale_bytes(int64_t rows, int32_t K, int32_t layout) {
  return layout == MOE_SCALES_GROUP32 ? group32_bytes(rows, K) : tiled_bytes(rows, K);
}

struct ForwardLayout {
  size_t status, hist, ids, w, counts, offsets, s2r, r2s, xq, xs, hq, hs, yp, total;
  int64_t rows_cap;
};

// Workspace carve-up for one forward: groups padded to pad_m, activation
// scales of x in xs_layout and of h in hs_layout.
ForwardLayout forward_layout(const moe_dims& D, int32_t pad_m, int32_t xs_layout,
                             int32_t hs_layout) {
  ForwardLayout L{};
  const size_t slots = size_t(D.T) * size_t(D.k);
  L.rows_cap = rows_capacity_of(D.T, D.E, D.k, pad_m);
  const size_t rc = size_t(L.rows_cap);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += round_up(bytes, 256);
    return o;
  };
  L.status = take(MOE_STATUS_BYTES);
  L.hist = take(moe::permute_scratch_bytes(D.T, D.E));
  L.ids = take(slots * 4);
  L.w = take(slots * 4);
  L.counts = take(size_t(D.E) * 4);
  L.offsets = take(size_t(D.E + 1) * 4);
  L.s2r = take(slots * 4);
  L.r2s = take(rc * 4);
  L.xq = take(rc * size_t(D.d));
  L.xs = take(act_scale_bytes(L.rows_cap, D.d, xs_layout));
  L.hq = take(rc * size_t(D.I));
  L.hs = take(act_scale_bytes(L.rows_cap, D.I, hs_layout));
  L.yp = take(rc * size_t(D.d) * 2);
  L.total = off;
  return L;
}

ForwardLayout forward_layout(const moe_dims& D, int32_t kernel) {
  return forward_layout(D, group_pad(kernel), scale_layout(kernel), scale_layout(kernel));
}

// The A4W4 forward: stage 1 on token tiles (groups of 128, TILED x scales),
// h scales in the layout of the stage-2 family.
ForwardLayout forward_layout_a4w4(const moe_dims& D, int32_t stage2_kernel) {
  return forward_layout(D, group_pad(MOE_GEMM_TOKEN_TILES), MOE_SCALES_TILED128,
                        scale_layout(stage2_kernel));
}

moe_status check_dims(const moe_dims* D) {
  if (!D) return MOE_ERR_INVALID_ARGUMENT;
  moe_status s = check_routing_shape(D->T, D->E, D->k);
  if (s != MOE_OK) return s;
  if ((s = check_width(D->d)) != MOE_OK) return s;
  return check_width(D->I);
}

moe_status check_gemm_args(int32_t E, int32_t K, int32_t N, int32_t kernel, int64_t rows_capacity,
                           const void* a, const void* a_sf, const int32_t* counts,
                           const int32_t* offsets,
                           const void* b, const void* b_sf, const void* out, const void* out_sf,
                           bool need_out_sf, const void* ws, size_t ws_bytes) {
  if (!a || !a_sf || !counts || !offsets || !b || !b_sf || !out || !ws ||
      (need_out_sf && !out_sf))
    return MOE_ERR_INVALID_ARGUMENT;
  if (E < 0 || rows_capacity < 0) return MOE_ERR_INVALID_ARGUMENT;
  if (E < 1 || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  moe_status s;
  if ((s = check_width(K)) != MOE_OK) return s;
  if ((s = check_width(N)) != MOE_OK) return s;
  if (!kernel_ok(kernel)) return MOE_ERR_UNSUPPORTED;
  if (rows_capacity % 128 != 0 || rows_capacity >= int64_t(INT32_MAX)) return MOE_ERR_UNSUPPORTED;
  if (!aligned(a, 16) || !aligned(a_sf, 16) || !aligned(b, 32) || !aligned(b_sf, 16) ||
      !aligned(out, 16) || (need_out_sf && !aligned(out_sf, 4)) || !aligned(offsets, 4) ||
      !aligned(counts, 4) || !aligned(ws, 4))
    return MOE_ERR_INVALID_ARGUMENT;
  if (ws_bytes < MOE_STATUS_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

template <class T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or option";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace or row capacity too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device: a bounded wait ran out";
    case MOE_ERR_DEVICE_BAD_INPUT: return "device: bad expert ids or offsets";
  }
  return "unknown status";
}

int32_t moe_abi_version(void) { return 1; }

size_t moe_tiled_scale_bytes(int64_t rows, int32_t K) {
  if (rows < 0 || check_width(K) != MOE_OK) return 0;
  return tiled_bytes(rows, K);
}

size_t moe_activation_scale_bytes(int64_t rows, int32_t K, int32_t scale_layout) {
  if (rows < 0 || check_width(K) != MOE_OK) return 0;
  if (scale_layout != MOE_SCALES_TILED128 && scale_layout != MOE_SCALES_GROUP32) return 0;
  return act_scale_bytes(rows, K, scale_layout);
}

int32_t moe_default_kernel(int32_t T, int32_t E, int32_t k) {
  if (check_routing_shape(T, E, k) != MOE_OK) return -1;
  return auto_kernel(T, E, k);
}

int64_t moe_rows_capacity(int32_t T, int32_t E, int32_t k, int32_t pad_m) {
  if (check_routing_shape(T, E, k) != MOE_OK || !pow2_in(pad_m, 1, 1024)) return -1;
  return rows_capacity_of(T, E, k, pad_m);
}

moe_status moe_prepack_scales(const uint8_t* src, int64_t rows, int32_t K, uint8_t* dst,
                              cudaStream_t stream) {
  if (rows < 0) return MOE_ERR_INVALID_ARGUMENT;
  moe_status s = check_width(K);
  if (s != MOE_OK) return s;
  if (rows == 0) return MOE_OK;
  if (!src || !dst || !aligned(dst, 16)) return MOE_ERR_INVALID_ARGUMENT;
  return from_cuda(moe::launch_prepack_scales(src, rows, K, dst, stream));
}

moe_status moe_prepack_weights(const uint8_t* src, int64_t rows, int32_t K, uint8_t* dst,
                               cudaStream_t stream) {
  if (rows < 0) return MOE_ERR_INVALID_ARGUMENT;
  moe_status s = check_width(K);
  if (s != MOE_OK) return s;
  if (rows % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (!src || !dst || !aligned(src, 16) || !aligned(dst, 32)) return MOE_ERR_INVALID_ARGUMENT;
  return from_cuda(moe::launch_prepack_weights(src, rows, K, dst, stream));
}

moe_status moe_route_topk(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* topk_ids,
                          float* topk_w, cudaStream_t stream) {
  moe_status s = check_routing_shape(T, E, k);
  if (s != MOE_OK) return s;
  if (T == 0 || k == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
    return MOE_ERR_INVALID_ARGUMENT;
  return from_cuda(moe::launch_route_topk(logits, T, E, k, topk_ids, topk_w, stream));
}

size_t moe_permute_workspace_size(int32_t T, int32_t E) {
  if (T < 0 || E < 1 || E > kMaxE) return 0;
  return MOE_STATUS_BYTES + round_up(moe::permute_scratch_bytes(T, E), 256);
}

moe_status moe_permute(const int32_t* topk_ids, int32_t T, int32_t E, int32_t k, int32_t pad_m,
                       int32_t* counts, int32_t* offsets, int32_t* slot_to_row,
                       int32_t* row_to_slot, int64_t rows_capacity, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
  moe_status s = check_routing_shape(T, E, k);
  if (s != MOE_OK) return s;
  if (!pow2_in(pad_m, 1, 1024)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || !ws || rows_capacity < 0) return MOE_ERR_INVALID_ARGUMENT;
  const bool any = T > 0 && k > 0;
  if (any && (!topk_ids || !slot_to_row || !row_to_slot)) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(counts, 4) || !aligned(offsets, 4) || !aligned(ws, 4) ||
      (any && (!aligned(topk_ids, 4) || !aligned(slot_to_row, 4) || !aligned(row_to_slot, 4))))
    return MOE_ERR_INVALID_ARGUMENT;
  const int64_t slots = int64_t(T) * k;
  if (rows_capacity < slots + (slots < E ? slots : int64_t(E)) * (pad_m - 1))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (ws_bytes < moe_permute_workspace_size(T, E)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(moe::launch_permute(topk_ids, T, E, k, pad_m, counts, offsets, slot_to_row,
                                       row_to_slot, rows_capacity, at<int>(ws, MOE_STATUS_BYTES),
                                       static_cast<int*>(ws), stream));
}

moe_status moe_quant_mxfp8(const uint16_t* x, int32_t T, int32_t d, const int32_t* slot_to_row,
                           int32_t k, uint8_t* codes, uint8_t* scales, int32_t scale_layout,
                           int64_t rows_capacity, cudaStream_t stream) {
  if (T < 0 || k < 0 || rows_capacity < 0) return MOE_ERR_INVALID_ARGUMENT;
  moe_status s = check_width(d);
  if (s != MOE_OK) return s;
  if (k > kMaxK || int64_t(T) * (k > 0 ? k : 1) >= int64_t(INT32_MAX)) return MOE_ERR_UNSUPPORTED;
  if (rows_capacity % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (scale_layout != MOE_SCALES_TILED128 && scale_layout != MOE_SCALES_GROUP32)
    return MOE_ERR_UNSUPPORTED;
  if (T == 0 || (slot_to_row && k == 0)) return MOE_OK;
  if (!x || !codes || !scales) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(codes, 8) || !aligned(scales, 4) ||
      (slot_to_row && !aligned(slot_to_row, 4)))
    return MOE_ERR_INVALID_ARGUMENT;
  if (!slot_to_row && rows_capacity < T) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(
      moe::launch_quant_mxfp8(x, T, d, slot_to_row, k, codes, scales, scale_layout, stream));
}

moe_status moe_quant_mxfp4(const uint16_t* x, int32_t T, int32_t d, const int32_t* slot_to_row,
                           int32_t k, uint8_t* codes, uint8_t* scales, int32_t scale_layout,
                           int64_t rows_capacity, cudaStream_t stream) {
  if (T < 0 || k < 0 || rows_capacity < 0) return MOE_ERR_INVALID_ARGUMENT;
  moe_status s = check_width(d);
  if (s != MOE_OK) return s;
  if (k > kMaxK || int64_t(T) * (k > 0 ? k : 1) >= int64_t(INT32_MAX)) return MOE_ERR_UNSUPPORTED;
  if (rows_capacity % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (scale_layout != MOE_SCALES_TILED128 && scale_layout != MOE_SCALES_GROUP32)
    return MOE_ERR_UNSUPPORTED;
  if (T == 0 || (slot_to_row && k == 0)) return MOE_OK;
  if (!x || !codes || !scales) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(codes, 4) || !aligned(scales, 4) ||
      (slot_to_row && !aligned(slot_to_row, 4)))
    return MOE_ERR_INVALID_ARGUMENT;
  if (!slot_to_row && rows_capacity < T) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(
      moe::launch_quant_mxfp4(x, T, d, slot_to_row, k, codes, scales, scale_layout, stream));
}

moe_status moe_grouped_gemm_w13_glu(const uint8_t* xq, const uint8_t* xs, const int32_t* counts,
                                    const int32_t* offsets, int32_t E, int32_t d, int32_t I,
                                    int32_t kernel, const uint8_t* w13, const uint8_t* w13_sf,
                                    uint8_t* hq, uint8_t* hs, int64_t rows_capacity, void* ws,
                                    size_t ws_bytes, cudaStream_t stream) {
  moe_status s = check_gemm_args(E, d, I, kernel, rows_capacity, xq, xs, counts, offsets, w13,
                                 w13_sf, hq, hs, true, ws, ws_bytes);
  if (s != MOE_OK) return s;
  if (kernel == MOE_GEMM_PAIR_TILES && !pair_shape_ok(d, I)) return MOE_ERR_UNSUPPORTED;
  if (rows_capacity == 0) return MOE_OK;
  return from_cuda(launch_w13(kernel, xq, xs, counts, offsets, E, d, I, w13, w13_sf, hq, hs,
                              rows_capacity, static_cast<int*>(ws), stream));
}

moe_status moe_grouped_gemm_w13_glu_a4w4(const uint8_t* xq, const uint8_t* xs,
                                         const int32_t* counts, const int32_t* offsets, int32_t E,
                                         int32_t d, int32_t I, int32_t hs_layout,
                                         const uint8_t* w13, const uint8_t* w13_sf, uint8_t* hq,
                                         uint8_t* hs, int64_t rows_capacity, void* ws,
                                         size_t ws_bytes, cudaStream_t stream) {
  moe_status s = check_gemm_args(E, d, I, MOE_GEMM_TOKEN_TILES, rows_capacity, xq, xs, counts,
                                 offsets, w13, w13_sf, hq, hs, true, ws, ws_bytes);
  if (s != MOE_OK) return s;
  if (d % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (hs_layout != MOE_SCALES_TILED128 && hs_layout != MOE_SCALES_GROUP32)
    return MOE_ERR_UNSUPPORTED;
  if (rows_capacity == 0) return MOE_OK;
  return from_cuda(moe::launch_gemm_w13_glu_a4w4(xq, xs, counts, offsets, E, d, I, w13, w13_sf,
                                                 hq, hs, hs_layout, rows_capacity,
                                                 static_cast<int*>(ws), stream));
}

moe_status moe_grouped_gemm_w2(const uint8_t* hq, const uint8_t* hs, const int32_t* counts,
                               const int32_t* offsets, int32_t E, int32_t I, int32_t d,
                               int32_t kernel, const uint8_t* w2, const uint8_t* w2_sf,
                               uint16_t* yp, int64_t rows_capacity, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  moe_status s = check_gemm_args(E, I, d, kernel, rows_capacity, hq, hs, counts, offsets, w2,
                                 w2_sf, yp, nullptr, false, ws, ws_bytes);
  if (s != MOE_OK) return s;
  if (kernel == MOE_GEMM_PAIR_TILES && !pair_shape_ok(d, I)) return MOE_ERR_UNSUPPORTED;
  if (rows_capacity == 0) return MOE_OK;
  return from_cuda(launch_w2(kernel, hq, hs, counts, offsets, E, I, d, w2, w2_sf, yp,
                             rows_capacity, static_cast<int*>(ws), stream));
}

moe_status moe_gemm_bf16(const uint16_t* a, const uint16_t* b, int64_t M, int32_t N, int32_t K,
                         int32_t epilogue, void* c, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0) return MOE_ERR_INVALID_ARGUMENT;
  if (epilogue != MOE_EPI_F32 && epilogue != MOE_EPI_BF16 && epilogue != MOE_EPI_SWIGLU_BF16)
    return MOE_ERR_UNSUPPORTED;
  if (K < 64 || K % 64 != 0 || K > (1 << 20) || N < 8 || N % 8 != 0 || N > (1 << 20) ||
      M >= int64_t(INT32_MAX))
    return MOE_ERR_UNSUPPORTED;
  if (epilogue == MOE_EPI_SWIGLU_BF16 && N % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (M == 0) return MOE_OK;
  if (!a || !b || !c || !ws) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(a, 16) || !aligned(b, 16) || !aligned(c, 16) || !aligned(ws, 16))
    return MOE_ERR_INVALID_ARGUMENT;
  if (ws_bytes < MOE_STATUS_BYTES + moe::bf16_partial_bytes(M, N, K, epilogue))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(moe::launch_gemm_bf16(a, b, M, N, K, epilogue, c,
                                         at<float>(ws, MOE_STATUS_BYTES),
                                         static_cast<int*>(ws), stream));
}

moe_status moe_gemm_bf16_cat(const uint16_t* a1, int32_t K1, const uint16_t* a2, int32_t K2,
                             const uint16_t* b, int64_t M, int32_t N, int32_t epilogue, void* c,
                             void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (M < 0 || N < 0 || K1 < 0 || K2 < 0) return MOE_ERR_INVALID_ARGUMENT;
  if (epilogue != MOE_EPI_F32 && epilogue != MOE_EPI_BF16 && epilogue != MOE_EPI_SWIGLU_BF16)
    return MOE_ERR_UNSUPPORTED;
  const int64_t K = int64_t(K1) + K2;
  if (K1 < 64 || K1 % 64 != 0 || K2 % 64 != 0 || K > (1 << 20) || N < 8 || N % 8 != 0 ||
      N > (1 << 20) || M >= int64_t(INT32_MAX))
    return MOE_ERR_UNSUPPORTED;
  if (epilogue == MOE_EPI_SWIGLU_BF16 && N % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (M == 0) return MOE_OK;
  if (!a1 || (K2 > 0 && !a2) || !b || !c || !ws) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(a1, 16) || (K2 > 0 && !aligned(a2, 16)) || !aligned(b, 16) || !aligned(c, 16) ||
      !aligned(ws, 16))
    return MOE_ERR_INVALID_ARGUMENT;
  if (ws_bytes < MOE_STATUS_BYTES + moe::bf16_partial_bytes(M, N, int(K), epilogue))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(moe::launch_gemm_bf16_cat(a1, K1, a2, K2, b, M, N, epilogue, c,
                                             at<float>(ws, MOE_STATUS_BYTES),
                                             static_cast<int*>(ws), stream));
}

size_t moe_gemm_bf16_workspace_size(int64_t M, int32_t N, int32_t K, int32_t epilogue) {
  if (M < 0 || N < 8 || N % 8 != 0 || K < 64 || K % 64 != 0) return 0;
  if (epilogue != MOE_EPI_F32 && epilogue != MOE_EPI_BF16 && epilogue != MOE_EPI_SWIGLU_BF16)
    return 0;
  return MOE_STATUS_BYTES + moe::bf16_partial_bytes(M, N, K, epilogue);
}

moe_status moe_router_logits(const uint16_t* x, const uint16_t* w_router, int32_t T,
                             int32_t d_in, int32_t E, float* logits, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
  if (T < 0 || E < 0) return MOE_ERR_INVALID_ARGUMENT;
  if (E < 1 || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  return moe_gemm_bf16(x, w_router, T, E, d_in, MOE_EPI_F32, logits, ws, ws_bytes, stream);
}

moe_status moe_unpermute_combine(const uint16_t* yp, const int32_t* slot_to_row,
                                 const float* topk_w, int32_t T, int32_t k, int32_t d,
                                 uint16_t* y, cudaStream_t stream) {
  if (T < 0 || k < 0) return MOE_ERR_INVALID_ARGUMENT;
  moe_status s = check_width(d);
  if (s != MOE_OK) return s;
  if (k > kMaxK || int64_t(T) * k >= int64_t(INT32_MAX)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y || (k > 0 && (!yp || !slot_to_row || !topk_w))) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(y, 16) || (k > 0 && (!aligned(yp, 16) || !aligned(slot_to_row, 4) ||
                                    !aligned(topk_w, 4))))
    return MOE_ERR_INVALID_ARGUMENT;
  return from_cuda(moe::launch_combine(yp, slot_to_row, topk_w, T, k, d, y, stream));
}

moe_status moe_workspace_size(const moe_dims* dims, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARGUMENT;
  moe_status s = check_dims(dims);
  if (s != MOE_OK) return s;
  size_t m = 0;
  for (const size_t t : {forward_layout(*dims, MOE_GEMM_TOKEN_TILES).total,
                         forward_layout(*dims, MOE_GEMM_WEIGHT_TILES).total,
                         forward_layout_a4w4(*dims, MOE_GEMM_TOKEN_TILES).total,
                         forward_layout_a4w4(*dims, MOE_GEMM_WEIGHT_TILES).total})
    m = t > m ? t : m;
  *bytes = m;
  return MOE_OK;
}

}  // extern "C"

namespace {

// The layer, MXFP8 (a4w4 = false) or with MXFP4 stage-1 activations. kernel
// is the GEMM family of both stages (MXFP8) or of stage 2 (A4W4, whose stage 1
// always runs on token tiles). Device problems go to `status_out` when given
// (the composed block's status word, already cleared by the caller), else to
// the status word at the start of ws, which this call clears first.
moe_status forward_impl(bool a4w4, const moe_dims* dims, int32_t kernel, const uint16_t* x,
                        const float* logits, const moe_weights* W, uint16_t* y,
                        int32_t* topk_ids_out, float* topk_w_out, void* ws, size_t ws_bytes,
                        cudaStream_t stream, int* status_out = nullptr) {
  moe_status s = check_dims(dims);
  if (s != MOE_OK) return s;
  if (a4w4 && dims->d % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (kernel == MOE_GEMM_AUTO) kernel = auto_kernel(dims->T, dims->E, dims->k);
  if (!kernel_ok(kernel)) return MOE_ERR_UNSUPPORTED;
  if (kernel == MOE_GEMM_PAIR_TILES && !pair_shape_ok(dims->d, dims->I))
    return MOE_ERR_UNSUPPORTED;
  const int32_t pad_m = group_pad(a4w4 ? int32_t(MOE_GEMM_TOKEN_TILES) : kernel);
  const moe_dims D = *dims;
  if (D.T == 0) return MOE_OK;
  if (!x || !logits || !W || !y || !ws || !W->w13 || !W->w13_sf || !W->w2 || !W->w2_sf)
    return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(logits, 4) || !aligned(ws, 256) ||
      !aligned(W->w13, 32) || !aligned(W->w2, 32) || !aligned(W->w13_sf, 16) ||
      !aligned(W->w2_sf, 16) || (topk_ids_out && !aligned(topk_ids_out, 4)) ||
      (topk_w_out && !aligned(topk_w_out, 4)))
    return MOE_ERR_INVALID_ARGUMENT;
  const ForwardLayout L = a4w4 ? forward_layout_a4w4(D, kernel) : forward_layout(D, kernel);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;

  int* status = status_out ? status_out : at<int>(ws, L.status);
  cudaError_t e = status_out ? cudaSuccess : cudaMemsetAsync(status, 0, sizeof(int), stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (D.k == 0) return from_cuda(cudaMemsetAsync(y, 0, size_t(D.T) * D.d * 2, stream));

  int* ids = topk_ids_out ? topk_ids_out : at<int>(ws, L.ids);
  float* w = topk_w_out ? topk_w_out : at<float>(ws, L.w);
  int* counts = at<int>(ws, L.counts);
  int* offsets = at<int>(ws, L.offsets);
  int* s2r = at<int>(ws, L.s2r);
  int* r2s = at<int>(ws, L.r2s);
  uint8_t* xq = at<uint8_t>(ws, L.xq);
  uint8_t* xs = at<uint8_t>(ws, L.xs);
  uint8_t* hq = at<uint8_t>(ws, L.hq);
  uint8_t* hs = at<uint8_t>(ws, L.hs);
  uint16_t* yp = at<uint16_t>(ws, L.yp);

  if ((e = moe::launch_route_topk(logits, D.T, D.E, D.k, ids, w, stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if ((e = moe::launch_permute(ids, D.T, D.E, D.k, pad_m, counts, offsets, s2r, r2s, L.rows_cap,
                               at<int>(ws, L.hist), status, stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (a4w4) {
    if ((e = moe::launch_quant_mxfp4(x, D.T, D.d, s2r, D.k, xq, xs, MOE_SCALES_TILED128,
                                     stream)) != cudaSuccess)
      return MOE_ERR_CUDA;
    if ((e = moe::launch_gemm_w13_glu_a4w4(xq, xs, counts, offsets, D.E, D.d, D.I, W->w13,
                                           W->w13_sf, hq, hs, scale_layout(kernel), L.rows_cap,
                                           status, stream)) != cudaSuccess)
      return MOE_ERR_CUDA;
    if ((e = launch_w2(kernel, hq, hs, counts, offsets, D.E, D.I, D.d, W->w2, W->w2_sf, yp,
                       L.rows_cap, status, stream)) != cudaSuccess)
      return MOE_ERR_CUDA;
    return from_cuda(moe::launch_combine(yp, s2r, w, D.T, D.k, D.d, y, stream));
  }
  if ((e = moe::launch_quant_mxfp8(x, D.T, D.d, s2r, D.k, xq, xs, scale_layout(kernel),
                                   stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if ((e = launch_w13(kernel, xq, xs, counts, offsets, D.E, D.d, D.I, W->w13, W->w13_sf, hq, hs,
                      L.rows_cap, status, stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if ((e = launch_w2(kernel, hq, hs, counts, offsets, D.E, D.I, D.d, W->w2, W->w2_sf, yp,
                     L.rows_cap, status, stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return from_cuda(moe::launch_combine(yp, s2r, w, D.T, D.k, D.d, y, stream));
}

}  // namespace

extern "C" {

moe_status moe_forward(const moe_dims* dims, int32_t kernel, const uint16_t* x,
                       const float* logits, const moe_weights* W, uint16_t* y,
                       int32_t* topk_ids_out, float* topk_w_out, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
  return forward_impl(false, dims, kernel, x, logits, W, y, topk_ids_out, topk_w_out, ws,
                      ws_bytes, stream);
}

moe_status moe_forward_a4w4(const moe_dims* dims, int32_t kernel, const uint16_t* x,
                            const float* logits, const moe_weights* W, uint16_t* y,
                            int32_t* topk_ids_out, float* topk_w_out, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
  return forward_impl(true, dims, kernel, x, logits, W, y, topk_ids_out, topk_w_out, ws,
                      ws_bytes, stream);
}

}  // extern "C"

namespace moe {

moe_status forward_with_status(bool a4w4, const moe_dims* dims, int32_t kernel,
                               const uint16_t* x, const float* logits, const moe_weights* W,
                               uint16_t* y, void* ws, size_t ws_bytes, int* status,
                               cudaStream_t stream) {
  return forward_impl(a4w4, dims, kernel, x, logits, W, y, nullptr, nullptr, ws, ws_bytes, stream,
                      status);
}

}  // namespace moe

extern "C" {

moe_status moe_check_device_status(const void* ws, cudaStream_t stream) {
  if (!ws || !aligned(ws, 4)) return MOE_ERR_INVALID_ARGUMENT;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v < 0 || v > int(MOE_ERR_DEVICE_BAD_INPUT)) return MOE_ERR_CUDA;
  return static_cast<moe_status>(v);
}

moe_status moe_clear_device_status(void* ws, cudaStream_t stream) {
  if (!ws || !aligned(ws, 4)) return MOE_ERR_INVALID_ARGUMENT;
  return from_cuda(cudaMemsetAsync(ws, 0, sizeof(int), stream));
}

moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us,
                                     cudaStream_t stream) {
  if (!ws || !aligned(ws, 4)) return MOE_ERR_INVALID_ARGUMENT;
  if (ws_bytes < MOE_STATUS_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (limit_us == 0 || limit_us > 10u * 1000u * 1000u) return MOE_ERR_UNSUPPORTED;
  return from_cuda(moe::launch_wait_timeout_selftest(static_cast<int*>(ws), limit_us, stream));
}

}  // extern "C"
