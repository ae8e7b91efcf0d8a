// MXFP8 (and, for the A4W4 stage 1, MXFP4) quantisation of the stage-1
// activations and the one-time prepack of the MXFP4 weights.
//
// MX rule (OCP MX v1.0; the pages' layer keeps its routed experts in MXFP4
// with one E8M0 scale per 32 values and runs an FP8 second stage, "Kimi K3.1
// Pro on AMD Instinct GPUs", "Kimi K3.1 Pro at a glance" and "The MXFP4 latent
// MoE on FlyDSL"): per 32 consecutive values of a row the scale code is
// clamp(floor(log2(amax)) - 8 + 127, 0, 254), and the elements are the E4M3
// round-to-nearest-even of v * 2^(127 - code), saturated to +-448.
//
// Layout of the work: each thread owns VEC consecutive bf16 of one token
// (VEC/8 16-byte loads; VEC = 8 for small batches, 16 for large ones); the
// 32/VEC lanes of a 32-block take its amax by xor-shuffles and the 128/VEC
// lanes of a 128-input group send its four scale codes out as one 32-bit word
// of the scale layout. The token is read once and written to each of its k
// grouped rows (VEC codes per thread and row, 32 * VEC contiguous codes per
// warp and row).
#include "internal.h"

namespace moe {

namespace {

constexpr int kQuantThreads = 256;
// Grouped rows of a token looked up together: all 16 for small batches
// (decode: one wave of threads, each waiting on its loads); one at a time for
// large ones, which keep occupancy instead.
constexpr int kSmallBatchThreads = 152 * 2048;
constexpr int kLargeBatch = 1;

// Grouped rows j0 .. j0 + B - 1 of token t (below nrows; the dense layout's
// row is t): independent loads issued back to back.
template <int B>
__device__ __forceinline__ void load_rows(const int* __restrict__ slot_to_row, int64_t t, int k,
                                          int nrows, int j0, int (&rows)[B]) {
#pragma unroll
  for (int q = 0; q < B; ++q)
    rows[q] = j0 + q >= nrows ? 0 : slot_to_row ? __ldg(slot_to_row + t * k + j0 + q) : int(t);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& q, float* f) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// MXFP8 (FP4 false: E4M3 elements, shared exponent floor(log2(amax)) - 8,
// codes [rows][d]) or MXFP4 (FP4 true, the A4W4 stage-1 activations: E2M1
// elements, shared exponent floor(log2(amax)) - 2, codes packed [rows][d/2]
// with the even element in the low nibble of each byte).
template <bool FP4, int LAYOUT, int kRowBatch, int VEC>
__global__ void __launch_bounds__(kQuantThreads)
    quant_mx_kernel(const uint4* __restrict__ x, int d, const int* __restrict__ slot_to_row,
                    int k, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                    int64_t total_vec) {
  static_assert(VEC == 8 || VEC == 16, "a thread owns 8 or 16 inputs");
  constexpr int kLoads = VEC / 8;
  constexpr int kBlockLanes = 32 / VEC;             // lanes of a 32-block
  constexpr int kGroupLanes = 128 / VEC;            // lanes of a 128-input group
  constexpr int kWords = FP4 ? VEC / 8 : VEC / 4;   // 32-bit code words per thread
  pdl_trigger();
  pdl_wait();
  const int64_t g = int64_t(blockIdx.x) * kQuantThreads + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const bool valid = g < total_vec;
  const int vpr = d / VEC;   // threads per token
  float f[VEC];
#pragma unroll
  for (int l = 0; l < kLoads; ++l) {
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (valid) raw = __ldg(x + g * kLoads + l);
    bf16x8_to_f32(raw, f + 8 * l);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < VEC; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
  for (int s = 1; s < kBlockLanes; s <<= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, s));
  const int code = FP4 ? mx_scale_code<2>(amax) : mx_scale_code(amax);
  const float m = mx_scale_mult(code);
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < kWords; ++i) {
    if (FP4)
      w[i] = e2m1x2(f[8 * i] * m, f[8 * i + 1] * m) | (e2m1x2(f[8 * i + 2] * m, f[8 * i + 3] * m) << 8) |
             (e2m1x2(f[8 * i + 4] * m, f[8 * i + 5] * m) << 16) |
             (e2m1x2(f[8 * i + 6] * m, f[8 * i + 7] * m) << 24);
    else
      w[i] = e4m3x4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3], m);
  }
  const int base = lane & ~(kGroupLanes - 1);
  const uint32_t s0 = __shfl_sync(0xffffffffu, code, base);
  const uint32_t s1 = __shfl_sync(0xffffffffu, code, base + kBlockLanes);
  const uint32_t s2 = __shfl_sync(0xffffffffu, code, base + 2 * kBlockLanes);
  const uint32_t s3 = __shfl_sync(0xffffffffu, code, base + 3 * kBlockLanes);
  if (!valid) return;
  const uint32_t sword = s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
  const int64_t t = g / vpr;
  const int v = int(g - t * vpr);
  const int64_t row_bytes = FP4 ? d >> 1 : d;
  const int64_t blk = int64_t(v) * VEC / 32;   // first 32-block of the thread
  const int nrows = slot_to_row ? k : 1;
  for (int j0 = 0; j0 < nrows; j0 += kRowBatch) {
    int rows[kRowBatch];
    load_rows<kRowBatch>(slot_to_row, t, k, nrows, j0, rows);
#pragma unroll
    for (int q = 0; q < kRowBatch; ++q) {
      if (j0 + q >= nrows) break;
      const int64_t row = rows[q];
      uint8_t* dst = codes + row * row_bytes + int64_t(v) * (4 * kWords);
      if (kWords == 4)
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      else if (kWords == 2)
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
      else
        *reinterpret_cast<uint32_t*>(dst) = w[0];
      if ((lane & (kGroupLanes - 1)) == 0) {
        const int64_t off = LAYOUT == kScalesGroup32 ? group32_sf_offset(row, blk, d)
                                                     : tiled_sf_offset(row, blk, d);
        *reinterpret_cast<uint32_t*>(scales + off) = sword;
      }
    }
  }
}

// canonical [rows][K/32] -> TILED; one thread per 32-bit output word.
__global__ void prepack_scales_kernel(const uint8_t* __restrict__ src, int64_t rows, int K,
                                      uint8_t* __restrict__ dst, int64_t words) {
  const int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= words) return;
  const int kt_count = K >> 7;
  const int64_t r = g / kt_count;
  const int kt = int(g - r * kt_count);
  uint32_t w = 0;
  if (r < rows) {
    const uint8_t* p = src + r * (K >> 5) + kt * 4;
    w = uint32_t(p[0]) | (uint32_t(p[1]) << 8) | (uint32_t(p[2]) << 16) | (uint32_t(p[3]) << 24);
  }
  *reinterpret_cast<uint32_t*>(dst + tiled_sf_offset(r, int64_t(kt) * 4, K)) = w;
}

// canonical packed E2M1 [rows][K/2] -> BOXED; one thread per 16-byte chunk of
// the output (a box row is 64 bytes = 4 chunks).
__global__ void prepack_weights_kernel(const uint4* __restrict__ src, int K,
                                       uint4* __restrict__ dst, int64_t chunks) {
  const int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= chunks) return;
  const int KT = K >> 7;
  const int64_t box = g >> 9;               // 128 rows x 4 chunks per box
  const int i = int(g >> 2) & 127;          // row inside the box
  const int j = int(g) & 3;                 // 16-byte chunk inside the row
  const int64_t rt = box / KT;
  const int kt = int(box - rt * KT);
  const int64_t row = rt * 128 + i;
  dst[g] = __ldg(src + row * (K >> 5) + kt * 4 + j);   // a row holds K/32 chunks
}

}  // namespace

namespace {

template <bool FP4, int LAYOUT>
cudaError_t launch_quant_layout(const uint16_t* x, int64_t T, int d, const int* slot_to_row, int k,
                                uint8_t* codes, uint8_t* scales, cudaStream_t st) {
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t total8 = T * (d / 8);
  const dim3 grid8(static_cast<unsigned>((total8 + kQuantThreads - 1) / kQuantThreads));
  if (total8 <= kSmallBatchThreads)   // decode-sized: PDL, 16 rows looked up at once
    return launch_ex(true, quant_mx_kernel<FP4, LAYOUT, 16, 8>, grid8, dim3(kQuantThreads), 0, st,
                     1, xv, d, slot_to_row, k, codes, scales, total8);
  // 16 inputs a thread: 16-byte MXFP8 code stores want a 16-byte aligned output
  if (!FP4 && reinterpret_cast<uintptr_t>(codes) % 16 != 0)
    return launch_ex(false, quant_mx_kernel<FP4, LAYOUT, kLargeBatch, 8>, grid8,
                     dim3(kQuantThreads), 0, st, 1, xv, d, slot_to_row, k, codes, scales, total8);
  const int64_t total = T * (d / 16);
  const dim3 grid(static_cast<unsigned>((total + kQuantThreads - 1) / kQuantThreads));
  return launch_ex(false, quant_mx_kernel<FP4, LAYOUT, kLargeBatch, 16>, grid,
                   dim3(kQuantThreads), 0, st, 1, xv, d, slot_to_row, k, codes, scales, total);
}

cudaError_t launch_quant(bool fp4, const uint16_t* x, int T, int d, const int* slot_to_row, int k,
                         uint8_t* codes, uint8_t* scales, int layout, cudaStream_t st) {
  if (int64_t(T) * d == 0 || (slot_to_row && k == 0)) return cudaSuccess;
  if (layout == kScalesGroup32)
    return fp4 ? launch_quant_layout<true, kScalesGroup32>(x, T, d, slot_to_row, k, codes, scales, st)
               : launch_quant_layout<false, kScalesGroup32>(x, T, d, slot_to_row, k, codes, scales, st);
  return fp4 ? launch_quant_layout<true, kScalesTiled128>(x, T, d, slot_to_row, k, codes, scales, st)
             : launch_quant_layout<false, kScalesTiled128>(x, T, d, slot_to_row, k, codes, scales, st);
}

}  // namespace

cudaError_t launch_quant_mxfp8(const uint16_t* x, int T, int d, const int* slot_to_row, int k,
                               uint8_t* codes, uint8_t* scales, int layout, cudaStream_t st) {
  return launch_quant(false, x, T, d, slot_to_row, k, codes, scales, layout, st);
}

cudaError_t launch_quant_mxfp4(const uint16_t* x, int T, int d, const int* slot_to_row, int k,
                               uint8_t* codes, uint8_t* scales, int layout, cudaStream_t st) {
  return launch_quant(true, x, T, d, slot_to_row, k, codes, scales, layout, st);
}

cudaError_t launch_prepack_scales(const uint8_t* src, int64_t rows, int K, uint8_t* dst,
                                  cudaStream_t st) {
  const int64_t rows_p = (rows + 127) / 128 * 128;
  const int64_t words = rows_p * (K / 128);
  if (words == 0) return cudaSuccess;
  const int64_t blocks = (words + 255) / 256;
  prepack_scales_kernel<<<dim3(unsigned(blocks)), 256, 0, st>>>(src, rows, K, dst, words);
  return cudaGetLastError();
}

}  // namespace moe

namespace moe {

cudaError_t launch_prepack_weights(const uint8_t* src, int64_t rows, int K, uint8_t* dst,
                                   cudaStream_t st) {
  const int64_t chunks = rows * (K / 2) / 16;
  if (chunks == 0) return cudaSuccess;
  const int64_t blocks = (chunks + 255) / 256;
  prepack_weights_kernel<<<dim3(unsigned(blocks)), 256, 0, st>>>(
      reinterpret_cast<const uint4*>(src), K, reinterpret_cast<uint4*>(dst), chunks);
  return cudaGetLastError();
}

}  // namespace moe
