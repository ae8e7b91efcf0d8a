// Routing-weighted combine: y[t] = bf16_rne(sum_j w[t][j] * Yp[slot_to_row[t*k+j]]).
//
// The layer ends with the weighted sum of the token's k expert outputs (the
// routed-MoE layer of "Kimi K3.1 Pro at a glance"). One thread per 8 outputs
// of a token: k 16-byte loads of grouped rows (issued 16 at a time), fp32
// fused multiply-adds in j order, one 16-byte bf16 store. Every byte of y is written once, every
// row of Yp is read once.
#include "internal.h"

namespace moe {

namespace {

constexpr int kCombineThreads = 256;
// Small batches (decode: one wave of threads, each waiting on its loads)
// issue all 16 terms' loads together; large batches keep occupancy instead.
constexpr int kSmallBatchThreads = 152 * 2048;
constexpr int kLargeBatch = 4;

template <int kBatch>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const uint4* __restrict__ yp, const int* __restrict__ slot_to_row,
                   const float* __restrict__ w, int k, int d, uint4* __restrict__ y,
                   int64_t total_vec) {
  pdl_trigger();
  pdl_wait();
  const int64_t g = int64_t(blockIdx.x) * kCombineThreads + threadIdx.x;
  if (g >= total_vec) return;
  const int vpr = d >> 3;
  const int64_t t = g / vpr;
  const int v = int(g - t * vpr);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  // kBatch terms at a time: their row indices, then their row loads, are
  // issued back to back (two memory latencies per batch, not two per term);
  // the sums still run in j order.
  for (int j0 = 0; j0 < k; j0 += kBatch) {
    int row[kBatch];
    float wj[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      row[q] = j0 + q < k ? __ldg(slot_to_row + t * k + j0 + q) : 0;
      wj[q] = j0 + q < k ? __ldg(w + t * k + j0 + q) : 0.0f;
    }
    uint4 val[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q)
      val[q] = j0 + q < k ? __ldcs(yp + int64_t(row[q]) * vpr + v) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      if (j0 + q >= k) break;
      const uint32_t q4[4] = {val[q].x, val[q].y, val[q].z, val[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(wj[q], __uint_as_float(q4[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(wj[q], __uint_as_float(q4[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    o[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  y[g] = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

cudaError_t launch_combine(const uint16_t* yp, const int* slot_to_row, const float* w, int T,
                           int k, int d, uint16_t* y, cudaStream_t st) {
  const int64_t total = int64_t(T) * (d / 8);
  if (total == 0) return cudaSuccess;
  const int64_t blocks = (total + kCombineThreads - 1) / kCombineThreads;
  const dim3 grid(static_cast<unsigned>(blocks));
  const uint4* ypv = reinterpret_cast<const uint4*>(yp);
  uint4* yv = reinterpret_cast<uint4*>(y);
  if (total <= kSmallBatchThreads)   // decode-sized
    return launch_ex(true, combine_kernel<16>, grid, dim3(kCombineThreads), 0, st, 1, ypv,
                     slot_to_row, w, k, d, yv, total);
  return launch_ex(false, combine_kernel<kLargeBatch>, grid, dim3(kCombineThreads), 0, st, 1, ypv,
                   slot_to_row, w, k, d, yv, total);
}

}  // namespace moe
