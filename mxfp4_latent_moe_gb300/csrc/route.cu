// Sigmoid top-k routing: one warp per token.
//
// "Kimi K3.1 Pro on AMD Instinct GPUs", "Kimi K3.1 Pro at a glance", Experts
// row: 896 routed experts, top-16, sigmoid routing. Selection is on the logits
// (sigmoid is monotone), logit descending with ties to the lower expert id;
// weights are sigmoid(l_j) / sum of the k selected sigmoids.
//
// Each lane holds the logits of experts lane, lane+32, ... (up to 32 per lane
// for E <= 1024) in registers and keeps its two best untaken ones. k rounds
// of a warp-wide (value desc, id asc) arg-max of the lanes' heads by
// butterfly shuffles pick the experts in output order. Reads are coalesced: a
// token's row is read once.
#include "internal.h"

namespace moe {

namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// The lane's best two values (by `better`) among those worse than (lv, li)
// when `limit`, else among all of its values; sentinels (-inf, INT_MAX) fill.
template <int NPL>
__device__ __forceinline__ void lane_top2(const float (&v)[NPL], int E, int lane, bool limit,
                                          float lv, int li, float& av, int& ai, float& bv,
                                          int& bi) {
  av = bv = -INFINITY;
  ai = bi = 0x7FFFFFFF;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E && (!limit || better(lv, li, v[i], e)) && better(v[i], e, bv, bi)) {
      if (better(v[i], e, av, ai)) {
        bv = av;
        bi = ai;
        av = v[i];
        ai = e;
      } else {
        bv = v[i];
        bi = e;
      }
    }
  }
}

template <int NPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                      int* __restrict__ ids, float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;  // warp-uniform
  const float* row = logits + int64_t(t) * E;
  float v[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldg(row + e) : -INFINITY;
  }
  // Each lane keeps its two best untaken values; a round is a warp arg-max of
  // the lanes' heads (value desc, id asc) and a pop on the winning lane. The
  // values a lane has given up are always its best ones, so once its two are
  // gone it rescans for the best two below its last pick.
  float av, bv;
  int ai, bi;
  lane_top2<NPL>(v, E, lane, false, 0.0f, 0, av, ai, bv, bi);
  float my_v = 0.0f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float wv = av;
    int wi = ai;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, wv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, wi, off);
      if (better(ov, oi, wv, wi)) {
        wv = ov;
        wi = oi;
      }
    }
    if ((wi & 31) == lane) {   // this lane's head won: pop it
      const float lv = av;
      const int li = ai;
      av = bv;
      ai = bi;
      bv = -INFINITY;
      bi = 0x7FFFFFFF;
      if (ai == 0x7FFFFFFF) lane_top2<NPL>(v, E, lane, true, lv, li, av, ai, bv, bi);
    }
    if (lane == j) {
      my_v = wv;
      my_id = wi;
    }
  }
  // sigmoid of the selected logits, renormalised over the k of them
  const float s = lane < k ? 1.0f / (1.0f + expf(-my_v)) : 0.0f;
  float sum = s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    ids[int64_t(t) * k + lane] = my_id;
    w[int64_t(t) * k + lane] = s / sum;
  }
}

template <int NPL>
cudaError_t launch_npl(const float* logits, int T, int E, int k, int* ids, float* w,
                       cudaStream_t st) {
  const dim3 grid((T + kWarpsPerBlock - 1) / kWarpsPerBlock);
  route_topk_kernel<NPL><<<grid, kWarpsPerBlock * 32, 0, st>>>(logits, T, E, k, ids, w);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int* ids, float* w,
                              cudaStream_t st) {
  if (T == 0 || k == 0) return cudaSuccess;
  const int npl = (E + 31) / 32;
  if (npl <= 1) return launch_npl<1>(logits, T, E, k, ids, w, st);
  if (npl <= 4) return launch_npl<4>(logits, T, E, k, ids, w, st);
  if (npl <= 8) return launch_npl<8>(logits, T, E, k, ids, w, st);
  if (npl <= 16) return launch_npl<16>(logits, T, E, k, ids, w, st);
  if (npl <= 28) return launch_npl<28>(logits, T, E, k, ids, w, st);
  return launch_npl<32>(logits, T, E, k, ids, w, st);
}

}  // namespace moe
