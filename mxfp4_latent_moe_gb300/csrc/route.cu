// Sigmoid top-k routing: one warp per token.
//
// "Kimi K3.1 Pro on AMD Instinct GPUs", "Kimi K3.1 Pro at a glance", Experts
// row: 896 routed experts, top-16, sigmoid routing. Selection is on the logits
// (sigmoid is monotone), logit descending with ties to the lower expert id;
// weights are sigmoid(l_j) / sum of the k selected sigmoids.
//
// Each lane holds the logits of experts lane, lane+32, ... (up to 32 per lane
// for E <= 1024) as 64-bit keys that order like (value desc, id asc): the
// high word maps the float monotonically onto unsigned integers (-0 joins +0),
// the low word is ~id, so all keys of a token differ. Reads are coalesced: a
// token's row is read once.
//
// Fast path: t0 = the k-th largest of the 32 lane maxima. At least k keys are
// >= t0 (the k lanes whose maximum is), so every one of the token's k largest
// keys is >= t0; when at most 32 keys are, they are gathered one per lane and
// sorted across the warp (bitonic network, 15 exchange steps), and lanes
// 0..k-1 hold the picks in order. For N(0,1) logits at E = 896, k = 16 about
// 22 keys pass on average and more than 32 for about 0.1% of tokens.
// Otherwise (the general path): a lane keeps its two best untaken keys
// (branch-free max/min updates); each of the k rounds takes the warp's best
// head with two warp reductions (max of the high words, then max of the low
// words among the lanes that hold it), and the owning lane pops it. Both paths
// give the same, exact result.
#include "internal.h"

namespace moe {

namespace {

constexpr int kWarpsPerBlock = 8;

// Monotone map of a float onto uint32 (a < b <=> key(a) < key(b); -0 and +0
// share a key) and its inverse (which returns +0 for both zeros).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// (value, id) -> 64-bit key; larger is better. 0 is below every real key.
__device__ __forceinline__ uint64_t route_key(float v, int e) {
  return (uint64_t(order_key(v)) << 32) | uint64_t(0xFFFFFFFFu - uint32_t(e));
}

// The lane's best two keys (a > b) among those below `limit` (all when limit
// is ~0); 0 fills a missing one.
template <int NPL>
__device__ __forceinline__ void lane_top2(const uint64_t (&key)[NPL], uint64_t limit, uint64_t& a,
                                          uint64_t& b) {
  a = b = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const uint64_t x = key[i] < limit ? key[i] : 0;
    const uint64_t lo = a < x ? a : x;
    a = a < x ? x : a;
    b = b < lo ? lo : b;
  }
}

// Descending sort of one key per lane across the warp (lane 0 the largest).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

template <int NPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                      int* __restrict__ ids, float* __restrict__ w) {
  __shared__ uint64_t cand[kWarpsPerBlock * 32];   // fast-path candidates, 32 per warp
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;  // warp-uniform
  const float* row = logits + int64_t(t) * E;
  uint64_t key[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? route_key(__ldg(row + e), e) : 0;
  }
  uint32_t my_hi = 0, my_lo = 0;
  // fast path: the keys >= t0, one per lane, sorted across the warp
  uint64_t mx = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) mx = key[i] > mx ? key[i] : mx;
  const uint64_t t0 = __shfl_sync(0xffffffffu, warp_sort_desc(mx, lane), k - 1);
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) cnt += key[i] >= t0 ? 1 : 0;
  int incl = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (total <= 32) {   // warp-uniform
    uint64_t* slots = cand + (threadIdx.x >> 5) * 32;
    int pos = incl - cnt;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (key[i] >= t0) slots[pos++] = key[i];
    __syncwarp();
    const uint64_t c = warp_sort_desc(lane < total ? slots[lane] : 0, lane);
    my_hi = uint32_t(c >> 32);
    my_lo = uint32_t(c);
  } else {
    // A lane gives up its keys in descending order, so once its two are
    // taken it rescans for the best two below the last one it gave up.
    uint64_t a, b;
    lane_top2<NPL>(key, ~uint64_t(0), a, b);
    for (int j = 0; j < k; ++j) {
      const uint32_t hi = uint32_t(a >> 32), lo = uint32_t(a);
      const uint32_t m_hi = __reduce_max_sync(0xffffffffu, hi);
      const uint32_t m_lo = __reduce_max_sync(0xffffffffu, hi == m_hi ? lo : 0u);
      const int id = int(0xFFFFFFFFu - m_lo);
      if ((id & 31) == lane) {   // this lane's head won: pop it
        const uint64_t taken = a;
        a = b;
        b = 0;
        if (a == 0) lane_top2<NPL>(key, taken, a, b);
      }
      if (lane == j) {
        my_hi = m_hi;
        my_lo = m_lo;
      }
    }
  }
  // sigmoid of the selected logits, renormalised over the k of them
  const float s = lane < k ? 1.0f / (1.0f + expf(-key_value(my_hi))) : 0.0f;
  float sum = s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    ids[int64_t(t) * k + lane] = int(0xFFFFFFFFu - my_lo);
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
