// The composed latent-MoE block: the routed MXFP4 experts between the BF16
// latent projections, with the router and the shared experts beside them.
//
// "Kimi K3.1 Pro on AMD Instinct GPUs", "Kimi K3.1 Pro at a glance": 896
// routed experts (top-16, sigmoid routing) plus two shared experts; the routed
// experts work in a 3,584-wide latent, half the 7,168-wide hidden size; the
// shared experts, the latent up/down projections and the router are BF16.
// Same page, "The MXFP4 latent MoE on FlyDSL": the two shared experts run on
// a second stream, concurrently with the routed experts. "Day 0 Kimi-K3
// Inference Deployment with ATOM on AMD Instinct MI355X GPUs", "Kimi-K3
// Architecture and Weights": Stable LatentMoE projects the 7,168-wide hidden
// state down to 3,584 before the expert computation.
//
// For hidden states h [T][hidden]:
//   main stream:  x      = bf16(h . Wdown^T)            [T][d]      (latent down)
//                 logits = h . Wrouter^T (fp32)          [T][E]
//                 y_lat  = the routed layer on (x, logits) [T][d]   (moe_forward)
//   side stream:  hs     = bf16(silu(h . G^T) * (h . U^T)) [T][Is]  (both shared
//                          experts as one gated MLP: their intermediate widths
//                          side by side, Is = 2 x 3,072)
//   joined:       out    = bf16([y_lat | hs] . Wout^T)  [T][hidden]
// where Wout = [Wup | Wsd]: the latent up projection and the shared experts'
// down projections side by side along the input dimension, so one GEMM adds
// the routed and the shared contributions in fp32 before a single rounding.
// The sum of two gated MLPs equals one gated MLP over their concatenated
// intermediate rows, which is how the shared experts are stored here.
#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

struct ForkJoin {
  cudaEvent_t fork = nullptr;
  cudaEvent_t join = nullptr;
};
// Per host thread and device: concurrent calls from different threads never
// share an event.
thread_local ForkJoin t_events[kMaxDevices];

ForkJoin* events_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  ForkJoin& e = t_events[dev];
  if (!e.fork && cudaEventCreateWithFlags(&e.fork, cudaEventDisableTiming) != cudaSuccess)
    return nullptr;
  if (!e.join && cudaEventCreateWithFlags(&e.join, cudaEventDisableTiming) != cudaSuccess)
    return nullptr;
  return &e;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
template <class T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}

struct BlockLayout {
  size_t status, x, logits, ylat, hs, main_part, side_part, layer, layer_bytes, total;
};

moe_dims layer_dims(const moe_block_dims& B) { return moe_dims{B.T, B.d, B.E, B.k, B.I}; }

BlockLayout block_layout(const moe_block_dims& B, size_t layer_bytes) {
  BlockLayout L{};
  const size_t T = size_t(B.T);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += round_up(bytes, 256);
    return o;
  };
  size_t main_part = moe::bf16_partial_bytes(B.T, B.d, B.hidden, moe::kEpiBf16);
  const size_t router_part = moe::bf16_partial_bytes(B.T, B.E, B.hidden, moe::kEpiF32);
  const size_t out_part =
      moe::bf16_partial_bytes(B.T, B.hidden, B.d + B.shared_I, moe::kEpiBf16);
  main_part = main_part > router_part ? main_part : router_part;
  main_part = main_part > out_part ? main_part : out_part;
  L.status = take(MOE_STATUS_BYTES);
  L.x = take(T * size_t(B.d) * 2);
  L.logits = take(T * size_t(B.E) * 4);
  L.ylat = take(T * size_t(B.d) * 2);
  L.hs = take(T * size_t(B.shared_I) * 2);
  // each GEMM workspace: a status word (unused: kernels report to the block's) + partials
  L.main_part = take(MOE_STATUS_BYTES + main_part);
  L.side_part =
      take(MOE_STATUS_BYTES + moe::bf16_partial_bytes(B.T, 2 * B.shared_I, B.hidden,
                                                      moe::kEpiSwiglu));
  L.layer = take(layer_bytes);
  L.layer_bytes = layer_bytes;
  L.total = off;
  return L;
}

moe_status check_block_dims(const moe_block_dims* B, size_t* layer_bytes) {
  if (!B) return MOE_ERR_INVALID_ARGUMENT;
  if (B->hidden < 0 || B->shared_I < 0) return MOE_ERR_INVALID_ARGUMENT;
  const moe_dims D = layer_dims(*B);
  const moe_status s = moe_workspace_size(&D, layer_bytes);   // T, d, E, k, I rules
  if (s != MOE_OK) return s;
  // BF16 GEMMs: K % 64 (hidden, and d + shared_I as the output GEMM's K);
  // N % 8 (d, E, hidden); the shared experts' SwiGLU: 2*shared_I % 256
  if (B->hidden < 64 || B->hidden % 64 != 0 || B->hidden > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  if (B->E % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (B->shared_I < 128 || B->shared_I % 128 != 0 || B->shared_I > (1 << 20))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_block_workspace_size(const moe_block_dims* dims, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARGUMENT;
  size_t layer_bytes = 0;
  const moe_status s = check_block_dims(dims, &layer_bytes);
  if (s != MOE_OK) return s;
  *bytes = block_layout(*dims, layer_bytes).total;
  return MOE_OK;
}

moe_status moe_block_forward(const moe_block_dims* dims, int32_t kernel, const uint16_t* h,
                             const moe_block_weights* W, uint16_t* out, void* ws, size_t ws_bytes,
                             cudaStream_t stream, cudaStream_t shared_stream) {
  size_t layer_bytes = 0;
  moe_status s = check_block_dims(dims, &layer_bytes);
  if (s != MOE_OK) return s;
  const moe_block_dims B = *dims;
  if (B.T == 0) return MOE_OK;
  if (!h || !W || !out || !ws || !W->w_down || !W->w_router || !W->w_shared13 || !W->w_out)
    return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(h, 16) || !aligned(out, 16) || !aligned(ws, 256) || !aligned(W->w_down, 16) ||
      !aligned(W->w_router, 16) || !aligned(W->w_shared13, 16) || !aligned(W->w_out, 16))
    return MOE_ERR_INVALID_ARGUMENT;
  const BlockLayout L = block_layout(B, layer_bytes);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const bool two_streams = shared_stream != stream;
  ForkJoin* ev = nullptr;
  if (two_streams && !(ev = events_on_current_device())) return MOE_ERR_CUDA;

  int* status = at<int>(ws, L.status);
  uint16_t* x = at<uint16_t>(ws, L.x);
  float* logits = at<float>(ws, L.logits);
  uint16_t* ylat = at<uint16_t>(ws, L.ylat);
  uint16_t* hs = at<uint16_t>(ws, L.hs);
  float* main_part = at<float>(ws, L.main_part + MOE_STATUS_BYTES);
  float* side_part = at<float>(ws, L.side_part + MOE_STATUS_BYTES);
  const cudaStream_t side = two_streams ? shared_stream : stream;

  if (cudaMemsetAsync(status, 0, sizeof(int), stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (two_streams) {   // the side stream starts after h is ready and the status is cleared
    if (cudaEventRecord(ev->fork, stream) != cudaSuccess ||
        cudaStreamWaitEvent(side, ev->fork, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  // shared experts (side stream): both as one gated MLP, h -> hs
  if (moe::launch_gemm_bf16(h, W->w_shared13, B.T, 2 * B.shared_I, B.hidden, moe::kEpiSwiglu,
                            hs, side_part, status, side) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (two_streams && cudaEventRecord(ev->join, side) != cudaSuccess) return MOE_ERR_CUDA;
  // latent down projection and router (main stream)
  if (moe::launch_gemm_bf16(h, W->w_down, B.T, B.d, B.hidden, moe::kEpiBf16, x, main_part, status,
                            stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_gemm_bf16(h, W->w_router, B.T, B.E, B.hidden, moe::kEpiF32, logits, main_part,
                            status, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  // routed experts in the latent (main stream)
  const moe_dims D = layer_dims(B);
  s = moe::forward_with_status(false, &D, kernel, x, logits, &W->routed, ylat,
                               at<void>(ws, L.layer), L.layer_bytes, status, stream);
  if (s != MOE_OK) return s;
  // join, then the latent up projection plus the shared experts' down projection
  if (two_streams && cudaStreamWaitEvent(stream, ev->join, 0) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_gemm_bf16_cat(ylat, B.d, hs, B.shared_I, W->w_out, B.T, B.hidden,
                                moe::kEpiBf16, out, main_part, status, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // extern "C"
