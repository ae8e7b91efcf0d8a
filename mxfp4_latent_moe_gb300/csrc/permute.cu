// Expert grouping: histogram, exclusive scan of padded counts, stable scatter.
//
// The grouped-MoE kernel ("The MXFP4 latent MoE on FlyDSL") works on rows
// grouped by expert. Rows of an expert follow ascending token order, so the
// result is unique and independent of scheduling and of atomic ordering.
//
// Tokens are cut into chunks of 256 (one per block, 8 warps of 32 tokens).
// Inside a chunk each warp builds, in shared memory, a 32-bit mask per expert
// with bit `lane` set when the lane's token picked that expert. A token picks
// an expert at most once, so a slot's rank among the chunk's slots of its
// expert is popc(mask of lower lanes in its warp) + popc(masks of lower warps).
//   1. permute_count:   per-chunk expert histograms hist[c][e]
//   2. permute_scan:    counts, padded offsets, chunk bases (exclusive over c)
//   3. permute_scatter: row = offsets[e] + base[c][e] + rank
// row_to_slot is set to -1 by a memset before the scatter fills the used rows.
// A batch of one chunk (T <= 256, decode) runs all of it in one block.
#include <mutex>

#include "internal.h"

namespace moe {

namespace {

constexpr int kChunk = 256;  // tokens per block
constexpr int kWarps = kChunk / 32;
constexpr int kIdBatch = 16;  // expert ids of a token loaded together

// Expert ids j0 .. j0 + 15 of token t (those below k): independent loads
// issued back to back, so a token pays one memory latency per 16 ids.
__device__ __forceinline__ void load_ids(const int* __restrict__ ids, int t, int k, int j0,
                                         int (&idv)[kIdBatch]) {
#pragma unroll
  for (int q = 0; q < kIdBatch; ++q)
    idv[q] = j0 + q < k ? __ldg(ids + int64_t(t) * k + j0 + q) : 0;
}

// Builds the per-warp expert masks of one chunk. An id out of range or
// repeated within a token records MOE_ERR_DEVICE_BAD_INPUT and is skipped
// (no write ever leaves the expert's own rows).
__device__ __forceinline__ void build_masks(const int* __restrict__ ids, int T, int E, int k,
                                           uint32_t* masks, int* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) masks[i] = 0u;
  pdl_wait();   // the ids come from the previous kernel
  __syncthreads();
  const int t = blockIdx.x * kChunk + threadIdx.x;
  if (t < T) {
    for (int j0 = 0; j0 < k; j0 += kIdBatch) {
      int idv[kIdBatch];
      load_ids(ids, t, k, j0, idv);
#pragma unroll
      for (int q = 0; q < kIdBatch; ++q) {
        if (j0 + q >= k) break;
        const int e = idv[q];
        if (e < 0 || e >= E) {
          set_status(status, MOE_ERR_DEVICE_BAD_INPUT);
          continue;
        }
        const uint32_t old = atomicOr(&masks[warp * E + e], 1u << lane);
        if (old & (1u << lane)) set_status(status, MOE_ERR_DEVICE_BAD_INPUT);
      }
    }
  }
  __syncthreads();
}

// Also sets this chunk's share of row_to_slot (ceil(rows / C) rows per
// block) to -1, after griddepcontrol.wait (inside build_masks): the scatter,
// two launches later, fills the used rows.
__global__ void __launch_bounds__(kChunk) permute_count_kernel(const int* __restrict__ ids,
                                                               int T, int E, int k,
                                                               int* __restrict__ hist,
                                                               int* status,
                                                               int* __restrict__ row_to_slot,
                                                               int64_t rows_capacity) {
  extern __shared__ uint32_t masks[];
  pdl_trigger();
  build_masks(ids, T, E, k, masks, status);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += __popc(masks[w * E + e]);
    hist[int64_t(blockIdx.x) * E + e] = s;
  }
  if (row_to_slot) {
    const int64_t per = (rows_capacity + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = min(rows_capacity, int64_t(blockIdx.x) * per);
    const int64_t r1 = min(rows_capacity, r0 + per);
    for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) row_to_slot[r] = -1;
  }
}

// One block of 1024 threads; E <= 1024.
__global__ void __launch_bounds__(1024) permute_scan_kernel(int* __restrict__ hist, int C, int E,
                                                            int pad_m, int* __restrict__ counts,
                                                            int* __restrict__ offsets) {
  __shared__ int warp_sums[32];
  pdl_trigger();
  pdl_wait();
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    // exclusive prefix over chunks, in place; 16 chunks' counts are loaded
    // before any of them is overwritten, so their loads are in flight
    // together instead of one memory latency per chunk
    constexpr int kBatch = 16;
    for (int c0 = 0; c0 < C; c0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        v[i] = c0 + i < C ? hist[int64_t(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (c0 + i < C) hist[int64_t(c0 + i) * E + e] = cnt;
        cnt += v[i];
      }
    }
    counts[e] = cnt;
  }
  const int padded = e < E ? (cnt + pad_m - 1) / pad_m * pad_m : 0;
  // block-wide exclusive scan of `padded`
  const int lane = e & 31, warp = e >> 5;
  int incl = padded;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, si, off);
      if (lane >= off) si += n;
    }
    warp_sums[lane] = si - s;  // exclusive over warps
  }
  __syncthreads();
  const int excl = incl - padded + warp_sums[warp];
  if (e < E) {
    offsets[e] = excl;
    if (e == E - 1) offsets[E] = excl + padded;
  }
}

__global__ void __launch_bounds__(kChunk) permute_scatter_kernel(
    const int* __restrict__ ids, int T, int E, int k, const int* __restrict__ hist,
    const int* __restrict__ offsets, int* __restrict__ slot_to_row, int* __restrict__ row_to_slot,
    int* status) {
  extern __shared__ uint32_t masks[];
  pdl_trigger();
  build_masks(ids, T, E, k, masks, status);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kChunk + threadIdx.x;
  if (t >= T) return;
  const uint32_t lower = (1u << lane) - 1u;
  for (int j0 = 0; j0 < k; j0 += kIdBatch) {
    int idv[kIdBatch];
    load_ids(ids, t, k, j0, idv);
#pragma unroll
    for (int q = 0; q < kIdBatch; ++q) {
      if (j0 + q >= k) break;
      const int e = idv[q];
      if (e < 0 || e >= E) continue;
      int rank = __popc(masks[warp * E + e] & lower);
      for (int w = 0; w < warp; ++w) rank += __popc(masks[w * E + e]);
      const int row = offsets[e] + hist[int64_t(blockIdx.x) * E + e] + rank;
      const int slot = t * k + j0 + q;
      slot_to_row[slot] = row;
      row_to_slot[row] = slot;
    }
  }
}

// Batches of one chunk (T <= 256, decode): histogram, scan and scatter in
// one block of 1024 threads, row_to_slot filled with -1 first (one launch
// instead of three and a memset). Only the launch itself overlaps the
// previous kernel; the fill runs after griddepcontrol.wait. Threads 0..255
// own the tokens (same masks and ranks as the three kernels above); all 1024
// share the fill, the mask clearing and the scan (one expert per thread,
// E <= 1024).
constexpr int kSingleThreads = 1024;

__global__ void __launch_bounds__(kSingleThreads)
    permute_single_kernel(const int* __restrict__ ids, int T, int E, int k, int pad_m,
                          int* __restrict__ counts, int* __restrict__ offsets,
                          int* __restrict__ slot_to_row, int* __restrict__ row_to_slot,
                          int64_t rows_capacity, int* status) {
  extern __shared__ uint32_t masks[];            // [kWarps][E], then offsets [E+1]
  int* off_s = reinterpret_cast<int*>(masks + kWarps * E);
  __shared__ int warp_sums[kSingleThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();
  // Everything below waits for the previous kernel in the stream: a library
  // kernel launched before this one may still read or write row_to_slot
  // (another grouping call on the same buffers, or a kernel still using
  // memory the caller has since handed over as row_to_slot).
  pdl_wait();
  {
    int64_t done = 0;
    if ((reinterpret_cast<uintptr_t>(row_to_slot) & 15u) == 0) {
      int4* r4 = reinterpret_cast<int4*>(row_to_slot);
      for (int64_t i = tid; i < rows_capacity / 4; i += kSingleThreads)
        r4[i] = make_int4(-1, -1, -1, -1);
      done = (rows_capacity / 4) * 4;
    }
    for (int64_t i = done + tid; i < rows_capacity; i += kSingleThreads) row_to_slot[i] = -1;
  }
  build_masks(ids, T, E, k, masks, status);      // ends with __syncthreads
  // expert tid: count, padded size, block-wide exclusive scan
  const int e = tid;
  int cnt = 0;
  if (e < E)
#pragma unroll
    for (int w = 0; w < kWarps; ++w) cnt += __popc(masks[w * E + e]);
  const int padded = e < E ? (cnt + pad_m - 1) / pad_m * pad_m : 0;
  int incl = padded;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, si, off);
      if (lane >= off) si += n;
    }
    warp_sums[lane] = si - s;  // exclusive over warps
  }
  __syncthreads();
  if (e < E) {
    const int base = incl - padded + warp_sums[warp];
    counts[e] = cnt;
    offsets[e] = base;
    off_s[e] = base;
    if (e == E - 1) {
      offsets[E] = base + padded;
      off_s[E] = base + padded;
    }
  }
  __syncthreads();
  const int t = tid;
  if (t >= T) return;
  const uint32_t lower = (1u << lane) - 1u;
  for (int j0 = 0; j0 < k; j0 += kIdBatch) {
    int idv[kIdBatch];
    load_ids(ids, t, k, j0, idv);
#pragma unroll
    for (int q = 0; q < kIdBatch; ++q) {
      if (j0 + q >= k) break;
      const int ex = idv[q];
      if (ex < 0 || ex >= E) continue;
      int rank = __popc(masks[warp * E + ex] & lower);
      for (int w = 0; w < warp; ++w) rank += __popc(masks[w * E + ex]);
      const int row = off_s[ex] + rank;
      const int slot = t * k + j0 + q;
      slot_to_row[slot] = row;
      row_to_slot[row] = slot;
    }
  }
}

}  // namespace

size_t permute_scratch_bytes(int T, int E) {
  const size_t C = size_t((T + kChunk - 1) / kChunk);
  return C * size_t(E) * sizeof(int);
}

cudaError_t launch_permute(const int* ids, int T, int E, int k, int pad_m, int* counts,
                           int* offsets, int* slot_to_row, int* row_to_slot,
                           int64_t rows_capacity, int* hist, int* status, cudaStream_t st) {
  const int C = (T + kChunk - 1) / kChunk;
  const size_t smem = size_t(kWarps) * E * sizeof(uint32_t);
  if (C == 1 && row_to_slot) {   // one chunk: a single launch
    return launch_ex(true, permute_single_kernel, dim3(1), dim3(kSingleThreads),
                      smem + size_t(E + 1) * sizeof(int), st, 1, ids, T, E, k, pad_m, counts,
                      offsets, slot_to_row, row_to_slot, rows_capacity, status);
  }
  // Count, scan and scatter chain by programmatic dependent launch: each
  // touches global memory only after griddepcontrol.wait, and the count
  // kernel also resets row_to_slot.
  const bool work = C > 0 && k > 0;
  if (work) {
    const cudaError_t err = launch_ex(true, permute_count_kernel, dim3(C), dim3(kChunk), smem,
                                      st, 1, ids, T, E, k, hist, status, row_to_slot,
                                      rows_capacity);
    if (err != cudaSuccess) return err;
  }
  cudaError_t err = launch_ex(work, permute_scan_kernel, dim3(1), dim3(1024), 0, st, 1, hist,
                              work ? C : 0, E, pad_m, counts, offsets);
  if (err != cudaSuccess) return err;
  if (!work && rows_capacity > 0 && row_to_slot) {   // no count kernel to reset it
    err = cudaMemsetAsync(row_to_slot, 0xFF, size_t(rows_capacity) * sizeof(int), st);
    if (err != cudaSuccess) return err;
  }
  if (work)
    err = launch_ex(true, permute_scatter_kernel, dim3(C), dim3(kChunk), smem, st, 1, ids, T, E,
                    k, hist, offsets, slot_to_row, row_to_slot, status);
  return err;
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free grouping (moe_permute_noalloc).
//
// moe_permute keeps its per-chunk expert histograms in a workspace the caller
// allocates. Some callers cannot do that: a host framework that owns every
// byte of device memory through its own pool and forbids libraries to
// allocate, or a latency-critical caller that must not call cudaMalloc on its
// serving path because cudaMalloc may synchronise the whole device. For them
// the histograms live in the fixed device array below, part of this library's
// image: every GPU that loads the library holds its 1 MiB until the process
// exits. Its device address is looked up once per device (the first call on
// that device, with that device current) and cached for the life of the
// process, keyed by device ordinal: callers that reset a device
// (cudaDeviceReset) or drive it through a non-primary context are not
// supported by this entry point.
// ---------------------------------------------------------------------------
namespace moe {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // histograms of ceil(T/256) x E ints
static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device, or nullptr.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

bool is_aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const int32_t* topk_ids, int32_t T, int32_t E, int32_t k,
                                          int32_t pad_m, int32_t* counts, int32_t* offsets,
                                          int32_t* slot_to_row, int32_t* row_to_slot,
                                          int64_t rows_capacity, int32_t* status,
                                          cudaStream_t stream) {
  if (rows_capacity < 0) return MOE_ERR_INVALID_ARGUMENT;
  const moe_status shape = moe::check_routing_shape(T, E, k);   // the rules of moe_permute
  if (shape != MOE_OK) return shape;
  if (!moe::pow2_in(pad_m, 1, 1024)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || !moe::is_aligned4(counts) || !moe::is_aligned4(offsets))
    return MOE_ERR_INVALID_ARGUMENT;
  const bool any = T > 0 && k > 0;
  if (any && (!topk_ids || !slot_to_row || !row_to_slot || !moe::is_aligned4(topk_ids) ||
              !moe::is_aligned4(slot_to_row) || !moe::is_aligned4(row_to_slot)))
    return MOE_ERR_INVALID_ARGUMENT;
  if (status && !moe::is_aligned4(status)) return MOE_ERR_INVALID_ARGUMENT;
  const int64_t slots = int64_t(T) * k;
  if (rows_capacity < slots + (slots < E ? slots : int64_t(E)) * (pad_m - 1))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (moe::permute_scratch_bytes(T, E) > moe::kNoAllocScratchBytes)
    return MOE_ERR_WORKSPACE_TOO_SMALL;  // more token chunks x experts than the fixed array holds
  void* scratch = moe::scratch_on_current_device();
  if (!scratch) return MOE_ERR_CUDA;
  const cudaError_t e =
      moe::launch_permute(topk_ids, T, E, k, pad_m, counts, offsets, slot_to_row, row_to_slot,
                          rows_capacity, static_cast<int*>(scratch), status, stream);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
