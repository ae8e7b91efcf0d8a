// Dense BF16 GEMMs of the steps next to the routed experts: the router GEMM
// that produces the logits, the latent down/up projections (7,168 <-> 3,584)
// and the two shared experts, all BF16 in the pages' layer ("Kimi K3.1 Pro at
// a glance" and "The MXFP4 latent MoE on FlyDSL" of "Kimi K3.1 Pro on AMD
// Instinct GPUs").
//
//   C[M][N] = A[M][K] . B[N][K]^T, bf16 operands, fp32 accumulation in
//   tensor memory (tcgen05.mma kind::f16, 4 MMAs of K = 16 per 64-input stage)
//   epilogue kEpiF32:    C in fp32 (router logits)
//   epilogue kEpiBf16:   C rounded to bf16 (projections, shared-expert down)
//   epilogue kEpiSwiglu: B holds N/2 gate rows then N/2 up rows; a tile pairs
//                        128 gate rows with the matching 128 up rows and
//                        writes h[M][N/2] = bf16(silu(g) * u)
//
// CTA organisation as the grouped GEMMs (persistent, one CTA per SM, 320
// threads): warp 0 TMA producer, warp 1 tensor-memory allocator + MMA issuer
// (both converged, one elected lane issues), warps 2-9 epilogue. Without
// scale factors the 512 tensor-memory columns hold two 256-column
// accumulators, so the next tile's MMAs never wait for the epilogue. Tiles
// run in groups of 8 row tiles with the row tile fastest, so the CTAs in
// flight share B tiles and keep a bounded slice of A in L2. Rows of A and B
// past M and N are zero-filled by TMA; stores past M and N are skipped.
// A may come in two parts along K, A = [A1 | A2] (A1 [M][K1], A2 [M][K2],
// two tensor maps): the composed block's output GEMM reads the routed
// experts' latent output and the shared experts' h side by side this way.
// Calls with too few tiles to cover the GPU (decode: one row tile) split K:
// each CTA accumulates one K-slice of a tile and writes its fp32 partial sums
// to the workspace; a second kernel adds the slices in a fixed order and
// applies the epilogue, so results do not depend on the split. Both kernels
// use programmatic dependent launch, so the reduction's launch and the next
// GEMM's set-up overlap the running kernel.
// Every wait is bounded (MOE_ERR_DEVICE_TIMEOUT in the status word).
#include "internal.h"

namespace moe {

namespace {

constexpr int BM = 128;            // rows of A per tile (MMA M)
constexpr int BN = 256;            // rows of B per tile (MMA N)
constexpr int BKB = 64;            // inputs per stage: 64 bf16 = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int GM = 8;              // row tiles per raster group
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t A_BYTES = BM * BKB * 2;
constexpr uint32_t B_BYTES = BN * BKB * 2;
constexpr uint32_t kStageTx = A_BYTES + B_BYTES;   // zero-filled box rows count too

constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + STAGES * A_BYTES;
constexpr uint32_t kOffBars = kOffB + STAGES * B_BYTES;
// full[S], empty[S], acc_full[2], acc_empty[2], drain
constexpr uint32_t kNumBars = 2 * STAGES + 5;
constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), A and B bf16 (bits 7-9, 10-12 = 1), both K-major, dense, M x N.
constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct Bf16Params {
  int64_t M;
  int N;          // rows of B
  int K;
  int K1T;        // stages whose A columns come from the first A map (the rest: the second)
  int MT, NT;     // row tiles of A; column tiles of C (EPI kEpiSwiglu: of h)
  int KS;         // K-slices per tile (1: no split)
  int KTS;        // 64-input stages per slice
  void* c;
  float* partial; // KS > 1: fp32 [KS][M][N] partial sums
  int* status;
};

// tile -> (row tile, column tile) in the grouped raster.
__device__ __forceinline__ void bf16_tile(int tile, int MT, int NT, int& mt, int& nt) {
  const int group = tile / (GM * NT);
  const int first = group * GM;
  const int gm = min(GM, MT - first);
  const int r = tile - group * GM * NT;
  nt = r / gm;
  mt = first + (r - nt * gm);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmap_a,
                     const __grid_constant__ CUtensorMap tmap_a2,
                     const __grid_constant__ CUtensorMap tmap_b, const Bf16Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;    // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = p.KTS;
  const int total = p.MT * p.NT * p.KS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);   // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  pdl_trigger();
  pdl_wait();   // the operands (and the partial-sum buffer) belong to earlier kernels
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const bool leader = elect_one_sync();
    uint32_t stage = 0, phase = 0;
    uint32_t filled = 0, last_parity = 0;
    bool failed = false;
    for (int work = blockIdx.x; work < total && !failed; work += gridDim.x) {
      int mt, nt;
      bf16_tile(work / p.KS, p.MT, p.NT, mt, nt);
      const int k0 = (work % p.KS) * KT;   // first stage of this K-slice
      for (int kt = k0; kt < k0 + KT; ++kt) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag)) {
          failed = true;
          break;
        }
        if (leader) {
          uint8_t* sa = smem + kOffA + stage * A_BYTES;
          uint8_t* sb = smem + kOffB + stage * B_BYTES;
          mbar_arrive_expect_tx(&full[stage], kStageTx);
          // A = [A1 | A2] along K: stages below K1T read A1, the rest A2
          if (kt < p.K1T) tma_load_2d(sa, &tmap_a, &full[stage], kt * BKB, mt * BM);
          else tma_load_2d(sa, &tmap_a2, &full[stage], (kt - p.K1T) * BKB, mt * BM);
          if (EPI == kEpiSwiglu) {   // 128 gate rows, then the matching 128 up rows
            tma_load_2d(sb, &tmap_b, &full[stage], kt * BKB, nt * 128);
            tma_load_2d(sb + B_BYTES / 2, &tmap_b, &full[stage], kt * BKB,
                        (p.N >> 1) + nt * 128);
          } else {
            tma_load_2d(sb, &tmap_b, &full[stage], kt * BKB, nt * BN);
          }
        }
        __syncwarp();
        filled |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (failed && leader) {
      *abort_flag = 1;
      set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
    }
    for (int s = 0; s < STAGES; ++s)
      if ((filled >> s) & 1u)
        if (!mbar_wait_warp(&full[s], (last_parity >> s) & 1u, nullptr) && leader)
          set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    const bool leader = elect_one_sync();
    constexpr uint32_t idesc = idesc_bf16(BM, BN);
    uint32_t stage = 0, phase = 0, acc_phases = 0;
    int buf = 0;
    bool failed = false;
    for (int work = blockIdx.x; work < total && !failed; work += gridDim.x) {
      if (!mbar_wait_warp(&acc_empty[buf], ((acc_phases >> buf) & 1u) ^ 1u, abort_flag)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem_base + uint32_t(buf) * BN;
      for (int kt = 0; kt < KT; ++kt) {
        if (!mbar_wait_warp(&full[stage], phase, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after();
        if (leader) {
          const uint64_t adesc = desc_sw128_kmajor(smem_u32(smem + kOffA + stage * A_BYTES));
          const uint64_t bdesc = desc_sw128_kmajor(smem_u32(smem + kOffB + stage * B_BYTES));
#pragma unroll
          for (int kk = 0; kk < BKB / 16; ++kk)   // 16 bf16 = 32 bytes = +2 in the address
            tc_mma_bf16(acc, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk), idesc,
                        (kt > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (failed) break;
      if (leader) tc_commit(&acc_full[buf]);
      __syncwarp();
      acc_phases ^= 1u << buf;
      buf ^= 1;
    }
    if (failed && leader) {
      *abort_flag = 1;
      set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
    }
    if (leader) tc_commit(drain);
    __syncwarp();
    if (!mbar_wait_warp(drain, 0, nullptr) && leader) set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
  } else {
    // ------------------------------------------------------------ epilogue
    // Two warps per tensor-memory lane quarter (warp % 4), splitting the
    // tile's columns in halves; each copies its 32 rows x 128 columns to
    // registers, releases the accumulator, then converts and stores.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint32_t acc_phases = 0;
    int buf = 0;
    for (int work = blockIdx.x; work < total; work += gridDim.x) {
      int mt, nt;
      bf16_tile(work / p.KS, p.MT, p.NT, mt, nt);
      const int ks = work % p.KS;
      bool ok = mbar_wait(&acc_full[buf], (acc_phases >> buf) & 1u, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tq = tmem_base + uint32_t(buf) * BN + (uint32_t(q * 32) << 16);
      uint32_t v[4][32];
      if (EPI == kEpiSwiglu) {   // gate columns [64 half, +64) and their up columns (+128)
        tmem_ld_32x32b_x32(tq + 64 * half, v[0]);
        tmem_ld_32x32b_x32(tq + 64 * half + 32, v[1]);
        tmem_ld_32x32b_x32(tq + 128 + 64 * half, v[2]);
        tmem_ld_32x32b_x32(tq + 128 + 64 * half + 32, v[3]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tq + 128 * half + 32 * c, v[c]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
      acc_phases ^= 1u << buf;
      buf ^= 1;
      const int64_t row = int64_t(mt) * BM + q * 32 + lane;
      if (row >= p.M) continue;
      if (p.KS > 1) {   // raw fp32 sums of this K-slice, in C's column order over all N rows of B
        float* dst = p.partial + (int64_t(ks) * p.M + row) * p.N;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          // columns of v[c]: swiglu gate (c < 2) / up (c >= 2) halves, else 128 half + 32 c
          const int colc = EPI == kEpiSwiglu
                               ? (c < 2 ? nt * 128 + 64 * half + 32 * c
                                        : (p.N >> 1) + nt * 128 + 64 * half + 32 * (c - 2))
                               : nt * BN + 128 * half + 32 * c;
#pragma unroll
          for (int w = 0; w < 8; ++w)
            if (colc + 4 * w < p.N)
              reinterpret_cast<uint4*>(dst + colc)[w] =
                  make_uint4(v[c][4 * w], v[c][4 * w + 1], v[c][4 * w + 2], v[c][4 * w + 3]);
        }
        continue;
      }
      if (EPI == kEpiSwiglu) {
        const int Nh = p.N >> 1;
        uint16_t* dst = static_cast<uint16_t*>(p.c) + row * Nh + int64_t(nt) * 128 + 64 * half;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float h2[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const float gf = __uint_as_float(v[c][2 * i + j]);
              const float uf = __uint_as_float(v[2 + c][2 * i + j]);
              h2[j] = __fdividef(gf * uf, 1.0f + __expf(-gf));   // silu(g) * u
            }
            o[i] = pack_bf16x2(h2[0], h2[1]);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int w = 0; w < 4; ++w) d4[w] = make_uint4(o[4 * w], o[4 * w + 1], o[4 * w + 2], o[4 * w + 3]);
        }
      } else {
        const int col0 = nt * BN + 128 * half;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int colc = col0 + 32 * c;
          if (EPI == kEpiF32) {
            float* dst = static_cast<float*>(p.c) + row * p.N + colc;
#pragma unroll
            for (int w = 0; w < 8; ++w)
              if (colc + 4 * w < p.N)   // N % 8 == 0: a float4 is all in or all out
                reinterpret_cast<uint4*>(dst)[w] =
                    make_uint4(v[c][4 * w], v[c][4 * w + 1], v[c][4 * w + 2], v[c][4 * w + 3]);
          } else {
            uint16_t* dst = static_cast<uint16_t*>(p.c) + row * p.N + colc;
#pragma unroll
            for (int w = 0; w < 4; ++w)
              if (colc + 8 * w < p.N)   // N % 8 == 0: 8 bf16 are all in or all out
                reinterpret_cast<uint4*>(dst)[w] = make_uint4(
                    pack_bf16x2(__uint_as_float(v[c][8 * w]), __uint_as_float(v[c][8 * w + 1])),
                    pack_bf16x2(__uint_as_float(v[c][8 * w + 2]), __uint_as_float(v[c][8 * w + 3])),
                    pack_bf16x2(__uint_as_float(v[c][8 * w + 4]), __uint_as_float(v[c][8 * w + 5])),
                    pack_bf16x2(__uint_as_float(v[c][8 * w + 6]), __uint_as_float(v[c][8 * w + 7])));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// Sum of the K-slices in slice order, then the epilogue; thread = 4 outputs.
template <int EPI>
__global__ void __launch_bounds__(256)
    bf16_splitk_reduce_kernel(const float* __restrict__ partial, int KS, int64_t M, int N,
                              void* __restrict__ c) {
  pdl_trigger();
  pdl_wait();
  const int n_out = EPI == kEpiSwiglu ? (N >> 1) : N;
  const int64_t g = int64_t(blockIdx.x) * 256 + threadIdx.x;   // group of 4 outputs
  const int64_t per_row = n_out >> 2;
  if (g >= M * per_row) return;
  const int64_t row = g / per_row;
  const int col = int(g - row * per_row) * 4;
  const int64_t slice = M * int64_t(N);
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, up[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < KS; ++s) {
    const float4 a = *reinterpret_cast<const float4*>(partial + s * slice + row * N + col);
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    if (EPI == kEpiSwiglu) {
      const float4 u = *reinterpret_cast<const float4*>(partial + s * slice + row * N + (N >> 1) + col);
      up[0] += u.x; up[1] += u.y; up[2] += u.z; up[3] += u.w;
    }
  }
  if (EPI == kEpiF32) {
    *reinterpret_cast<float4*>(static_cast<float*>(c) + row * N + col) =
        make_float4(acc[0], acc[1], acc[2], acc[3]);
    return;
  }
  if (EPI == kEpiSwiglu) {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = __fdividef(acc[i] * up[i], 1.0f + __expf(-acc[i]));
  }
  *reinterpret_cast<uint2*>(static_cast<uint16_t*>(c) + row * n_out + col) =
      make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
}

// bf16 [rows][K] K-major operand: boxes of 64 inputs (128 bytes) x box_rows,
// 128-byte swizzle, rows past the end zero-filled.
bool encode_bf16(CUtensorMap* map, const void* base, int K, int64_t rows, int box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
  const cuuint32_t box[2] = {64u, cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int EPI>
cudaError_t launch_epi_main(const Bf16Params& p, const CUtensorMap& ta, const CUtensorMap& ta2,
                            const CUtensorMap& tb, cudaStream_t st);

template <int EPI>
cudaError_t launch_epi(const Bf16Params& p, const CUtensorMap& ta, const CUtensorMap& ta2,
                       const CUtensorMap& tb, cudaStream_t st) {
  if (p.KS > 1) {
    cudaError_t err = launch_epi_main<EPI>(p, ta, ta2, tb, st);
    if (err != cudaSuccess) return err;
    const int n_out = EPI == kEpiSwiglu ? (p.N >> 1) : p.N;
    const int64_t groups = p.M * (n_out / 4);
    return launch_ex(true, bf16_splitk_reduce_kernel<EPI>, dim3(unsigned((groups + 255) / 256)),
                     dim3(256), 0, st, 1, static_cast<const float*>(p.partial), p.KS, p.M, p.N,
                     p.c);
  }
  return launch_epi_main<EPI>(p, ta, ta2, tb, st);
}

template <int EPI>
cudaError_t launch_epi_main(const Bf16Params& p, const CUtensorMap& ta, const CUtensorMap& ta2,
                            const CUtensorMap& tb, cudaStream_t st) {
  cudaError_t err = cudaFuncSetAttribute(gemm_bf16_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemBytes));
  if (err != cudaSuccess) return err;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int64_t work = int64_t(p.MT) * p.NT * p.KS;
  const int grid = int(work < sms ? work : sms);
  return launch_ex(true, gemm_bf16_kernel<EPI>, dim3(grid), dim3(kThreads), kSmemBytes, st, 1, ta,
                   ta2, tb, p);
}

}  // namespace

// K-slices for a call: 1 unless the tiles cover less than half of the 152
// SMs; then as many equal slices as fit one wave of 152 CTAs, each at least 4
// stages long. Depends only on the shape, so the workspace size can be stated
// before the call.
int bf16_k_splits(int64_t M, int N, int K, int epilogue) {
  const int64_t MT = (M + BM - 1) / BM;
  const int64_t NT = epilogue == kEpiSwiglu ? (N / 2) / 128 : (N + BN - 1) / BN;
  const int64_t tiles = MT * NT;
  const int KT = K / BKB;
  if (tiles >= 76 || KT < 8) return 1;
  int ks = int(152 / tiles);
  ks = ks < KT / 4 ? ks : KT / 4;
  ks = ks < 32 ? ks : 32;
  while (ks > 1 && KT % ks != 0) --ks;   // equal slices
  return ks > 1 ? ks : 1;
}

size_t bf16_partial_bytes(int64_t M, int N, int K, int epilogue) {
  const int ks = bf16_k_splits(M, N, K, epilogue);
  return ks > 1 ? size_t(ks) * size_t(M) * size_t(N) * 4 : 0;
}

cudaError_t launch_gemm_bf16_cat(const uint16_t* a1, int K1, const uint16_t* a2, int K2,
                                 const uint16_t* b, int64_t M, int N, int epilogue, void* c,
                                 float* partial, int* status, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const int K = K1 + K2;
  CUtensorMap ta, ta2, tb;
  if (!encode_bf16(&ta, a1, K1, M, BM)) return cudaErrorInvalidValue;
  if (K2 > 0) {
    if (!encode_bf16(&ta2, a2, K2, M, BM)) return cudaErrorInvalidValue;
  } else {
    ta2 = ta;   // never read: every stage is below K1T
  }
  if (!encode_bf16(&tb, b, K, N, epilogue == kEpiSwiglu ? 128 : BN)) return cudaErrorInvalidValue;
  Bf16Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.K1T = K1 / BKB;
  p.MT = int((M + BM - 1) / BM);
  p.NT = epilogue == kEpiSwiglu ? (N / 2) / 128 : (N + BN - 1) / BN;
  p.KS = bf16_k_splits(M, N, K, epilogue);
  p.KTS = (K / BKB) / p.KS;
  p.partial = partial;
  p.c = c;
  p.status = status;
  if (epilogue == kEpiF32) return launch_epi<kEpiF32>(p, ta, ta2, tb, st);
  if (epilogue == kEpiBf16) return launch_epi<kEpiBf16>(p, ta, ta2, tb, st);
  return launch_epi<kEpiSwiglu>(p, ta, ta2, tb, st);
}

cudaError_t launch_gemm_bf16(const uint16_t* a, const uint16_t* b, int64_t M, int N, int K,
                             int epilogue, void* c, float* partial, int* status, cudaStream_t st) {
  return launch_gemm_bf16_cat(a, K, nullptr, 0, b, M, N, epilogue, c, partial, status, st);
}

}  // namespace moe
