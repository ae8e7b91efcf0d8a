// Grouped GEMMs of the routed experts for few tokens per expert (decode
// batches), on tcgen05 block-scaled tensor cores with the operands swapped:
// the expert's weights are the MMA's M side (128 weight rows per MMA) and its
// tokens the N side, so an expert holding a handful of tokens costs N = 32 of
// tensor work (not M = 128) while its weights stream from HBM exactly once.
//
// Same layer steps as gemm.cu ("The MXFP4 latent MoE on FlyDSL" of "Kimi K3.1
// Pro on AMD Instinct GPUs"; Experts row of "Kimi K3.1 Pro at a glance"):
//   stage 1 (MODE 0): G = W1 . Xq^T and U = W3 . Xq^T, two MMAs per K step into
//                     two accumulators that share tensor-memory lanes, then
//                     h = silu(G) * U -> MXFP8 in the epilogue
//   stage 2 (MODE 1): Yp^T = W2 . Hq^T for 256 output features per tile (two
//                     MMAs of 128 weight rows), -> bf16
// MXFP4 weights are the A operand (E2M1, kind::mxf8f6f4 format 5), MXFP8
// activations the B operand (E4M3), one E8M0 scale per 32 inputs each side.
//
// Groups are padded to 32 rows and the per-expert token counts are read on
// the device: a tile is (expert, weight rows, NT-row chunk of the group), MMA
// N = NT, with NT = 32, or 64 once the experts average more than ~24 tokens
// (a 64-token chunk costs the same MMA issue time as a 32-token one, so an
// expert with 25-64 tokens then streams its weights through one CTA instead
// of two). The activations' scales are in the GROUP32 layout, one 512-byte
// block per 32 rows x 128 inputs, so 32 rows' scales reach one tensor-memory
// column with one aligned copy per stage (a 64-row chunk: two blocks, merged
// in shared memory so that one copy fills two adjacent columns). A stage is 32 KB of expanded weights + 4 or 8 KB of
// tokens, so five stages fit: 80 KB of weights in flight per SM, the
// quantity that bounds HBM streaming here.
//
// CTA: persistent, one per SM, 320 threads: warp 0 TMA producer, warp 1
// tensor-memory allocator + MMA issuer (both warps converged, one elected
// lane issues), warps 2-9 epilogue (two per lane quarter, 16 tokens each). Accumulators are double-buffered, so the
// next tile's MMAs never wait for the epilogue. The MX block of h is 32
// consecutive features = the 32 lanes of one warp: its amax is one warp
// reduction per token.
#include "internal.h"

namespace moe {

namespace {

constexpr int WM = 128;            // weight rows per MMA (M)
constexpr int BK = 128;            // inputs per stage
constexpr int GPAD = 32;           // group padding (rows) of this family
constexpr int STAGES = 5;
constexpr int kThreads = 320;

constexpr uint32_t A_TILE = WM * BK;         // one 128-row E2M1 tile in smem (expanded)
constexpr uint32_t A_TILE_TX = A_TILE / 2;   // its packed bytes (TMA transaction count)
constexpr uint32_t A_STAGE = 2 * A_TILE;
constexpr uint32_t SF_ATOM = 512;
constexpr uint32_t kMaxE = 1024;

// Per chunk width NT (tokens per tile, the MMA's N): accumulator buffer b
// holds acc0 at columns [2NT b, 2NT b + NT) and acc1 (up rows / upper w2
// rows) at [2NT b + NT, 2NT (b + 1)); scale slots from column 4NT, 16 per
// stage (A0 +0, A1 +4, B +8; a 64-token chunk's B scales fill +8 and +9).
template <int NT>
struct DecodeLayout {
  static_assert(NT == 32 || NT == 64, "32- or 64-token chunks");
  static constexpr uint32_t kAccStride = 2 * NT;
  static constexpr uint32_t kAcc1Col = NT;
  static constexpr uint32_t kSfCol = 4 * NT;
  static constexpr uint32_t kTmemCols = NT == 32 ? 256 : 512;
  static_assert(kSfCol + 16 * STAGES <= kTmemCols, "tensor memory budget");
  static constexpr uint32_t B_STAGE = NT * BK;                 // NT rows of E4M3 tokens
  static constexpr uint32_t SFB_STAGE = (NT / 32) * SF_ATOM;   // GROUP32 blocks
  static constexpr uint32_t kOffA = 0;
  static constexpr uint32_t kOffB = kOffA + STAGES * A_STAGE;
  static constexpr uint32_t kOffSfa = kOffB + STAGES * B_STAGE;
  static constexpr uint32_t kOffSfb = kOffSfa + STAGES * 2 * SF_ATOM;
  static constexpr uint32_t kOffBars = kOffSfb + STAGES * SFB_STAGE;
  // full[S], empty[S], acc_full[2], acc_empty[2], drain
  static constexpr uint32_t kNumBars = 2 * STAGES + 5;
  static constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
  static constexpr uint32_t kOffSched = kOffMisc + 16;
  static constexpr uint32_t kSmemBytes = kOffSched + 3 * (kMaxE + 1) * 4 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct DecodeParams {
  const uint8_t* a_sf;  // TILED scales of the weights
  const uint8_t* b_sf;  // GROUP32 scales of the activations
  const int* counts;    // [E] tokens per expert
  const int* offsets;   // [E+1] group offsets (multiples of 32)
  int E;
  int K;                // inputs per row
  int I;                // MODE 0: h width; MODE 1: w2 inputs
  int d;                // MODE 1: output width
  int n_tiles;          // weight tiles per expert: I/128 (MODE 0), ceil(d/256) (MODE 1)
  int64_t rows_capacity;
  uint8_t* out_q;       // MODE 0: hq [rows][I]
  uint8_t* out_sf;      // MODE 0: hs TILED (rows, I)
  uint16_t* out_bf16;   // MODE 1: yp [rows][d]
  int* status;
};

// Tile -> (expert, weight tile, first token row). An expert has
// ceil(counts[e]/NT) token chunks; the chunk index runs fastest.
template <int NT>
__device__ __forceinline__ void decode_tile(int tile, const int* prefix, const int* offs,
                                            const int* cnts, int E, int& e, int& nt, int& row0) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  e = lo;
  const int chunks = (cnts[e] + NT - 1) / NT;
  const int r = tile - prefix[e];
  nt = r / chunks;
  row0 = offs[e] + (r - nt * chunks) * NT;
}

template <int MODE, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_decode_kernel(const __grid_constant__ CUtensorMap tmap_w,
                               const __grid_constant__ CUtensorMap tmap_x, const DecodeParams p) {
  using L = DecodeLayout<NT>;
  constexpr uint32_t kOffA = L::kOffA, kOffB = L::kOffB, kOffSfa = L::kOffSfa,
                     kOffSfb = L::kOffSfb, kOffBars = L::kOffBars, kOffMisc = L::kOffMisc,
                     kOffSched = L::kOffSched, B_STAGE = L::B_STAGE, SFB_STAGE = L::SFB_STAGE,
                     kAccStride = L::kAccStride, kAcc1Col = L::kAcc1Col, kSfCol = L::kSfCol,
                     kTmemCols = L::kTmemCols;
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
  int* total_holder = reinterpret_cast<int*>(smem + kOffMisc + 8);
  int* prefix = reinterpret_cast<int*>(smem + kOffSched);
  int* offs = prefix + (kMaxE + 1);
  int* cnts = offs + (kMaxE + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int KT = p.K / BK;

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
  pdl_wait();   // the groups and activations come from the previous kernels
  for (int i = threadIdx.x; i <= E; i += kThreads) {
    offs[i] = p.offsets[i];
    if (i < E) cnts[i] = p.counts[i];
  }
  __syncthreads();
  if (warp == 0) {  // tile prefix over experts: lane owns a run of experts
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int s = 0;
    bool bad = false;  // groups must be multiples of 32 rows holding their counts
    for (int e = e0; e < e1; ++e) {
      const int rows = offs[e + 1] - offs[e];
      bad |= rows < 0 || rows % GPAD != 0 || cnts[e] < 0 || cnts[e] > rows;
      s += max(0, (cnts[e] + NT - 1) / NT) * p.n_tiles;
    }
    bad = __any_sync(0xffffffffu, bad);
    int incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += n;
    }
    int run = incl - s;
    for (int e = e0; e < e1; ++e) {
      prefix[e] = run;
      run += max(0, (cnts[e] + NT - 1) / NT) * p.n_tiles;
    }
    if (lane == 31) {
      const bool ok = !bad && offs[0] == 0 && int64_t(offs[E]) <= p.rows_capacity;
      if (!ok && blockIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE_BAD_INPUT);
      prefix[E] = incl;
      *total_holder = ok ? incl : 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = *total_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const bool leader = elect_one_sync();
    uint32_t stage = 0, phase = 0;
    uint32_t filled = 0, last_parity = 0;
    bool failed = false;
    for (int tile = blockIdx.x; tile < total && !failed; tile += gridDim.x) {
      int e, nt, row0;
      decode_tile<NT>(tile, prefix, offs, cnts, E, e, nt, row0);
      // weight rows: MODE 0 gate and up rows, MODE 1 the tile's two 128-row halves
      const int64_t wrow0 = MODE == 0 ? int64_t(e) * 2 * p.I + int64_t(nt) * WM
                                      : int64_t(e) * p.d + int64_t(nt) * 2 * WM;
      const bool two = MODE == 0 || nt * 2 * WM + WM < p.d;
      const int64_t wrow1 = MODE == 0 ? wrow0 + p.I : wrow0 + WM;
      // a 64-row chunk's second 32 rows' scales, if those rows are in the group
      // (past it they are padding or another expert's rows, and past the last
      // group the scale array may end)
      const bool sfb1 = NT == 64 && row0 + 32 < offs[e + 1];
      const uint32_t tx = (two ? 2u : 1u) * (A_TILE_TX + SF_ATOM) + B_STAGE + SF_ATOM +
                          (sfb1 ? SF_ATOM : 0u);
      for (int kt = 0; kt < KT; ++kt) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag)) {
          failed = true;
          break;
        }
        if (leader) {
          uint8_t* sa = smem + kOffA + stage * A_STAGE;
          uint8_t* sb = smem + kOffB + stage * B_STAGE;
          uint8_t* ssfa = smem + kOffSfa + stage * 2 * SF_ATOM;
          uint8_t* ssfb = smem + kOffSfb + stage * SFB_STAGE;
          mbar_arrive_expect_tx(&full[stage], tx);
          tma_load_2d(sa, &tmap_w, &full[stage], 0, boxed_row(wrow0 >> 7, kt, KT));
          bulk_load(ssfa, p.a_sf + ((wrow0 >> 7) * KT + kt) * SF_ATOM, SF_ATOM, &full[stage]);
          if (two) {
            tma_load_2d(sa + A_TILE, &tmap_w, &full[stage], 0, boxed_row(wrow1 >> 7, kt, KT));
            bulk_load(ssfa + SF_ATOM, p.a_sf + ((wrow1 >> 7) * KT + kt) * SF_ATOM, SF_ATOM,
                      &full[stage]);
          }
          tma_load_2d(sb, &tmap_x, &full[stage], kt * BK, row0);
          bulk_load(ssfb, p.b_sf + (int64_t(row0 >> 5) * KT + kt) * SF_ATOM, SF_ATOM,
                    &full[stage]);
          if (sfb1)
            bulk_load(ssfb + SF_ATOM, p.b_sf + (int64_t((row0 >> 5) + 1) * KT + kt) * SF_ATOM,
                      SF_ATOM, &full[stage]);
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
    const uint32_t idesc = idesc_mxf8f6f4(kFmtE2M1, kFmtE4M3, WM, NT);
    uint32_t stage = 0, phase = 0;
    uint32_t acc_phases = 0;  // bit b: phase parity of accumulator buffer b
    int buf = 0;
    bool failed = false;
    for (int tile = blockIdx.x; tile < total && !failed; tile += gridDim.x) {
      int e, nt, row0;
      decode_tile<NT>(tile, prefix, offs, cnts, E, e, nt, row0);
      const bool two = MODE == 0 || nt * 2 * WM + WM < p.d;
      if (!mbar_wait_warp(&acc_empty[buf], ((acc_phases >> buf) & 1u) ^ 1u, abort_flag)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem_base + uint32_t(buf) * kAccStride;
      for (int kt = 0; kt < KT; ++kt) {
        if (!mbar_wait_warp(&full[stage], phase, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after();
        if constexpr (NT == 64) {
          // A 64-token chunk's B scales: the MMA reads token row r's scales
          // from tensor-memory column (r / 32) of its slot, lane r % 32. A
          // GROUP32 block holds lane i's row scales in the first 4 of its 16
          // bytes and leaves the rest unused, so the second block's word moves
          // into the first block's second word and one copy (4-column aligned,
          // as tcgen05.cp needs) places both. Past the group the second block
          // holds stale bytes: those tokens' results are not stored.
          uint32_t* blk = reinterpret_cast<uint32_t*>(smem + kOffSfb + stage * SFB_STAGE);
          blk[4 * lane + 1] = blk[SF_ATOM / 4 + 4 * lane];
          fence_proxy_async_shared();   // generic writes before the tensor core's copy
          __syncwarp();
        }
        if (leader) {
          const uint32_t sa = smem_u32(smem + kOffA + stage * A_STAGE);
          const uint32_t sb = smem_u32(smem + kOffB + stage * B_STAGE);
          const uint32_t ssfa = smem_u32(smem + kOffSfa + stage * 2 * SF_ATOM);
          const uint32_t ssfb = smem_u32(smem + kOffSfb + stage * SFB_STAGE);
          // A0: +0, A1: +4, B: +8 (a 64-token chunk's rows 32-63 at +9)
          const uint32_t sf_t = tmem_base + kSfCol + stage * 16;
          tc_cp_32x128b_x4(sf_t, desc_sf_block(ssfa));
          if (two) tc_cp_32x128b_x4(sf_t + 4, desc_sf_block(ssfa + SF_ATOM));
          tc_cp_32x128b_x4(sf_t + 8, desc_sf_block(ssfb));
          const uint64_t adesc = desc_sw128_kmajor(sa);
          const uint64_t bdesc = desc_sw128_kmajor(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint32_t id = idesc_with_sf_id(idesc, uint32_t(kk));
            const uint32_t accum = (kt > 0 || kk > 0) ? 1u : 0u;
            tc_mma_mx(acc, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk), id, sf_t,
                      sf_t + 8, accum);
            if (two)
              tc_mma_mx(acc + kAcc1Col, adesc + uint64_t((A_TILE >> 4) + 2 * kk),
                        bdesc + uint64_t(2 * kk), id, sf_t + 4, sf_t + 8, accum);
          }
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
    // Thread = one weight row (tensor-memory lane) of the tile; the two warps
    // of a lane quarter take tokens [0, NT/2) and [NT/2, NT) of the chunk.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint32_t acc_phases = 0;
    int buf = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, nt, row0;
      decode_tile<NT>(tile, prefix, offs, cnts, E, e, nt, row0);
      const bool two = MODE == 0 || nt * 2 * WM + WM < p.d;
      bool ok = mbar_wait(&acc_full[buf], (acc_phases >> buf) & 1u, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
      tc_fence_after();
      constexpr int HT = NT / 2;   // tokens per warp
      const uint32_t tq = tmem_base + uint32_t(buf) * kAccStride + (uint32_t(q * 32) << 16) +
                          uint32_t(HT * half);
      uint32_t v0[HT], v1[HT];
      if constexpr (NT == 32) {
        tmem_ld_32x32b_x16(tq, v0);
        if (two) tmem_ld_32x32b_x16(tq + kAcc1Col, v1);
      } else {
        tmem_ld_32x32b_x32(tq, v0);
        if (two) tmem_ld_32x32b_x32(tq + kAcc1Col, v1);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);   // the whole warp has read its part
      acc_phases ^= 1u << buf;
      buf ^= 1;
      // rows of the chunk past the expert's tokens are padding: not stored
      const int live = cnts[e] - (row0 - offs[e]) - HT * half;
#pragma unroll
      for (int i = 0; i < HT; ++i) {
        if (i >= live) break;
        const int64_t row = int64_t(row0) + HT * half + i;
        if (MODE == 0) {
          const float gf = __uint_as_float(v0[i]);
          const float h = __fdividef(gf * __uint_as_float(v1[i]), 1.0f + __expf(-gf));
          // amax over the warp's 32 features = one MX block of the token's h row
          const float amax =
              __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h))));
          const int code = mx_scale_code(amax);
          const int feat = nt * WM + q * 32 + lane;
          p.out_q[row * p.I + feat] = uint8_t(e4m3x2(h * mx_scale_mult(code), 0.0f) & 0xFFu);
          if (lane == 0) p.out_sf[group32_sf_offset(row, feat >> 5, p.I)] = uint8_t(code);
        } else {
          const int feat = nt * 2 * WM + q * 32 + lane;
          p.out_bf16[row * p.d + feat] =
              __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v0[i])));
          if (two)
            p.out_bf16[row * p.d + feat + WM] =
                __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v1[i])));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

template <int MODE, int NT>
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tw, const CUtensorMap& tx,
                          cudaStream_t st) {
  constexpr uint32_t smem = DecodeLayout<NT>::kSmemBytes;
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_decode_kernel<MODE, NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (err != cudaSuccess) return err;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int64_t max_tiles = (p.rows_capacity / GPAD) * p.n_tiles;
  const int grid = int(max_tiles < sms ? (max_tiles > 0 ? max_tiles : 1) : sms);
  return launch_ex(true, grouped_gemm_decode_kernel<MODE, NT>, dim3(grid), dim3(kThreads), smem,
                   st, 1, tw, tx, p);
}

// Chunk width from the grouped-row capacity: rows_capacity is about
// T*k + 31*E for groups padded to 32 (T*k >= E), so more than 55 rows of
// capacity per expert means more than ~24 routed rows per expert, where two
// 32-token chunks per expert start to outnumber one 64-token chunk.
int chunk_width(int64_t rows_capacity, int E) { return rows_capacity > 55 * int64_t(E) ? 64 : 32; }

}  // namespace

cudaError_t launch_gemm_decode_w13_glu(const uint8_t* xq, const uint8_t* xs, const int* counts,
                                       const int* offsets, int E, int d, int I,
                                       const uint8_t* w13, const uint8_t* w13_sf, uint8_t* hq,
                                       uint8_t* hs, int64_t rows_capacity, int* status,
                                       cudaStream_t st) {
  const int nt = chunk_width(rows_capacity, E);
  CUtensorMap tw, tx;
  if (!encode_boxed_weights(&tw, w13, int64_t(E) * 2 * I, d)) return cudaErrorInvalidValue;
  if (!encode_operand(&tx, xq, false, d, rows_capacity, nt)) return cudaErrorInvalidValue;
  DecodeParams p{};
  p.a_sf = w13_sf;
  p.b_sf = xs;
  p.counts = counts;
  p.offsets = offsets;
  p.E = E;
  p.K = d;
  p.I = I;
  p.d = d;
  p.n_tiles = I / WM;
  p.rows_capacity = rows_capacity;
  p.out_q = hq;
  p.out_sf = hs;
  p.status = status;
  return nt == 64 ? launch_decode<0, 64>(p, tw, tx, st) : launch_decode<0, 32>(p, tw, tx, st);
}

cudaError_t launch_gemm_decode_w2(const uint8_t* hq, const uint8_t* hs, const int* counts,
                                  const int* offsets, int E, int I, int d, const uint8_t* w2,
                                  const uint8_t* w2_sf, uint16_t* yp, int64_t rows_capacity,
                                  int* status, cudaStream_t st) {
  const int nt = chunk_width(rows_capacity, E);
  CUtensorMap tw, tx;
  if (!encode_boxed_weights(&tw, w2, int64_t(E) * d, I)) return cudaErrorInvalidValue;
  if (!encode_operand(&tx, hq, false, I, rows_capacity, nt)) return cudaErrorInvalidValue;
  DecodeParams p{};
  p.a_sf = w2_sf;
  p.b_sf = hs;
  p.counts = counts;
  p.offsets = offsets;
  p.E = E;
  p.K = I;
  p.I = I;
  p.d = d;
  p.n_tiles = (d + 2 * WM - 1) / (2 * WM);
  p.rows_capacity = rows_capacity;
  p.out_bf16 = yp;
  p.status = status;
  return nt == 64 ? launch_decode<1, 64>(p, tw, tx, st) : launch_decode<1, 32>(p, tw, tx, st);
}

}  // namespace moe
