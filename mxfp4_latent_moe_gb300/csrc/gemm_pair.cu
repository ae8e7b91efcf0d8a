// Grouped GEMMs of the routed experts on CTA pairs (tcgen05 cta_group::2):
// the expert's weights are the MMA's M side, 256 weight rows per MMA split
// over the two CTAs of a 2-CTA cluster, and its tokens the N side, up to 128
// (stage 1) or 256 (stage 2) per tile in steps of 16.
//
// Same layer steps as gemm.cu ("The MXFP4 latent MoE on FlyDSL" of "Kimi K3.1
// Pro on AMD Instinct GPUs"; Experts row of "Kimi K3.1 Pro at a glance"):
//   stage 1 (MODE 0): G = W1 . Xq^T, U = W3 . Xq^T (two MMAs per K step into two
//                     accumulators on the same tensor-memory lanes), then
//                     h = silu(G) * U -> MXFP8 in the epilogue
//   stage 2 (MODE 1): Yp^T = W2 . Hq^T, 256 output features per tile -> bf16
//
// Why this arrangement, for prefill batches (hundreds of tokens per expert):
//  - Per CTA and pipeline stage the pair moves half the operand bytes of a
//    single-CTA tile of the same MMA work: each CTA holds its own 128 weight
//    rows and half of the tile's tokens, and the tensor cores of the pair
//    exchange the token halves. So six (stage 2) or five (stage 1) stages fit
//    in shared memory, 2.5-3k cycles of MMA work in flight, and each SM
//    receives 65 (stage 2) or 81 (stage 1) bytes per MMA cycle where the
//    single-CTA token tiles need 96.
//  - One elected thread of the pair issues the MMAs of both SMs, halving the
//    issue work per unit of tensor work.
//  - Tokens are the N side, so the last tile of an expert is as wide as its
//    remaining tokens rounded up to 16, not to 128: at 32,768 tokens (about
//    585 per expert) that is about 8% less tensor work than 128-row tiles.
//  - Weights as the M side pair naturally: both CTAs multiply the same tokens,
//    so every expert's gate/up or down rows fill whole 256-row pairs.
//
// Cluster of two CTAs (ranks 0 and 1), persistent, 320 threads each:
//   warp 0      TMA producer in both CTAs: its CTA's weight box(es) (E2M1,
//               expanded to byte slots by TMA), its half of the tile's tokens
//               (E4M3), its weights' scale atoms and all of the tile's token
//               scale atoms (each SM's tensor memory needs the scales of every
//               token column), all into its own shared memory by cta_group::2
//               TMA loads whose bytes complete on rank 0's full barrier; rank
//               0's producer expects the bytes of both CTAs.
//   warp 1      tensor-memory allocation (both CTAs, collectively); on rank 0
//               then the MMA issuer of the pair: waits until both CTAs'
//               stage has landed, copies the scale atoms into both CTAs'
//               tensor memory (tcgen05.cp.cta_group::2: each CTA's own shared
//               memory into its own tensor memory), issues the MMAs, and frees
//               the stage in both CTAs with one multicast commit.
//   warps 2-9   epilogue in both CTAs on their own 128 weight rows: tcgen05.ld
//               of the accumulator, release (rank 1's warps arrive remotely on
//               rank 0's accumulator-empty barrier, relaxed: their tensor-memory
//               reads have completed by tcgen05.wait::ld, and a release at
//               cluster scope costs far more latency per tile), then the GLU +
//               MX requant (MODE 0) or the bf16 conversion (MODE 1) while the
//               next tile accumulates.
// A first version announced the second CTA's landed stages to rank 0 through
// a relay warp (cluster-scope release and acquire per stage) and ran 2.3x
// slower than the single-CTA token tiles; completing the TMA bytes directly
// on rank 0's barrier removes that per-stage handshake.
// Every wait is bounded (MOE_ERR_DEVICE_TIMEOUT, then drain and exit).
#include "internal.h"

namespace moe {

namespace {

template <int MODE>
struct PairCfg;
template <>
struct PairCfg<0> {                   // w13 + GLU + MXFP8 requant
  static constexpr int NTOK = 128;    // tokens per tile (largest MMA N)
  static constexpr int NA = 2;        // weight boxes per CTA per stage (gate, up)
  static constexpr int STAGES = 5;
};
template <>
struct PairCfg<1> {                   // w2 -> bf16
  static constexpr int NTOK = 256;
  static constexpr int NA = 1;
  static constexpr int STAGES = 6;
};

constexpr int kThreads = 320;
constexpr int BK = 128;                       // inputs per stage
constexpr int PM = 256;                       // weight rows per MMA (the pair's M)
constexpr uint32_t A_BOX = 128 * BK;          // one 128x128 E2M1 box in smem (expanded)
constexpr uint32_t A_BOX_TX = A_BOX / 2;      // its packed bytes (TMA transaction count)
constexpr uint32_t SF_ATOM = 512;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcc1Col = 128;            // MODE 0: up accumulator after the gate one
constexpr uint32_t kSfCol = 256;              // scale slots: 16 columns per stage
constexpr uint32_t kMaxE = 1024;

template <int MODE>
struct PairLayout {
  static constexpr int S = PairCfg<MODE>::STAGES;
  static constexpr uint32_t A_STAGE = PairCfg<MODE>::NA * A_BOX;
  static constexpr uint32_t B_ROWS = PairCfg<MODE>::NTOK / 2;   // TMA box rows of the tokens
  static constexpr uint32_t B_STAGE = B_ROWS * BK;
  static constexpr uint32_t SFA_STAGE = PairCfg<MODE>::NA * SF_ATOM;
  static constexpr uint32_t SFB_STAGE = (PairCfg<MODE>::NTOK / 128) * SF_ATOM;
  static constexpr uint32_t OFF_A = 0;
  static constexpr uint32_t OFF_B = OFF_A + S * A_STAGE;
  static constexpr uint32_t OFF_SFA = OFF_B + S * B_STAGE;
  static constexpr uint32_t OFF_SFB = OFF_SFA + S * SFA_STAGE;
  static constexpr uint32_t OFF_BARS = OFF_SFB + S * SFB_STAGE;
  static constexpr uint32_t NUM_BARS = 2 * S + 3;   // full[S], empty[S], acc_full, acc_empty, drain
  static constexpr uint32_t OFF_MISC = OFF_BARS + NUM_BARS * 8;
  static constexpr uint32_t OFF_SCHED = OFF_MISC + 16;
  static constexpr uint32_t SMEM = OFF_SCHED + 3 * (kMaxE + 1) * 4 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(A_STAGE % 1024 == 0 && B_STAGE % 1024 == 0, "128-byte swizzle atoms");
};

struct PairParams {
  const uint8_t* a_sf;   // TILED scales of the weights
  const uint8_t* b_sf;   // TILED scales of the activations
  const int* counts;     // [E] tokens per expert
  const int* offsets;    // [E+1] group offsets (multiples of 128)
  int E;
  int K;                 // inputs per row
  int I;                 // MODE 0: h width; MODE 1: w2 inputs
  int d;                 // MODE 1: output width
  int n_wtiles;          // weight tiles (256 rows of the pair) per expert
  int64_t rows_capacity;
  uint8_t* out_q;        // MODE 0: hq [rows][I]
  uint8_t* out_sf;       // MODE 0: hs TILED (rows, I)
  uint16_t* out_bf16;    // MODE 1: yp [rows][d]
  int* status;
};

// Unit -> (expert, weight tile, first token row, tokens). An expert has
// ceil(counts[e]/NTOK) token chunks; the chunk index runs fastest.
template <int NTOK>
__device__ __forceinline__ void pair_unit(int unit, const int* prefix, const int* offs,
                                          const int* cnts, int E, int& e, int& wt, int& row0,
                                          int& ntok) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= unit) lo = mid;
    else hi = mid - 1;
  }
  e = lo;
  const int chunks = (cnts[e] + NTOK - 1) / NTOK;
  const int r = unit - prefix[e];
  wt = r / chunks;
  const int c = r - wt * chunks;
  row0 = offs[e] + c * NTOK;
  ntok = min(NTOK, cnts[e] - c * NTOK);
}

// tmap_w: BOXED weight codes; tmap_x: activation codes (box NTOK/2 rows);
// tmap_wsf / tmap_xsf: the TILED scale arrays viewed as rows of 128 bytes,
// boxes of 4 rows = one 512-byte scale atom.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_w,
                             const __grid_constant__ CUtensorMap tmap_x,
                             const __grid_constant__ CUtensorMap tmap_wsf,
                             const __grid_constant__ CUtensorMap tmap_xsf, const PairParams p) {
  using Cfg = PairCfg<MODE>;
  using Lay = PairLayout<MODE>;
  constexpr int S = Lay::S;
  constexpr int NTOK = Cfg::NTOK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::OFF_BARS);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Lay::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::OFF_MISC + 4);
  int* total_holder = reinterpret_cast<int*>(smem + Lay::OFF_MISC + 8);
  int* prefix = reinterpret_cast<int*>(smem + Lay::OFF_SCHED);
  int* offs = prefix + (kMaxE + 1);
  int* cnts = offs + (kMaxE + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int KT = p.K / BK;
  const uint32_t rank = cluster_rank();
  const int pair0 = int(blockIdx.x) >> 1, pairs = int(gridDim.x) >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);    // rank 0: its producer's expect-tx (both CTAs' bytes)
      mbar_init(&empty[s], 1);   // the pair's multicast commit
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 16);   // one arrival per epilogue warp of both CTAs (rank 0 only)
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc2(tmem_holder, kTmemCols);
    tmem_relinquish2();
  }
  pdl_trigger();
  pdl_wait();   // the groups and activations come from the previous kernels
  for (int i = threadIdx.x; i <= E; i += kThreads) {
    offs[i] = p.offsets[i];
    if (i < E) cnts[i] = p.counts[i];
  }
  __syncthreads();
  if (warp == 0) {  // unit prefix over experts: lane owns a run of experts
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int s = 0;
    bool bad = false;  // groups must be multiples of 128 rows holding their counts
    for (int e = e0; e < e1; ++e) {
      const int rows = offs[e + 1] - offs[e];
      bad |= rows < 0 || rows % 128 != 0 || cnts[e] < 0 || cnts[e] > rows;
      s += max(0, (cnts[e] + NTOK - 1) / NTOK) * p.n_wtiles;
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
      run += max(0, (cnts[e] + NTOK - 1) / NTOK) * p.n_wtiles;
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
  cluster_sync_all();   // both CTAs' barriers exist before any remote arrival or commit
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = *total_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Both CTAs load their halves of a stage into their own shared memory;
    // the bytes complete on rank 0's full barrier, where rank 0 expects both.
    const bool leader = elect_one_sync();
    uint32_t stage = 0, phase = 0;
    uint32_t filled = 0, last_parity = 0;
    bool failed = false;
    for (int unit = pair0; unit < total && !failed; unit += pairs) {
      int e, wt, row0, ntok;
      pair_unit<NTOK>(unit, prefix, offs, cnts, E, e, wt, row0, ntok);
      const int n = (ntok + 15) & ~15;   // MMA N
      // this CTA's 128 weight rows (gate and up rows for MODE 0) and tokens
      const int64_t wrow = MODE == 0 ? int64_t(e) * 2 * p.I + int64_t(wt) * PM + rank * 128
                                     : int64_t(e) * p.d + int64_t(wt) * PM + rank * 128;
      const int64_t wrow_up = wrow + p.I;   // MODE 0 only
      const int32_t brow = row0 + int32_t(rank) * (n >> 1);
      const bool two_sfb = n > 128;
      const uint32_t tx_cta = Cfg::NA * (A_BOX_TX + SF_ATOM) + Lay::B_STAGE +
                              (two_sfb ? 2u : 1u) * SF_ATOM;
      for (int kt = 0; kt < KT; ++kt) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag)) {
          failed = true;
          break;
        }
        if (leader) {
          uint8_t* sa = smem + Lay::OFF_A + stage * Lay::A_STAGE;
          uint8_t* sb = smem + Lay::OFF_B + stage * Lay::B_STAGE;
          uint8_t* ssfa = smem + Lay::OFF_SFA + stage * Lay::SFA_STAGE;
          uint8_t* ssfb = smem + Lay::OFF_SFB + stage * Lay::SFB_STAGE;
          const uint32_t bar = peer_addr(&full[stage], 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * tx_cta);
          tma_load_2d_pair(sa, &tmap_w, bar, 0, boxed_row(wrow >> 7, kt, KT));
          tma_load_2d_pair(ssfa, &tmap_wsf, bar, 0, int32_t(((wrow >> 7) * KT + kt) * 4));
          if (MODE == 0) {
            tma_load_2d_pair(sa + A_BOX, &tmap_w, bar, 0, boxed_row(wrow_up >> 7, kt, KT));
            tma_load_2d_pair(ssfa + SF_ATOM, &tmap_wsf, bar, 0,
                             int32_t(((wrow_up >> 7) * KT + kt) * 4));
          }
          tma_load_2d_pair(sb, &tmap_x, bar, kt * BK, brow);
          tma_load_2d_pair(ssfb, &tmap_xsf, bar, 0, int32_t((int64_t(row0 >> 7) * KT + kt) * 4));
          if (two_sfb)
            tma_load_2d_pair(ssfb + SF_ATOM, &tmap_xsf, bar, 0,
                             int32_t((int64_t((row0 >> 7) + 1) * KT + kt) * 4));
        }
        __syncwarp();
        filled |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (failed && leader) {
      *abort_flag = 1;
      set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
    }
    // drain: every copy of both CTAs has landed before either CTA may exit
    // (rank 0's full barriers count them all; rank 1 waits for rank 0 at the
    // final cluster barrier)
    if (rank == 0)
      for (int s = 0; s < S; ++s)
        if ((filled >> s) & 1u)
          if (!mbar_wait_warp(&full[s], (last_parity >> s) & 1u, nullptr) && leader)
            set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
  } else if (warp == 1 && rank == 0) {
    // ----------------------------------------------- MMA issuer of the pair
    const bool leader = elect_one_sync();
    uint32_t stage = 0, phase = 0, acc_phase = 0;
    bool failed = false;
    for (int unit = pair0; unit < total && !failed; unit += pairs) {
      int e, wt, row0, ntok;
      pair_unit<NTOK>(unit, prefix, offs, cnts, E, e, wt, row0, ntok);
      const int n = (ntok + 15) & ~15;
      const uint32_t idesc = idesc_mxf8f6f4(kFmtE2M1, kFmtE4M3, PM, n);
      if (!mbar_wait_cluster_warp(acc_empty, acc_phase ^ 1u, abort_flag)) {
        failed = true;
        break;
      }
      tc_fence_after();
      for (int kt = 0; kt < KT; ++kt) {
        if (!mbar_wait_warp(&full[stage], phase, abort_flag)) {
          failed = true;
          break;
        }
        tc_fence_after();
        if (leader) {
          const uint32_t sa = smem_u32(smem + Lay::OFF_A + stage * Lay::A_STAGE);
          const uint32_t sb = smem_u32(smem + Lay::OFF_B + stage * Lay::B_STAGE);
          const uint32_t ssfa = smem_u32(smem + Lay::OFF_SFA + stage * Lay::SFA_STAGE);
          const uint32_t ssfb = smem_u32(smem + Lay::OFF_SFB + stage * Lay::SFB_STAGE);
          // scale slots of the stage: A (gate) +0, A (up) +4, tokens +8 (and +12)
          const uint32_t sf_t = tmem_base + kSfCol + stage * 16;
          tc_cp2(sf_t, desc_sf_block(ssfa));
          if (MODE == 0) tc_cp2(sf_t + 4, desc_sf_block(ssfa + SF_ATOM));
          tc_cp2(sf_t + 8, desc_sf_block(ssfb));
          if (n > 128) tc_cp2(sf_t + 12, desc_sf_block(ssfb + SF_ATOM));
          const uint64_t adesc = desc_sw128_kmajor(sa);
          const uint64_t bdesc = desc_sw128_kmajor(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint32_t id = idesc_with_sf_id(idesc, uint32_t(kk));
            const uint32_t accum = (kt > 0 || kk > 0) ? 1u : 0u;
            tc_mma_mx2(tmem_base, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk), id, sf_t,
                       sf_t + 8, accum);
            if (MODE == 0)
              tc_mma_mx2(tmem_base + kAcc1Col, adesc + uint64_t((A_BOX >> 4) + 2 * kk),
                         bdesc + uint64_t(2 * kk), id, sf_t + 4, sf_t + 8, accum);
          }
          // the stage is free in both CTAs once these MMAs have read it
          tc_commit2_mc(&empty[stage], uint16_t(0x3));
        }
        __syncwarp();
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (failed) break;
      if (leader) tc_commit2_mc(acc_full, uint16_t(0x3));
      __syncwarp();
      acc_phase ^= 1u;
    }
    if (failed && leader) {
      *abort_flag = 1;
      set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
    }
    // drain: all issued tensor-core work is complete before tensor memory is freed
    if (leader) tc_commit2_mc(drain, uint16_t(0x1));
    __syncwarp();
    if (!mbar_wait_warp(drain, 0, nullptr) && leader) set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    // Two warps per tensor-memory lane quarter (warp % 4): thread = one weight
    // row of this CTA (lane), the two warps split the tile's token columns.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t acc_empty_pair = peer_addr(acc_empty, 0);
    uint32_t acc_phase = 0;
    for (int unit = pair0; unit < total; unit += pairs) {
      int e, wt, row0, ntok;
      pair_unit<NTOK>(unit, prefix, offs, cnts, E, e, wt, row0, ntok);
      bool ok = mbar_wait(acc_full, acc_phase, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tq = tmem_base + (uint32_t(q * 32) << 16);
      const int c0 = half * (NTOK / 2);        // first token column of this warp
      if (MODE == 0) {
        uint32_t g[64], u[64];
        {
          uint32_t (&g0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&g[0]);
          uint32_t (&g1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&g[32]);
          uint32_t (&u0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&u[0]);
          uint32_t (&u1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&u[32]);
          tmem_ld_32x32b_x32(tq + c0, g0);
          tmem_ld_32x32b_x32(tq + c0 + 32, g1);
          tmem_ld_32x32b_x32(tq + kAcc1Col + c0, u0);
          tmem_ld_32x32b_x32(tq + kAcc1Col + c0 + 32, u1);
        }
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(acc_empty);
          else mbar_arrive_remote_relaxed(acc_empty_pair);
        }
        acc_phase ^= 1u;
        // h of weight row i (this lane) for each token column; its MX block of
        // 32 consecutive features is the warp's 32 lanes
        const int i = wt * PM + int(rank) * 128 + q * 32 + lane;
        const int64_t sf_block = i >> 5;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          if (c0 + c < ntok) {   // padding tokens are not stored (warp-uniform test)
            const float gf = __uint_as_float(g[c]);
            const float h = __fdividef(gf * __uint_as_float(u[c]), 1.0f + __expf(-gf));
            const float amax =
                __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h))));
            const int code = mx_scale_code(amax);
            const int64_t row = int64_t(row0) + c0 + c;
            p.out_q[row * p.I + i] = uint8_t(e4m3x2(h * mx_scale_mult(code), 0.0f) & 0xFFu);
            if (lane == 0) p.out_sf[tiled_sf_offset(row, sf_block, p.I)] = uint8_t(code);
          }
        }
      } else {
        uint32_t v[128];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tmem_ld_32x32b_x32(tq + c0 + 32 * k,
                             *reinterpret_cast<uint32_t(*)[32]>(&v[32 * k]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(acc_empty);
          else mbar_arrive_remote_relaxed(acc_empty_pair);
        }
        acc_phase ^= 1u;
        const int j = wt * PM + int(rank) * 128 + q * 32 + lane;   // output feature
        uint16_t* out = p.out_bf16 + int64_t(row0 + c0) * p.d + j;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c0 + c < ntok)   // padding tokens are not stored
            out[int64_t(c) * p.d] =
                __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[c])));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA of the pair frees tensor memory or exits while the other may
  // still arrive on its barriers or use its shared memory
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc2(tmem_base, kTmemCols);
}

template <int MODE>
cudaError_t launch_pair(const PairParams& p, const CUtensorMap& tw, const CUtensorMap& tx,
                        const CUtensorMap& twsf, const CUtensorMap& txsf, cudaStream_t st) {
  auto kernel = grouped_gemm_pair_kernel<MODE>;
  constexpr uint32_t smem = PairLayout<MODE>::SMEM;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (err != cudaSuccess) return err;
  // units: at most one per 128 grouped rows per weight tile
  const int64_t max_units = (p.rows_capacity / 128) * p.n_wtiles;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  cfg.gridDim = dim3(unsigned(sms));
  int clusters = 0;
  err = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
  if (err != cudaSuccess) return err;
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  const int64_t pairs = max_units < clusters ? (max_units > 0 ? max_units : 1) : clusters;
  return launch_ex(true, kernel, dim3(unsigned(2 * pairs)), dim3(kThreads), smem, st, 2, tw, tx,
                   twsf, txsf, p);
}

}  // namespace

cudaError_t launch_gemm_pair_w13_glu(const uint8_t* xq, const uint8_t* xs, const int* counts,
                                     const int* offsets, int E, int d, int I, const uint8_t* w13,
                                     const uint8_t* w13_sf, uint8_t* hq, uint8_t* hs,
                                     int64_t rows_capacity, int* status, cudaStream_t st) {
  CUtensorMap tw, tx, twsf, txsf;
  if (!encode_boxed_weights(&tw, w13, int64_t(E) * 2 * I, d)) return cudaErrorInvalidValue;
  if (!encode_operand(&tx, xq, false, d, rows_capacity, PairLayout<0>::B_ROWS))
    return cudaErrorInvalidValue;
  if (!encode_scale_atoms(&twsf, w13_sf, int64_t(E) * 2 * I * (d / 32)) ||
      !encode_scale_atoms(&txsf, xs, rows_capacity * (d / 32)))
    return cudaErrorInvalidValue;
  PairParams p{};
  p.a_sf = w13_sf;
  p.b_sf = xs;
  p.counts = counts;
  p.offsets = offsets;
  p.E = E;
  p.K = d;
  p.I = I;
  p.d = d;
  p.n_wtiles = I / PM;
  p.rows_capacity = rows_capacity;
  p.out_q = hq;
  p.out_sf = hs;
  p.status = status;
  return launch_pair<0>(p, tw, tx, twsf, txsf, st);
}

cudaError_t launch_gemm_pair_w2(const uint8_t* hq, const uint8_t* hs, const int* counts,
                                const int* offsets, int E, int I, int d, const uint8_t* w2,
                                const uint8_t* w2_sf, uint16_t* yp, int64_t rows_capacity,
                                int* status, cudaStream_t st) {
  CUtensorMap tw, tx, twsf, txsf;
  if (!encode_boxed_weights(&tw, w2, int64_t(E) * d, I)) return cudaErrorInvalidValue;
  if (!encode_operand(&tx, hq, false, I, rows_capacity, PairLayout<1>::B_ROWS))
    return cudaErrorInvalidValue;
  if (!encode_scale_atoms(&twsf, w2_sf, int64_t(E) * d * (I / 32)) ||
      !encode_scale_atoms(&txsf, hs, rows_capacity * (I / 32)))
    return cudaErrorInvalidValue;
  PairParams p{};
  p.a_sf = w2_sf;
  p.b_sf = hs;
  p.counts = counts;
  p.offsets = offsets;
  p.E = E;
  p.K = I;
  p.I = I;
  p.d = d;
  p.n_wtiles = d / PM;
  p.rows_capacity = rows_capacity;
  p.out_bf16 = yp;
  p.status = status;
  return launch_pair<1>(p, tw, tx, twsf, txsf, st);
}

}  // namespace moe
