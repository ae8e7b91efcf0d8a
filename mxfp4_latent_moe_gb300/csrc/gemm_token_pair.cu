// Grouped GEMMs of the routed experts over CTA pairs: the prefill path for
// the full 256-row pairs of 128-row m-tiles of the experts that hold an even
// number of m-tiles or at least kPairMinMtiles of them (runs_as_pairs).
//
// Same arithmetic as the single-CTA token tiles (gemm.cu; "Kimi K3.1 Pro on
// AMD Instinct GPUs" and "The MXFP4 latent MoE on FlyDSL" for the MXFP4
// weights and the FP8 second stage):
//   stage 1 (MODE 0): [gate | up] = Xq . [W1 | W3]^T, h = silu(gate) * up,
//                     h -> MXFP8 (E4M3 + E8M0 per 32) in the epilogue
//   stage 2 (MODE 1): Yp = Hq . W2^T -> bf16
// but one tcgen05.mma.cta_group::2 (kind::mxf8f6f4, or kind::mxf4 for the
// A4W4 stage 1) covers 256 token rows, 128 in each CTA's shared memory and
// accumulator, against the tile's 256 weight rows, 128 in each CTA's shared
// memory (stage 1: the gate rows in the first CTA, the up rows in the second;
// the two SMs' tensor cores exchange them). Per pipeline stage each CTA then
// holds 16 KB of tokens and 16 KB of weights instead of 16 KB and 32 KB, so
// six stages fit in shared memory instead of four. With four, a stage's slot
// is held for its copies' latency plus the MMA's completion (about 2,600
// cycles at full load), which caps the tensor pipe near 75%; six cover it.
// A heavy expert's odd last m-tile has no partner and runs in the single-CTA
// kernel, launched after this one, with every m-tile of the experts that do
// not run as pairs. Measured on the full layer: with 2 or 4 m-tiles per
// expert (uniform routing at T = 8,192 and 24,576) pairs made it 7-9%
// (MXFP8) and 11-12% (A4W4) faster, at the skewed T = 8,192 (heavy experts)
// 2% and 5%; with five per expert (T = 32,768), pairs plus a second launch
// for every expert's odd last m-tile made it 3% slower.
//
// CTA organisation: 2-CTA clusters, persistent, 320 threads per CTA.
//   warp 0      TMA producer in both CTAs: its 128 token rows, its 128 weight
//               rows (E2M1 expanded by TMA to byte slots, 16U4_ALIGN16B), its
//               tokens' scale atom and both weight scale atoms (each SM's
//               tensor memory needs the scales of all 256 weight rows), all by
//               cta_group::2 TMA loads whose bytes complete on the first CTA's
//               full barrier (which expects both CTAs' bytes).
//   warp 1      tensor-memory allocation (both CTAs, collectively); in the
//               first CTA the MMA issuer of the pair: copies the stage's scale
//               atoms into both CTAs' tensor memory (tcgen05.cp.cta_group::2,
//               each CTA's own shared memory into its own tensor memory),
//               issues the 4 MMAs, and frees the stage in both CTAs with one
//               multicast commit.
//   warps 2-9   epilogue in both CTAs: tcgen05.ld of the accumulator (one
//               token row and half the columns per thread) straight into
//               registers, release of the accumulator, then the fused GLU +
//               MX requant (MODE 0) or the bf16 conversion (MODE 1) overlapped
//               with the next tile's MMAs. The second CTA's warps release on
//               the first CTA's barrier with a relaxed remote arrive: its
//               tensor-memory reads have completed (tcgen05.wait::ld) before
//               it, and a release at cluster scope made each handoff about
//               1,800 cycles slower.
// Units are (expert, n-tile, pair of m-tiles) with the pair fastest, so CTA
// pairs running at the same time share one expert's weight tile through L2.
// The expert row offsets are read on the device: no host synchronisation.
// Every wait is bounded; on expiry the CTA records MOE_ERR_DEVICE_TIMEOUT,
// drains its outstanding copies and tensor-core work, frees tensor memory and
// exits.
#include "internal.h"

namespace moe {

namespace {

constexpr int BM = 128;            // token rows per CTA (half the pair's MMA M)
constexpr int PM = 2 * BM;         // token rows per CTA pair (the MMA's M)
constexpr int BK = 128;            // inputs per pipeline stage (MXFP8 activations)
constexpr int BK4 = 256;           // inputs per pipeline stage (A4W4: MXFP4 activations)
constexpr int BN = 256;            // MMA N: weight rows per tile, 128 in each CTA
constexpr int STAGES = 6;
constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;    // accumulator: columns [0, 256)
constexpr uint32_t kSfCol = 256;   // scale slots: 32 columns per stage
// A: this CTA's 128 token rows x 128 bytes (128 E4M3 inputs, or 256 packed
// E2M1 inputs).
constexpr uint32_t A_BYTES = BM * 128;
// B: this CTA's 128 weight rows. MXFP8 path: TMA's 16U4_ALIGN16B expansion
// puts each 16 E2M1 codes (8 packed bytes) in the low half of a 16-byte slot,
// so a 128-input row takes 128 bytes of shared memory; the transaction count
// is the packed size, half of that. A4W4 path: two packed 8 KB boxes (the
// stage's two 128-input halves), no expansion, the same 16 KB.
constexpr uint32_t B_BYTES = (BN / 2) * 128;
constexpr uint32_t B_TX_BYTES = B_BYTES / 2;
constexpr uint32_t B_BOX = 8192;   // one BOXED weight box: 128 rows x 64 bytes
// scale atoms per stage and CTA: MXFP8 A 1, B 2 (all 256 weight rows);
// A4W4 A 2, B 4 (512 bytes each)
constexpr uint32_t SF_ATOM = 512;
constexpr uint32_t SFA_BYTES = 1024;
constexpr uint32_t SFB_BYTES = 2048;
constexpr uint32_t kStageTx = A_BYTES + B_TX_BYTES + SF_ATOM + 2 * SF_ATOM;
constexpr uint32_t kStageTxA4 = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;

constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + STAGES * A_BYTES;
constexpr uint32_t kOffSfa = kOffB + STAGES * B_BYTES;
constexpr uint32_t kOffSfb = kOffSfa + STAGES * SFA_BYTES;
constexpr uint32_t kOffBars = kOffSfb + STAGES * SFB_BYTES;
constexpr uint32_t kNumBars = 2 * STAGES + 3;  // full[S], empty[S], acc_full, acc_empty, drain
constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
constexpr uint32_t kOffSched = kOffMisc + 16;
constexpr uint32_t kMaxE = kMaxExperts;
constexpr uint32_t kSmemBytes = kOffSched + 3 * (kMaxE + 1) * 4 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct PairParams {
  const int* counts;     // [E] tokens per expert
  const int* offsets;    // [E+1]
  int E;
  int K;                 // inputs per row (d for MODE 0, I for MODE 1)
  int I;                 // MODE 0: gate/up width; MODE 1: unused
  int d;                 // MODE 1: output width; MODE 0: unused
  int n_tiles;           // per expert
  int64_t rows_capacity;
  uint8_t* out_q;        // MODE 0: hq [rows][I]
  uint8_t* out_sf;       // MODE 0: hs TILED (rows, I)
  uint16_t* out_bf16;    // MODE 1: yp [rows][d]
  int* status;
  bool out32;            // the output base is 32-byte aligned: 32-byte stores
};

// Full pairs of 128-row m-tiles of an expert that runs as pairs:
// floor(ceil(counts[e]/128)/2), else 0. An odd last m-tile, and every m-tile
// of a lighter expert, is left to the single-CTA token-tile kernel.
__device__ __forceinline__ int full_pairs(int count) {
  const int m = (count + BM - 1) / BM;
  return runs_as_pairs(m) ? (m >> 1) : 0;
}

// Unit -> (expert, n-tile, first row of the pair); the pair index runs fastest.
__device__ __forceinline__ void pair_unit(int tile, const int* prefix, const int* offs,
                                          const int* cnts, int E, int& e, int& nt, int& row0) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  e = lo;
  const int r = tile - prefix[e];
  const int mpairs = full_pairs(cnts[e]);
  nt = r / mpairs;
  row0 = offs[e] + (r - nt * mpairs) * PM;
}

// MODE 0: w13 + GLU + MXFP8 requant of h (scales of h in layout HSL);
// MODE 1: w2 -> bf16. A4: MXFP4 activations and kind::mxf4 (MODE 0 only).
// tmap_a: activation codes (128-row boxes); tmap_b: BOXED weight codes;
// tmap_asf / tmap_bsf: the TILED scale arrays as rows of 128 bytes, boxes of
// 4 rows (one 512-byte atom).
template <int MODE, bool A4, int HSL>
__global__ void __launch_bounds__(kThreads, 1)
    token_pair_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                           const __grid_constant__ CUtensorMap tmap_b,
                           const __grid_constant__ CUtensorMap tmap_asf,
                           const __grid_constant__ CUtensorMap tmap_bsf, const PairParams p) {
  static_assert(!A4 || MODE == 0, "the A4W4 path is stage 1 only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* total_holder = reinterpret_cast<int*>(smem + kOffMisc + 8);
  int* prefix = reinterpret_cast<int*>(smem + kOffSched);
  int* offs = prefix + (kMaxE + 1);
  int* cnts = offs + (kMaxE + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int KT = p.K / (A4 ? BK4 : BK);   // pipeline stages per tile
  const int KT128 = p.K / 128;            // 128-input tiles of the scale and weight layouts
  const uint32_t rank = cluster_rank();
  const int pair0 = int(blockIdx.x) >> 1, pairs = int(gridDim.x) >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);    // first CTA: its producer's expect-tx (both CTAs' bytes)
      mbar_init(&empty[s], 1);   // the pair's multicast commit
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 16);   // one arrival per epilogue warp of both CTAs (first CTA)
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
  if (warp == 0) {  // tile prefix over experts: lane owns a run of experts
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int s = 0;
    bool bad = false;  // groups must be multiples of BM rows holding their counts
    for (int e = e0; e < e1; ++e) {
      const int rows = offs[e + 1] - offs[e];
      bad |= rows < 0 || rows % BM != 0 || cnts[e] < 0 || cnts[e] > rows;
      s += max(0, full_pairs(cnts[e])) * p.n_tiles;
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
      run += max(0, full_pairs(cnts[e])) * p.n_tiles;
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
    // The whole warp runs the loop (converged); the elected lane issues. Both
    // CTAs load their halves; the bytes complete on the first CTA's barrier.
    const bool leader = elect_one_sync();
    uint32_t stage = 0, phase = 0;
    uint32_t filled = 0, last_parity = 0;  // per-stage bits of the last fill
    bool failed = false;
    for (int unit = pair0; unit < total && !failed; unit += pairs) {
      int e, nt, row0;
      pair_unit(unit, prefix, offs, cnts, E, e, nt, row0);
      const int arow = row0 + int(rank) * BM;   // this CTA's first token row
      // this CTA's weight rows (row tile of 128) and the tile's two weight tiles
      int64_t b_rt, b_rt0, b_rt1;
      if (MODE == 0) {
        b_rt0 = (int64_t(e) * 2 * p.I + int64_t(nt) * 128) >> 7;   // gate rows
        b_rt1 = b_rt0 + (p.I >> 7);                                 // up rows
      } else {
        b_rt0 = (int64_t(e) * p.d + int64_t(nt) * BN) >> 7;
        b_rt1 = b_rt0 + 1;
      }
      b_rt = rank == 0 ? b_rt0 : b_rt1;
      for (int kt = 0; kt < KT; ++kt) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag)) {
          failed = true;
          break;
        }
        if (leader) {
          uint8_t* sa = smem + kOffA + stage * A_BYTES;
          uint8_t* sb = smem + kOffB + stage * B_BYTES;
          uint8_t* ssfa = smem + kOffSfa + stage * SFA_BYTES;
          uint8_t* ssfb = smem + kOffSfb + stage * SFB_BYTES;
          const uint32_t bar = peer_addr(&full[stage], 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2u * (A4 ? kStageTxA4 : kStageTx));
          const int32_t a_atom = (arow >> 7) * KT128;   // first scale atom of the row tile
          if (A4) {
            // packed activations: one 128-byte box row = 256 inputs; weights:
            // this CTA's boxes of both 128-input halves (64-byte swizzle);
            // scales of both halves (adjacent atoms)
            tma_load_2d_pair(sa, &tmap_a, bar, kt * 128, arow);
            tma_load_2d_pair(ssfa, &tmap_asf, bar, 0, (a_atom + 2 * kt) * 4);
            tma_load_2d_pair(ssfa + SF_ATOM, &tmap_asf, bar, 0, (a_atom + 2 * kt + 1) * 4);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_2d_pair(sb + h * B_BOX, &tmap_b, bar, 0, boxed_row(b_rt, 2 * kt + h, KT128));
            // weight scales of all 256 rows: [gate h0, gate h1, up h0, up h1]
            tma_load_2d_pair(ssfb, &tmap_bsf, bar, 0, int32_t((b_rt0 * KT128 + 2 * kt) * 4));
            tma_load_2d_pair(ssfb + SF_ATOM, &tmap_bsf, bar, 0,
                             int32_t((b_rt0 * KT128 + 2 * kt + 1) * 4));
            tma_load_2d_pair(ssfb + 2 * SF_ATOM, &tmap_bsf, bar, 0,
                             int32_t((b_rt1 * KT128 + 2 * kt) * 4));
            tma_load_2d_pair(ssfb + 3 * SF_ATOM, &tmap_bsf, bar, 0,
                             int32_t((b_rt1 * KT128 + 2 * kt + 1) * 4));
          } else {
            tma_load_2d_pair(sa, &tmap_a, bar, kt * BK, arow);
            tma_load_2d_pair(ssfa, &tmap_asf, bar, 0, (a_atom + kt) * 4);
            tma_load_2d_pair(sb, &tmap_b, bar, 0, boxed_row(b_rt, kt, KT128));
            tma_load_2d_pair(ssfb, &tmap_bsf, bar, 0, int32_t((b_rt0 * KT128 + kt) * 4));
            tma_load_2d_pair(ssfb + SF_ATOM, &tmap_bsf, bar, 0, int32_t((b_rt1 * KT128 + kt) * 4));
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
    // drain: every copy of both CTAs has landed before either CTA may exit
    // (the first CTA's full barriers count them all; the second CTA waits for
    // the first at the final cluster barrier)
    if (rank == 0)
      for (int s = 0; s < STAGES; ++s)
        if ((filled >> s) & 1u)
          if (!mbar_wait_warp(&full[s], (last_parity >> s) & 1u, nullptr) && leader)
            set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
  } else if (warp == 1 && rank == 0) {
    // ---------------------------------------------------------- MMA issuer
    // Converged warp; the elected lane issues every tcgen05 instruction (a
    // commit tracks the operations of the thread that issues it).
    const bool leader = elect_one_sync();
    const uint32_t idesc = A4 ? idesc_mxf8f6f4(kFmtMxf4E2M1, kFmtMxf4E2M1, PM, BN)
                              : idesc_mxf8f6f4(kFmtE4M3, kFmtE2M1, PM, BN);
    uint32_t stage = 0, phase = 0, acc_phase = 0;
    bool failed = false;
    for (int unit = pair0; unit < total && !failed; unit += pairs) {
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
        if (leader && A4) {
          const uint32_t sa = smem_u32(smem + kOffA + stage * A_BYTES);
          const uint32_t sb = smem_u32(smem + kOffB + stage * B_BYTES);
          const uint32_t ssfa = smem_u32(smem + kOffSfa + stage * SFA_BYTES);
          const uint32_t ssfb = smem_u32(smem + kOffSfb + stage * SFB_BYTES);
          // tensor-memory scale slots: A half h at +4h; B half h at +8+8h
          // (gate rows = MMA N rows 0..127), +12+8h (up rows, N rows 128..255)
          const uint32_t sfa_t = tmem_base + kSfCol + stage * 32;
          const uint32_t sfb_t = sfa_t + 8;
          tc_cp2(sfa_t, desc_sf_block(ssfa));
          tc_cp2(sfa_t + 4, desc_sf_block(ssfa + SF_ATOM));
          tc_cp2(sfb_t, desc_sf_block(ssfb));
          tc_cp2(sfb_t + 4, desc_sf_block(ssfb + 2 * SF_ATOM));
          tc_cp2(sfb_t + 8, desc_sf_block(ssfb + SF_ATOM));
          tc_cp2(sfb_t + 12, desc_sf_block(ssfb + 3 * SF_ATOM));
          const uint64_t adesc = desc_sw128_kmajor(sa);
#pragma unroll
          for (int j = 0; j < BK4 / 64; ++j) {
            // MMA j: inputs [64j, 64j+64) of the stage = 32 bytes of each row;
            // A: +32j bytes in its 128-byte swizzle row; B: half j/2, +32(j%2)
            // bytes in the 64-byte rows; scale bytes 2(j%2), 2(j%2)+1 of half j/2
            const int h = j >> 1;
            const uint64_t bdesc = desc_sw64_kmajor(sb + uint32_t(h) * B_BOX);
            tc_mma_mxf4_2(tmem_base + kAccCol, adesc + uint64_t(2 * j),
                          bdesc + uint64_t(2 * (j & 1)),
                          idesc_with_sf_id(idesc, uint32_t(2 * (j & 1))), sfa_t + 4 * h,
                          sfb_t + 8 * h, (kt > 0 || j > 0) ? 1u : 0u);
          }
        } else if (leader) {
          const uint32_t sa = smem_u32(smem + kOffA + stage * A_BYTES);
          const uint32_t sb = smem_u32(smem + kOffB + stage * B_BYTES);
          const uint32_t ssfa = smem_u32(smem + kOffSfa + stage * SFA_BYTES);
          const uint32_t ssfb = smem_u32(smem + kOffSfb + stage * SFB_BYTES);
          const uint32_t sfa_t = tmem_base + kSfCol + stage * 32;
          const uint32_t sfb_t = sfa_t + 4;
          tc_cp2(sfa_t, desc_sf_block(ssfa));
          tc_cp2(sfb_t, desc_sf_block(ssfb));
          tc_cp2(sfb_t + 4, desc_sf_block(ssfb + SF_ATOM));
          const uint64_t adesc = desc_sw128_kmajor(sa);
          const uint64_t bdesc = desc_sw128_kmajor(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            // +32 bytes along K inside the swizzle atom = +2 in the address field
            tc_mma_mx2(tmem_base + kAccCol, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk),
                       idesc_with_sf_id(idesc, uint32_t(kk)), sfa_t, sfb_t,
                       (kt > 0 || kk > 0) ? 1u : 0u);
          }
        }
        // the stage is free in both CTAs once these MMAs have read it
        if (leader) tc_commit2_mc(&empty[stage], uint16_t(0x3));
        __syncwarp();
        if (++stage == STAGES) {
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
    // Eight warps, two per tensor-memory lane quarter (a warp may only access
    // quarter warp%4); the two split the tile's columns in halves. A warp
    // copies its 32 rows x 128 accumulator columns into registers, hands the
    // accumulator back to the MMA issuer at once, and finishes the math and
    // the stores while the next tile accumulates.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t acc_empty_pair = peer_addr(acc_empty, 0);
    uint32_t acc_phase = 0;
    for (int unit = pair0; unit < total; unit += pairs) {
      int e, nt, row0;
      pair_unit(unit, prefix, offs, cnts, E, e, nt, row0);
      const int arow = row0 + int(rank) * BM;
      bool ok = mbar_wait(acc_full, acc_phase, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
      tc_fence_after();
      const int64_t row = int64_t(arow) + q * 32 + lane;
      const uint32_t tq = tmem_base + kAccCol + (uint32_t(q * 32) << 16);
      // MODE 0: gate columns [64 half, 64 half + 64) and the matching up
      // columns (+128). MODE 1: output columns [128 half, 128 half + 128).
      const bool active = MODE == 0 || nt * BN + half * 128 < p.d;
      // rows past the expert's tokens are padding: not stored
      const bool live = arow - offs[e] + q * 32 + lane < cnts[e];
      uint32_t v[4][32];
      if (MODE == 0) {
        tmem_ld_32x32b_x32(tq + 64 * half, v[0]);
        tmem_ld_32x32b_x32(tq + 64 * half + 32, v[1]);
        tmem_ld_32x32b_x32(tq + 128 + 64 * half, v[2]);
        tmem_ld_32x32b_x32(tq + 128 + 64 * half + 32, v[3]);
      } else if (active) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tq + 128 * half + 32 * c, v[c]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {   // the whole warp has read its part
        if (rank == 0) mbar_arrive(acc_empty);
        else mbar_arrive_remote_relaxed(acc_empty_pair);
      }
      acc_phase ^= 1u;
      if (MODE == 0) {
        uint32_t sword = 0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float h[32];
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float gf = __uint_as_float(v[c][i]);
            const float uf = __uint_as_float(v[2 + c][i]);
            h[i] = __fdividef(gf * uf, 1.0f + __expf(-gf));  // silu(g) * u
            amax = fmaxf(amax, fabsf(h[i]));
          }
          const int code = mx_scale_code(amax);
          const float m = mx_scale_mult(code);
          uint4 o[2];
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            o[w].x = e4m3x4(h[16 * w + 0], h[16 * w + 1], h[16 * w + 2], h[16 * w + 3], m);
            o[w].y = e4m3x4(h[16 * w + 4], h[16 * w + 5], h[16 * w + 6], h[16 * w + 7], m);
            o[w].z = e4m3x4(h[16 * w + 8], h[16 * w + 9], h[16 * w + 10], h[16 * w + 11], m);
            o[w].w = e4m3x4(h[16 * w + 12], h[16 * w + 13], h[16 * w + 14], h[16 * w + 15], m);
          }
          if (live) {
            uint4* dst = reinterpret_cast<uint4*>(p.out_q + row * p.I + int64_t(nt) * 128 +
                                                  (2 * half + c) * 32);
            if (p.out32) {
              st_global_32B(dst, o[0].x, o[0].y, o[0].z, o[0].w, o[1].x, o[1].y, o[1].z, o[1].w);
            } else {
              dst[0] = o[0];
              dst[1] = o[1];
            }
          }
          sword |= uint32_t(code) << (8 * c);
        }
        if (live) {
          const int64_t b = int64_t(nt) * 4 + 2 * half;   // first of the two 32-blocks
          const int64_t off = HSL == kScalesGroup32 ? group32_sf_offset(row, b, p.I)
                                                    : tiled_sf_offset(row, b, p.I);
          *reinterpret_cast<uint16_t*>(p.out_sf + off) = uint16_t(sword);
        }
      } else if (active && live) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[c][2 * i]),
                                                            __uint_as_float(v[c][2 * i + 1]));
            o[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          uint4* dst = reinterpret_cast<uint4*>(p.out_bf16 + row * p.d + nt * BN + 128 * half +
                                                32 * c);
          if (p.out32) {
            st_global_32B(dst, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
            st_global_32B(dst + 2, o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15]);
          } else {
#pragma unroll
            for (int w = 0; w < 4; ++w)
              dst[w] = make_uint4(o[4 * w], o[4 * w + 1], o[4 * w + 2], o[4 * w + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA of a pair frees tensor memory or exits while the other may
  // still arrive on its barriers or use its shared memory
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc2(tmem_base, kTmemCols);
}

template <int MODE, bool A4 = false, int HSL = kScalesTiled128>
cudaError_t launch_pairs(const PairParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                         const CUtensorMap& tasf, const CUtensorMap& tbsf, cudaStream_t st) {
  auto kernel = token_pair_gemm_kernel<MODE, A4, HSL>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemBytes));
  if (err != cudaSuccess) return err;
  // units: at most one per 256 grouped rows per n-tile
  const int64_t max_units = (p.rows_capacity / PM) * p.n_tiles;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(unsigned(sms));
  int clusters = 0;
  err = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
  if (err != cudaSuccess) return err;
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  const int64_t pairs = max_units < clusters ? (max_units > 0 ? max_units : 1) : clusters;
  return launch_ex(true, kernel, dim3(unsigned(2 * pairs)), dim3(kThreads), kSmemBytes, st, 2, ta,
                   tb, tasf, tbsf, p);
}

}  // namespace

cudaError_t launch_token_pairs_w13_glu(const uint8_t* xq, const uint8_t* xs, const int* counts,
                                       const int* offsets, int E, int d, int I, const uint8_t* w13,
                                       const uint8_t* w13_sf, uint8_t* hq, uint8_t* hs,
                                       int64_t rows_capacity, int* status, cudaStream_t st) {
  CUtensorMap ta, tb, tasf, tbsf;
  if (!encode_operand(&ta, xq, false, d, rows_capacity, BM) ||
      !encode_boxed_weights(&tb, w13, int64_t(E) * 2 * I, d) ||
      !encode_scale_atoms(&tasf, xs, rows_capacity * (d / 32)) ||
      !encode_scale_atoms(&tbsf, w13_sf, int64_t(E) * 2 * I * (d / 32)))
    return cudaErrorInvalidValue;
  PairParams p{};
  p.counts = counts;
  p.offsets = offsets;
  p.E = E;
  p.K = d;
  p.I = I;
  p.d = d;
  p.n_tiles = I / 128;
  p.rows_capacity = rows_capacity;
  p.out_q = hq;
  p.out_sf = hs;
  p.status = status;
  p.out32 = (reinterpret_cast<uintptr_t>(hq) & 31u) == 0;
  return launch_pairs<0>(p, ta, tb, tasf, tbsf, st);
}

cudaError_t launch_token_pairs_w13_glu_a4w4(const uint8_t* xq, const uint8_t* xs,
                                            const int* counts, const int* offsets, int E, int d,
                                            int I, const uint8_t* w13, const uint8_t* w13_sf,
                                            uint8_t* hq, uint8_t* hs, int hs_layout,
                                            int64_t rows_capacity, int* status, cudaStream_t st) {
  CUtensorMap ta, tb, tasf, tbsf;
  // packed activations: d/2 bytes per row, 128-byte boxes of 128 rows
  if (!encode_operand(&ta, xq, false, d / 2, rows_capacity, BM) ||
      !encode_boxed_weights_packed(&tb, w13, int64_t(E) * 2 * I, d) ||
      !encode_scale_atoms(&tasf, xs, rows_capacity * (d / 32)) ||
      !encode_scale_atoms(&tbsf, w13_sf, int64_t(E) * 2 * I * (d / 32)))
    return cudaErrorInvalidValue;
  PairParams p{};
  p.counts = counts;
  p.offsets = offsets;
  p.E = E;
  p.K = d;
  p.I = I;
  p.d = d;
  p.n_tiles = I / 128;
  p.rows_capacity = rows_capacity;
  p.out_q = hq;
  p.out_sf = hs;
  p.status = status;
  p.out32 = (reinterpret_cast<uintptr_t>(hq) & 31u) == 0;
  if (hs_layout == kScalesGroup32)
    return launch_pairs<0, true, kScalesGroup32>(p, ta, tb, tasf, tbsf, st);
  return launch_pairs<0, true, kScalesTiled128>(p, ta, tb, tasf, tbsf, st);
}

cudaError_t launch_token_pairs_w2(const uint8_t* hq, const uint8_t* hs, const int* counts,
                                  const int* offsets, int E, int I, int d, const uint8_t* w2,
                                  const uint8_t* w2_sf, uint16_t* yp, int64_t rows_capacity,
                                  int* status, cudaStream_t st) {
  CUtensorMap ta, tb, tasf, tbsf;
  if (!encode_operand(&ta, hq, false, I, rows_capacity, BM) ||
      !encode_boxed_weights(&tb, w2, int64_t(E) * d, I) ||
      !encode_scale_atoms(&tasf, hs, rows_capacity * (I / 32)) ||
      !encode_scale_atoms(&tbsf, w2_sf, int64_t(E) * d * (I / 32)))
    return cudaErrorInvalidValue;
  PairParams p{};
  p.counts = counts;
  p.offsets = offsets;
  p.E = E;
  p.K = I;
  p.I = I;
  p.d = d;
  p.n_tiles = (d + BN - 1) / BN;
  p.rows_capacity = rows_capacity;
  p.out_bf16 = yp;
  p.status = status;
  p.out32 = (reinterpret_cast<uintptr_t>(yp) & 31u) == 0;
  return launch_pairs<1>(p, ta, tb, tasf, tbsf, st);
}

}  // namespace moe
