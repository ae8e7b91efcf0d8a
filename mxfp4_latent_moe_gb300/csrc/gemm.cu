// Grouped GEMMs of the routed experts on tcgen05 block-scaled tensor cores.
//
// The pages' layer runs the routed experts through a grouped-MoE kernel with
// MXFP4 weights and an FP8 second stage ("Kimi K3.1 Pro on AMD Instinct GPUs",
// "The MXFP4 latent MoE on FlyDSL"; shapes from the Experts row of "Kimi K3.1
// Pro at a glance": gate/up 3,584 -> 2 x 3,072, down 3,072 -> 3,584). Here:
//
//   stage 1 (MODE 0): [gate | up] = Xq . [W1 | W3]^T, h = silu(gate) * up,
//                     h -> MXFP8 (E4M3 + E8M0 per 32) in the epilogue
//   stage 2 (MODE 1): Yp = Hq . W2^T -> bf16
//
// Both are D[128 x 256] += A[128 x 128] . B[256 x 128]^T per pipeline stage,
// with A = MXFP8 activations (E4M3) and B = MXFP4 weights (E2M1), one E8M0
// scale per 32 inputs on each side, via tcgen05.mma kind::mxf8f6f4
// (4 MMAs of K = 32 per stage, fp32 accumulators in tensor memory).
//
// CTA organisation (persistent, one CTA per SM, 320 threads):
//   warp 0      TMA producer: A box 128x128 bytes, B box(es) of E2M1 expanded
//               by TMA to one byte slot per element (16U4_ALIGN16B), both
//               128-byte swizzled; the stage's scale atoms by bulk copy.
//   warp 1      tensor-memory allocator + MMA issuer: copies the stage's scale
//               atoms into tensor memory (tcgen05.cp), issues the 4 MMAs,
//               frees the smem stage with tcgen05.commit.
//   Warps 0 and 1 run their loops converged (all lanes wait, one elected lane
//   issues); a loop run by one lane with the rest parked issues its tcgen05
//   and mbarrier instructions several times slower.
//   warps 2-9   epilogue: tcgen05.ld of the accumulator (one row and half the
//               columns per thread) straight into registers, release of the
//               accumulator, then the fused GLU + MX requant (MODE 0) or the
//               bf16 conversion (MODE 1) overlapped with the next tile's MMAs.
// Tiles are (expert, n-tile, m-tile) with the m-tile fastest, so CTAs running
// at the same time share one expert's weight tile through L2. The expert row
// offsets are read on the device: no host synchronisation.
// Both stages run as 2-CTA clusters: the pair takes n-tiles 2j and 2j + 1 of
// one (expert, m-tile), each CTA loads one 64-row half of the A tile and
// multicasts it to both, so the activations cross from L2 once per pair
// (on prefill about 10% faster stage 1 and 3-5% faster stage 2).
// In the token-tile family this kernel runs the m-tiles of the experts with
// 1, 3, 5 or 7 of them and the odd last m-tile of the heavier odd ones
// (`tail_only`); every other full pair of m-tiles runs before it as one
// 256-row MMA over two SMs (gemm_token_pair.cu). A stage here writes 49.5 KB
// of shared memory per 512 cycles of MMA work, near the SM's TMA ingest
// rate, so four stages cover the copies' latency only in part (the tensor
// pipe runs about three quarters busy); the pair's stages need two thirds of
// that.
// Every wait is bounded; on expiry the CTA records MOE_ERR_DEVICE_TIMEOUT,
// drains its outstanding copies and tensor-core work, frees tensor memory and
// exits.
#include "internal.h"

namespace moe {

namespace {

constexpr int BM = 128;            // rows per tile (MMA M)
constexpr int BK = 128;            // inputs per pipeline stage (MXFP8 activations)
constexpr int BK4 = 256;           // inputs per pipeline stage (A4W4: MXFP4 activations)
constexpr int BN = 256;            // MMA N
constexpr int STAGES = 4;
constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;    // accumulator: columns [0, 256)
constexpr uint32_t kSfCol = 256;   // scale slots: 32 columns per stage
// A: 128 rows x 128 bytes (128 E4M3 inputs, or 256 packed E2M1 inputs).
constexpr uint32_t A_BYTES = BM * 128;
// B, MXFP8 path: TMA's 16U4_ALIGN16B expansion puts each 16 E2M1 codes (8
// packed bytes) in the low half of a 16-byte slot, so a 128-input row takes
// 128 bytes of shared memory; the mbarrier transaction count is the packed
// size, half of that. A4W4 path: four packed 8 KB boxes (gate and up rows,
// two 128-input halves), no expansion, the same 32 KB.
constexpr uint32_t B_BYTES = BN * 128;
constexpr uint32_t B_TX_BYTES = B_BYTES / 2;
constexpr uint32_t B_BOX = 8192;   // one BOXED weight box: 128 rows x 64 bytes
// scale atoms per stage: MXFP8 A 1, B 2; A4W4 A 2, B 4 (512 bytes each)
constexpr uint32_t SFA_BYTES = 1024;
constexpr uint32_t SFB_BYTES = 2048;
constexpr uint32_t kStageTx = A_BYTES + B_TX_BYTES + 512 + 1024;
constexpr uint32_t kStageTxA4 = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;

constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + STAGES * A_BYTES;
constexpr uint32_t kOffSfa = kOffB + STAGES * B_BYTES;
constexpr uint32_t kOffSfb = kOffSfa + STAGES * SFA_BYTES;
constexpr uint32_t kOffBars = kOffSfb + STAGES * SFB_BYTES;
constexpr uint32_t kNumBars = 2 * STAGES + 3;  // full[S], empty[S], acc_full, acc_empty, drain
constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
constexpr uint32_t kOffSched = kOffMisc + 16;
constexpr uint32_t kMaxE = 1024;
constexpr uint32_t kSmemBytes = kOffSched + 3 * (kMaxE + 1) * 4 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct GemmParams {
  const uint8_t* a_sf;   // TILED scales of A
  const uint8_t* b_sf;   // TILED scales of B
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
  bool tail_only;        // only each expert's odd last m-tile (the others ran as CTA pairs)
};

// ---- 2-CTA clusters: the A tile multicast to both CTAs of a pair ----------
// TMA load delivered to the same shared-memory offset (and mbarrier) in every
// CTA of `mask`.
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* map, uint64_t* bar,
                                               int32_t x, int32_t y, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "h"(mask)
      : "memory");
}
// tcgen05.commit arriving on the same mbarrier in every CTA of `mask`.
__device__ __forceinline__ void tc_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// m-tiles of an expert this launch covers: all ceil(count/BM), or with
// tail_only, for an expert that runs as CTA pairs, the last one when their
// number is odd (the full pairs before it run in the CTA-pair kernel).
__device__ __forceinline__ int expert_mtiles(int count, bool tail_only) {
  const int m = (count + BM - 1) / BM;
  return tail_only && runs_as_pairs(m) ? (m & 1) : m;
}
// The first m-tile of the expert that this launch covers.
__device__ __forceinline__ int expert_first_mtile(int count, bool tail_only) {
  const int m = (count + BM - 1) / BM;
  return tail_only && runs_as_pairs(m) ? m - 1 : 0;
}

// Tile -> (expert, n-tile, first row); the m-tile index runs fastest.
__device__ __forceinline__ void decode_tile(int tile, const int* prefix, const int* offs,
                                            const int* cnts, int E, bool tail_only, int& e,
                                            int& nt, int& row0) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  e = lo;
  const int r = tile - prefix[e];
  const int mtiles = expert_mtiles(cnts[e], tail_only);
  nt = r / mtiles;
  row0 = offs[e] + (expert_first_mtile(cnts[e], tail_only) + r - nt * mtiles) * BM;
}

// MODE 0: w13 + GLU + MXFP8 requant of h (scales of h in layout HSL);
// MODE 1: w2 -> bf16. A4: MXFP4 activations and kind::mxf4 (MODE 0 only).
// CL = 2: CTA pairs (2-CTA clusters) take n-tiles 2j and 2j + 1 of the same
// (expert, m-tile): each loads one 64-row half of the A tile and multicasts
// it to both, so each CTA reads half of A; each CTA's MMA commit frees the
// stage in both CTAs (the empty barriers count 2). With an odd number of
// n-tiles the last pair's second CTA has no n-tile: it still loads its half
// of A and consumes the stages, but issues no MMA and stores nothing.
template <int MODE, bool A4, int HSL, int CL>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
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
  const uint32_t crank = CL == 2 ? cluster_rank() : 0u;
  const int unit0 = int(blockIdx.x) / CL, units_step = int(gridDim.x) / CL;
  const int ntu = (p.n_tiles + CL - 1) / CL;   // n-tile units per expert and m-tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CL);   // each CTA of the pair frees the stage
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 8);   // one arrival per epilogue warp
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
    bool bad = false;  // groups must be multiples of BM rows holding their counts
    for (int e = e0; e < e1; ++e) {
      const int rows = offs[e + 1] - offs[e];
      bad |= rows < 0 || rows % BM != 0 || cnts[e] < 0 || cnts[e] > rows;
      s += max(0, expert_mtiles(cnts[e], p.tail_only)) * ntu;
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
      run += max(0, expert_mtiles(cnts[e], p.tail_only)) * ntu;
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
  if (CL == 2) cluster_sync_all();   // both CTAs' barriers exist before any remote arrival
  const uint32_t tmem_base = *tmem_holder;
  const int total = *total_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (converged); the elected lane issues.
    const bool leader = elect_one_sync();
    uint32_t stage = 0, phase = 0;
    uint32_t filled = 0, last_parity = 0;  // per-stage bits of the last fill
    bool failed = false;
    for (int unit = unit0; unit < total && !failed; unit += units_step) {
      int e, nu, row0;
      decode_tile(unit, prefix, offs, cnts, E, p.tail_only, e, nu, row0);
      const int nt = nu * CL + int(crank);
      const bool dummy = CL == 2 && nt >= p.n_tiles;   // pair partner without an n-tile
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
          // A: the whole tile, or this CTA's 64-row half multicast to the pair
          const int32_t ax = kt * (A4 ? 128 : BK);
          auto load_a = [&]() {
            if (CL == 2)
              tma_load_2d_mc(sa + crank * (A_BYTES / 2), &tmap_a, &full[stage], ax,
                             row0 + int(crank) * (BM / 2), uint16_t(0x3));
            else
              tma_load_2d(sa, &tmap_a, &full[stage], ax, row0);
          };
          if (A4) {
            // packed activations: one 128-byte box row = 256 inputs; weights:
            // the gate and up boxes of both 128-input halves, 64-byte swizzle
            const int64_t g_rt = (int64_t(e) * 2 * p.I + int64_t(nt) * 128) >> 7;
            const int64_t u_rt = g_rt + (p.I >> 7);
            mbar_arrive_expect_tx(&full[stage],
                                  A_BYTES + 1024u + (dummy ? 0u : 4u * B_BOX + 2048u));
            load_a();
            bulk_load(ssfa, p.a_sf + (int64_t(row0 >> 7) * KT128 + 2 * kt) * 512, 1024,
                      &full[stage]);
            if (!dummy) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                tma_load_2d(sb + h * 2 * B_BOX, &tmap_b, &full[stage], 0,
                            boxed_row(g_rt, 2 * kt + h, KT128));
                tma_load_2d(sb + h * 2 * B_BOX + B_BOX, &tmap_b, &full[stage], 0,
                            boxed_row(u_rt, 2 * kt + h, KT128));
              }
              bulk_load(ssfb, p.b_sf + (g_rt * KT128 + 2 * kt) * 512, 1024, &full[stage]);
              bulk_load(ssfb + 1024, p.b_sf + (u_rt * KT128 + 2 * kt) * 512, 1024,
                        &full[stage]);
            }
          } else if (MODE == 0) {
            const int64_t g_row = int64_t(e) * 2 * p.I + int64_t(nt) * 128;
            const int64_t u_row = g_row + p.I;
            mbar_arrive_expect_tx(&full[stage],
                                  A_BYTES + 512u + (dummy ? 0u : B_TX_BYTES + 1024u));
            load_a();
            bulk_load(ssfa, p.a_sf + (int64_t(row0 >> 7) * KT128 + kt) * 512, 512, &full[stage]);
            if (!dummy) {
              tma_load_2d(sb, &tmap_b, &full[stage], 0, boxed_row(g_row >> 7, kt, KT128));
              tma_load_2d(sb + B_BYTES / 2, &tmap_b, &full[stage], 0,
                          boxed_row(u_row >> 7, kt, KT128));
              bulk_load(ssfb, p.b_sf + ((g_row >> 7) * KT128 + kt) * 512, 512, &full[stage]);
              bulk_load(ssfb + 512, p.b_sf + ((u_row >> 7) * KT128 + kt) * 512, 512,
                        &full[stage]);
            }
          } else {
            const int64_t b_row = int64_t(e) * p.d + int64_t(nt) * BN;
            const bool upper = nt * BN + 128 < p.d;
            const uint32_t btx = dummy ? 0u : (upper ? B_TX_BYTES + 1024u : B_TX_BYTES / 2 + 512u);
            mbar_arrive_expect_tx(&full[stage], A_BYTES + 512u + btx);
            load_a();
            bulk_load(ssfa, p.a_sf + (int64_t(row0 >> 7) * KT128 + kt) * 512, 512, &full[stage]);
            if (!dummy) {
              tma_load_2d(sb, &tmap_b, &full[stage], 0, boxed_row(b_row >> 7, kt, KT128));
              bulk_load(ssfb, p.b_sf + ((b_row >> 7) * KT128 + kt) * 512, 512, &full[stage]);
              if (upper) {
                tma_load_2d(sb + B_BYTES / 2, &tmap_b, &full[stage], 0,
                            boxed_row((b_row >> 7) + 1, kt, KT128));
                bulk_load(ssfb + 512, p.b_sf + (((b_row >> 7) + 1) * KT128 + kt) * 512, 512,
                          &full[stage]);
              }
            }
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
    // drain: every issued copy has landed before the CTA may exit
    for (int s = 0; s < STAGES; ++s)
      if ((filled >> s) & 1u)
        if (!mbar_wait_warp(&full[s], (last_parity >> s) & 1u, nullptr) && leader)
          set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // Converged warp; the elected lane issues every tcgen05 instruction (a
    // commit tracks the operations of the thread that issues it).
    const bool leader = elect_one_sync();
    const uint32_t idesc = A4 ? idesc_mxf8f6f4(kFmtMxf4E2M1, kFmtMxf4E2M1, BM, BN)
                              : idesc_mxf8f6f4(kFmtE4M3, kFmtE2M1, BM, BN);
    uint32_t stage = 0, phase = 0, acc_phase = 0;
    bool failed = false;
    for (int unit = unit0; unit < total && !failed; unit += units_step) {
      // only the second CTA of a pair, with an odd n-tile count, has idle units
      bool dummy = false;
      if (CL == 2 && crank == 1 && (p.n_tiles & 1)) {
        int e, nu, row0;
        decode_tile(unit, prefix, offs, cnts, E, p.tail_only, e, nu, row0);
        dummy = nu * CL + int(crank) >= p.n_tiles;
      }
      if (!mbar_wait_warp(acc_empty, acc_phase ^ 1u, abort_flag)) {
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
        if (leader && dummy) {
          // no n-tile here: only free the stage (the partner reads its A half)
        } else if (leader && A4) {
          const uint32_t sa = smem_u32(smem + kOffA + stage * A_BYTES);
          const uint32_t sb = smem_u32(smem + kOffB + stage * B_BYTES);
          const uint32_t ssfa = smem_u32(smem + kOffSfa + stage * SFA_BYTES);
          const uint32_t ssfb = smem_u32(smem + kOffSfb + stage * SFB_BYTES);
          // tensor-memory scale slots: A half h at +4h; B half h at +8+8h
          // (gate rows), +12+8h (up rows = MMA rows 128..255)
          const uint32_t sfa_t = tmem_base + kSfCol + stage * 32;
          const uint32_t sfb_t = sfa_t + 8;
          tc_cp_32x128b_x4(sfa_t, desc_sf_block(ssfa));
          tc_cp_32x128b_x4(sfa_t + 4, desc_sf_block(ssfa + 512));
          tc_cp_32x128b_x4(sfb_t, desc_sf_block(ssfb));
          tc_cp_32x128b_x4(sfb_t + 4, desc_sf_block(ssfb + 1024));
          tc_cp_32x128b_x4(sfb_t + 8, desc_sf_block(ssfb + 512));
          tc_cp_32x128b_x4(sfb_t + 12, desc_sf_block(ssfb + 1536));
          const uint64_t adesc = desc_sw128_kmajor(sa);
#pragma unroll
          for (int j = 0; j < BK4 / 64; ++j) {
            // MMA j: inputs [64j, 64j+64) of the stage = 32 bytes of each row;
            // A: +32j bytes in its 128-byte swizzle row; B: half j/2, +32(j%2)
            // bytes in the 64-byte rows; scale bytes 2(j%2), 2(j%2)+1 of half j/2
            const int h = j >> 1;
            const uint64_t bdesc = desc_sw64_kmajor(sb + uint32_t(h) * 2 * B_BOX);
            tc_mma_mxf4(tmem_base + kAccCol, adesc + uint64_t(2 * j),
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
          tc_cp_32x128b_x4(sfa_t, desc_sf_block(ssfa));
          tc_cp_32x128b_x4(sfb_t, desc_sf_block(ssfb));
          tc_cp_32x128b_x4(sfb_t + 4, desc_sf_block(ssfb + 512));
          const uint64_t adesc = desc_sw128_kmajor(sa);
          const uint64_t bdesc = desc_sw128_kmajor(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            // +32 bytes along K inside the swizzle atom = +2 in the address field
            tc_mma_mx(tmem_base + kAccCol, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk),
                      idesc_with_sf_id(idesc, uint32_t(kk)), sfa_t, sfb_t,
                      (kt > 0 || kk > 0) ? 1u : 0u);
          }
        }
        // the stage is free once this CTA's MMAs have read it; in a pair the
        // commit arrives in both CTAs (each multicasts A into the other)
        if (leader) {
          if (CL == 2) tc_commit_mc(&empty[stage], uint16_t(0x3));
          else tc_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (failed) break;
      if (leader) tc_commit(acc_full);
      __syncwarp();
      acc_phase ^= 1u;
    }
    if (failed && leader) {
      *abort_flag = 1;
      set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
    }
    // drain: all issued tensor-core work is complete before tensor memory is freed
    if (leader) tc_commit(drain);
    __syncwarp();
    if (!mbar_wait_warp(drain, 0, nullptr) && leader) set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
  } else {
    // ------------------------------------------------------------ epilogue
    // Eight warps, two per tensor-memory lane quarter (a warp may only access
    // quarter warp%4); the two split the tile's columns in halves. A warp
    // copies its 32 rows x 128 accumulator columns into registers, hands the
    // accumulator back to the MMA issuer at once, and finishes the math and
    // the stores while the next tile accumulates.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint32_t acc_phase = 0;
    for (int unit = unit0; unit < total; unit += units_step) {
      int e, nu, row0;
      decode_tile(unit, prefix, offs, cnts, E, p.tail_only, e, nu, row0);
      const int nt = nu * CL + int(crank);
      const bool dummy = CL == 2 && nt >= p.n_tiles;   // warp-uniform
      bool ok = mbar_wait(acc_full, acc_phase, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
      tc_fence_after();
      const int64_t row = int64_t(row0) + q * 32 + lane;
      const uint32_t tq = tmem_base + kAccCol + (uint32_t(q * 32) << 16);
      // MODE 0: gate columns [64 half, 64 half + 64) and the matching up
      // columns (+128). MODE 1: output columns [128 half, 128 half + 128).
      const bool active = !dummy && (MODE == 0 || nt * BN + half * 128 < p.d);
      // rows past the expert's tokens are padding: not stored
      const bool live = row0 - offs[e] + q * 32 + lane < cnts[e];
      uint32_t v[4][32];
      if (MODE == 0) {   // (a pair's idle CTA reads and drops stale values)
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
      if (lane == 0) mbar_arrive(acc_empty);   // the whole warp has read its part
      acc_phase ^= 1u;
      if (MODE == 0 && active) {
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
  tc_fence_after();
  // neither CTA of a pair exits while the other may still arrive on its
  // barriers or write into its shared memory
  if (CL == 2) cluster_sync_all();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// One CTA waits on a barrier that nothing signals; the bounded wait gives up
// and records MOE_ERR_DEVICE_TIMEOUT.
__global__ void wait_timeout_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar, 0, nullptr, limit_ns)) set_status(status, MOE_ERR_DEVICE_TIMEOUT);
  }
}

// CTAs per cluster of the token-tile GEMMs (2: A-tile pairs; 1 runs the same
// kernel one CTA per tile)
constexpr int kPairCL = 2;

template <int MODE, bool A4 = false, int HSL = kScalesTiled128>
cudaError_t launch_mode(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                        cudaStream_t st) {
  constexpr int CL = kPairCL;
  auto kernel = grouped_gemm_kernel<MODE, A4, HSL, CL>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemBytes));
  if (err != cudaSuccess) return err;
  const int64_t max_units = (p.rows_capacity / BM) * ((p.n_tiles + CL - 1) / CL);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  int slots = sms;   // resident CTA groups: one CTA per SM
  if (CL > 1) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(CL * sms);
    int clusters = 0;
    err = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (err != cudaSuccess) return err;
    if (clusters <= 0) return cudaErrorInvalidConfiguration;
    slots = clusters;
  }
  const int64_t groups = max_units < slots ? (max_units > 0 ? max_units : 1) : slots;
  return launch_ex(true, kernel, dim3(unsigned(groups * CL)), dim3(kThreads), kSmemBytes, st, CL, ta,
                    tb, p);
}

}  // namespace

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// 2-D K-major operand map: dim0 = K inputs, dim1 = rows; 128-input boxes,
// 128-byte swizzle.
bool encode_operand(CUtensorMap* map, const void* base, bool e2m1, int K, int64_t rows,
                    int box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(e2m1 ? K / 2 : K)};
  const cuuint32_t box[2] = {128u, cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(map, e2m1 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Weights in the BOXED layout: 64-byte rows (128 E2M1 inputs), one 128-row
// box per (row tile, input tile), 128-byte swizzle.
bool encode_boxed_weights(CUtensorMap* map, const void* base, int64_t rows, int K) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {128u, cuuint64_t(rows / 128) * cuuint64_t(K / 128) * 128u};
  const cuuint64_t strides[1] = {64u};
  const cuuint32_t box[2] = {128u, 128u};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides,
         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same BOXED weights as packed bytes for the A4W4 GEMM: 64-byte rows
// (128 E2M1 inputs) read as UINT8 with 64-byte swizzle, no expansion.
bool encode_boxed_weights_packed(CUtensorMap* map, const void* base, int64_t rows, int K) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {64u, cuuint64_t(rows / 128) * cuuint64_t(K / 128) * 128u};
  const cuuint64_t strides[1] = {64u};
  const cuuint32_t box[2] = {64u, 128u};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A TILED scale array of `bytes` bytes as a 2-D map of 128-byte rows, boxes
// of 4 rows (one 512-byte atom), no swizzle. Rows past the array are zero
// filled, so an atom of a tile row past the groups reads as zeros.
bool encode_scale_atoms(CUtensorMap* map, const void* base, int64_t bytes) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn || bytes <= 0 || bytes % 512 != 0) return false;
  const cuuint64_t dims[2] = {128u, cuuint64_t(bytes / 128)};
  const cuuint64_t strides[1] = {128u};
  const cuuint32_t box[2] = {128u, 4u};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// The token-tile family: the full pairs of m-tiles of the experts that run
// as pairs (runs_as_pairs) on CTA pairs (gemm_token_pair.cu), then the rest
// here, one CTA per m-tile.
cudaError_t launch_gemm_w13_glu(const uint8_t* xq, const uint8_t* xs, const int* counts,
                                const int* offsets, int E, int d, int I, const uint8_t* w13,
                                const uint8_t* w13_sf, uint8_t* hq, uint8_t* hs,
                                int64_t rows_capacity, int* status, cudaStream_t st) {
  cudaError_t err = launch_token_pairs_w13_glu(xq, xs, counts, offsets, E, d, I, w13, w13_sf, hq,
                                               hs, rows_capacity, status, st);
  if (err != cudaSuccess) return err;
  CUtensorMap ta, tb;
  if (!encode_operand(&ta, xq, false, d, rows_capacity, BM / kPairCL))
    return cudaErrorInvalidValue;
  if (!encode_boxed_weights(&tb, w13, int64_t(E) * 2 * I, d)) return cudaErrorInvalidValue;
  GemmParams p{};
  p.a_sf = xs;
  p.b_sf = w13_sf;
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
  p.tail_only = true;
  return launch_mode<0>(p, ta, tb, st);
}

cudaError_t launch_gemm_w13_glu_a4w4(const uint8_t* xq, const uint8_t* xs, const int* counts,
                                     const int* offsets, int E, int d, int I, const uint8_t* w13,
                                     const uint8_t* w13_sf, uint8_t* hq, uint8_t* hs,
                                     int hs_layout, int64_t rows_capacity, int* status,
                                     cudaStream_t st) {
  cudaError_t err = launch_token_pairs_w13_glu_a4w4(xq, xs, counts, offsets, E, d, I, w13, w13_sf,
                                                    hq, hs, hs_layout, rows_capacity, status, st);
  if (err != cudaSuccess) return err;
  CUtensorMap ta, tb;
  // packed activations: d/2 bytes per row, 128-byte boxes of 128 rows
  if (!encode_operand(&ta, xq, false, d / 2, rows_capacity, BM / kPairCL))
    return cudaErrorInvalidValue;
  if (!encode_boxed_weights_packed(&tb, w13, int64_t(E) * 2 * I, d)) return cudaErrorInvalidValue;
  GemmParams p{};
  p.a_sf = xs;
  p.b_sf = w13_sf;
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
  p.tail_only = true;
  if (hs_layout == kScalesGroup32) return launch_mode<0, true, kScalesGroup32>(p, ta, tb, st);
  return launch_mode<0, true, kScalesTiled128>(p, ta, tb, st);
}

cudaError_t launch_gemm_w2(const uint8_t* hq, const uint8_t* hs, const int* counts,
                           const int* offsets, int E, int I, int d, const uint8_t* w2,
                           const uint8_t* w2_sf, uint16_t* yp, int64_t rows_capacity, int* status,
                           cudaStream_t st) {
  cudaError_t err = launch_token_pairs_w2(hq, hs, counts, offsets, E, I, d, w2, w2_sf, yp,
                                          rows_capacity, status, st);
  if (err != cudaSuccess) return err;
  CUtensorMap ta, tb;
  if (!encode_operand(&ta, hq, false, I, rows_capacity, BM / kPairCL))
    return cudaErrorInvalidValue;
  if (!encode_boxed_weights(&tb, w2, int64_t(E) * d, I)) return cudaErrorInvalidValue;
  GemmParams p{};
  p.a_sf = hs;
  p.b_sf = w2_sf;
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
  p.tail_only = true;
  return launch_mode<1>(p, ta, tb, st);
}

cudaError_t launch_wait_timeout_selftest(int* status, uint32_t limit_us, cudaStream_t st) {
  wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(status, uint64_t(limit_us) * 1000ull);
  return cudaGetLastError();
}

}  // namespace moe
