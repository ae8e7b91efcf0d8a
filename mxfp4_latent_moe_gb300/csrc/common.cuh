// Device helpers shared by the libmoe kernels (sm_103a): status word, bounded
// waits, the MX quantisation rule, and inline-PTX wrappers for mbarrier, TMA
// (cp.async.bulk[.tensor]) and the 5th-generation tensor cores (tcgen05).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Device status word (first 4 bytes of every workspace). The first error wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. The layer's latency-bound kernels are
// launched with programmatic stream serialisation (launch_ex): a kernel may
// start while the previous one in the stream is still running. Each kernel lets its successor launch
// as soon as it starts (pdl_trigger), and waits for its predecessor to finish
// and its writes to be visible (pdl_wait) before it touches memory that a
// predecessor may write or read; only set-up (barriers, tensor memory,
// shared memory) runs before the wait. Both are no-ops for a kernel launched
// without the attribute.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch, with programmatic stream serialisation when `pdl` (the layer's
// latency-bound launches: the GEMMs and the decode-sized small kernels; the
// prefill-sized small kernels measured slightly faster without it) and a
// cluster of cluster_x CTAs along x when cluster_x > 1.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                             size_t smem, cudaStream_t st, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = unsigned(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, args...);
  return err != cudaSuccess ? err : cudaGetLastError();
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Every spin-wait in these kernels gives up after this long and records
// MOE_ERR_DEVICE_TIMEOUT instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// ---------------------------------------------------------------------------
// MX rule (OCP MX v1.0) for MXFP8 = E4M3 elements + one E8M0 scale per 32.
// ---------------------------------------------------------------------------

// Scale code clamp(floor(log2(amax)) - EMAX + 127, 0, 254); 0 for amax == 0.
// EMAX is the exponent of the element format's largest power of two: 8 for
// E4M3 (MXFP8), 2 for E2M1 (MXFP4). floor(log2) is read exactly from the fp32
// bit pattern (normal or subnormal).
template <int EMAX = 8>
__device__ __forceinline__ int mx_scale_code(float amax) {
  const uint32_t b = __float_as_uint(amax);
  if (b == 0u) return 0;
  const int field = int(b >> 23) & 0xFF;
  const int fl = field ? field - 127 : (31 - __clz(int(b))) - 149;
  const int code = fl - EMAX + 127;
  return code < 0 ? 0 : (code > 254 ? 254 : code);
}

// 2^(127 - code) as an fp32 (exact for code in [0, 253]; finite fp32 data
// never gives a code above 246).
__device__ __forceinline__ float mx_scale_mult(int code) {
  return __uint_as_float(uint32_t(254 - code) << 23);
}

// Two fp32 -> two E4M3 codes (a in the low byte): round to nearest even,
// saturate to +-448. Values far below the smallest subnormal are sent as a
// signed zero so the sign of zero results never depends on the converter's
// handling of fp32 subnormal inputs.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  a = fabsf(a) < 0x1p-11f ? copysignf(0.0f, a) : a;
  b = fabsf(b) < 0x1p-11f ? copysignf(0.0f, b) : b;
  return uint32_t(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Two fp32 -> two E2M1 codes in one byte (a in the low nibble): round to
// nearest even, saturate to +-6. Magnitudes below 0.25 round to zero anyway;
// they are sent as a signed zero so the sign of zero results never depends on
// the converter's handling of tiny or subnormal inputs.
__device__ __forceinline__ uint32_t e2m1x2(float a, float b) {
  a = fabsf(a) < 0.25f ? copysignf(0.0f, a) : a;
  b = fabsf(b) < 0.25f ? copysignf(0.0f, b) : b;
  return uint32_t(__nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest));
}

// Four scaled values -> four E4M3 codes packed little-endian.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d, float m) {
  return e4m3x2(a * m, b * m) | (e4m3x2(c * m, d * m) << 16);
}

// Byte offset of the scale of row r, 32-block b in the TILED scale layout of
// an operand with K inputs per row (K % 128 == 0): one 512-byte atom per 128
// rows x 128 inputs; inside it row r sits at lane r%32, column (r/32)%4, byte
// b%4 of the tensor-core scale-factor copy.
__host__ __device__ __forceinline__ int64_t tiled_sf_offset(int64_t r, int64_t b, int64_t K) {
  return ((r >> 7) * (K >> 7) + (b >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3);
}

// Byte offset of the scale of row r, 32-block b in the GROUP32 scale layout
// (activations of the weight-tile GEMMs): one 512-byte block per 32 rows x
// 128 inputs, row r's four scale codes at bytes (r%32)*16 .. +3, the other
// twelve bytes of each 16 unused. A tcgen05.cp of the block puts the 32 rows
// in tensor-memory column 0.
__host__ __device__ __forceinline__ int64_t group32_sf_offset(int64_t r, int64_t b, int64_t K) {
  return ((r >> 5) * (K >> 7) + (b >> 2)) * 512 + (r & 31) * 16 + (b & 3);
}

enum ScaleLayout : int { kScalesTiled128 = 0, kScalesGroup32 = 1 };

// BOXED weight layout (moe_prepack_weights): a packed E2M1 matrix of R rows x
// K inputs stored as contiguous 8 KB boxes of 128 rows x 128 inputs, box
// (row tile rt, input tile kt) at index rt*(K/128) + kt, rows of 64 bytes
// inside. Seen by TMA as a 2-D tensor of 64-byte rows; this is the row
// coordinate of box (rt, kt).
__host__ __device__ __forceinline__ int32_t boxed_row(int64_t rt, int kt, int KT) {
  return int32_t((rt * KT + kt) * 128);
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}

// Waits until the phase with the given parity has completed. Gives up (returns
// false) after limit_ns, or early when *abort becomes non-zero.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u) {
      if (abort && *abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

// Warp-uniform form of mbar_wait for a converged warp: every lane polls and
// the warp agrees on the outcome (false if any lane gave up).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               uint64_t limit_ns = kWaitLimitNs) {
  const bool ok = mbar_wait(bar, parity, abort, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// One lane of a converged warp (elect.sync). The TMA producer and the MMA
// issuer keep their warps converged and issue from the elected lane: on
// sm_103a tcgen05 and mbarrier instructions from a warp whose other lanes are
// parked at a divergence point issue several times slower.
__device__ __forceinline__ bool elect_one_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0u;
}

// Orders this thread's earlier generic-proxy shared-memory writes before its
// later async-proxy operations (TMA, tcgen05.cp) on shared memory.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Token tiles of one expert (128 rows each, "m-tiles"): an expert with an
// even number of them, or with at least kPairMinMtiles, runs its full pairs
// of m-tiles as CTA pairs (one 256-row MMA over two SMs) and only an odd last
// one in the single-CTA kernel; any other expert (1, 3, 5 or 7 m-tiles) runs
// whole in the single-CTA kernel. An odd last m-tile runs in a second launch
// that streams the expert's weights again: with five m-tiles per expert
// (uniform routing at T = 32,768) that cost more than the pairs saved.
constexpr int kPairMinMtiles = 8;
__device__ __forceinline__ bool runs_as_pairs(int mtiles) {
  return mtiles >= kPairMinMtiles || (mtiles >= 2 && (mtiles & 1) == 0);
}

// One 32-byte store (the address 32-byte aligned). A warp's 32 rows then
// write whole 32-byte sectors; with 16-byte stores, which leave each sector
// half written per request, the GEMM epilogues' stores cost the stage-2
// kernel about 1.7 times as much time.
__device__ __forceinline__ void st_global_32B(void* dst, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t a4, uint32_t a5, uint32_t a6,
                                              uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a0),
               "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

// ---------------------------------------------------------------------------
// TMA / bulk copies (global -> shared, completion counted on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, copies, loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives once on `bar` when every tcgen05 operation this thread issued
// before it has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// D(tmem) (+)= A(smem) x B(smem)^T with per-32 E8M0 scale factors in tmem.
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Copies a 32-row x 16-byte block from shared memory into tensor-memory
// columns [taddr, taddr+4), replicated to all four 32-lane sub-partitions.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t src_desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc)
               : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// Each thread of the warp reads 16 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): K-major operand written by
// TMA with 128-byte swizzle, rows of 128 bytes, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128_kmajor(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);  // start address
  d |= uint64_t(1) << 16;                  // leading byte offset (unused here)
  d |= uint64_t(1024 >> 4) << 32;          // stride byte offset: next 8-row atom
  d |= uint64_t(1) << 46;                  // descriptor version (tcgen05)
  d |= uint64_t(2) << 61;                  // 128-byte swizzle
  return d;
}

// Same for a K-major operand with 64-byte rows and 64-byte swizzle (8-row
// atoms 512 bytes apart): the packed E2M1 weight boxes of the A4W4 GEMM.
__device__ __forceinline__ uint64_t desc_sw64_kmajor(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);  // start address
  d |= uint64_t(1) << 16;                  // leading byte offset (unused here)
  d |= uint64_t(512 >> 4) << 32;           // stride byte offset: next 8-row atom
  d |= uint64_t(1) << 46;                  // descriptor version (tcgen05)
  d |= uint64_t(4) << 61;                  // 64-byte swizzle
  return d;
}

// Descriptor of a scale-factor block: 32 rows x 16 bytes, no swizzle, 8-row
// core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t desc_sf_block(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(128 >> 4) << 32;
  d |= uint64_t(1) << 46;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::mxf8f6f4 with E8M0 scales:
// A/B formats (E4M3 = 0, E2M1 = 5), both K-major, dense, shape M x N.
// The scale-factor ids (bits 4-5 for B, 29-30 for A) pick the byte of the
// 32-bit scale column, i.e. which 32-input block of the stage the MMA uses.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4(uint32_t a_fmt, uint32_t b_fmt, int M,
                                                      int N) {
  return (a_fmt << 7) | (b_fmt << 10) | (uint32_t(N >> 3) << 17) | (1u << 23) |
         (uint32_t(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_with_sf_id(uint32_t idesc, uint32_t id) {
  return idesc | (id << 4) | (id << 29);
}

constexpr uint32_t kFmtE4M3 = 0;
constexpr uint32_t kFmtE2M1 = 5;
// kind::mxf4 takes only E2M1 operands, coded 1 in its instruction descriptor
// (same field positions as kind::mxf8f6f4; scale_vec::2X, UE8M0 scales: each
// MMA of K = 64 reads two scale bytes per row starting at the byte its
// scale-factor id selects, 0 or 2).
constexpr uint32_t kFmtMxf4E2M1 = 1;

// D(tmem) (+)= A(smem) x B(smem)^T, both packed E2M1 (K = 64 per MMA), two
// E8M0 scale factors per row per MMA from tensor memory.
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// ---------------------------------------------------------------------------
// 2-CTA clusters and the tcgen05 cta_group::2 forms (an MMA spread over the
// tensor cores of a pair of SMs; both CTAs allocate tensor memory together).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
          "memory");
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// 2-D TMA load into this CTA's shared memory whose bytes complete on the
// mbarrier at cluster address `bar` (this CTA's or its pair partner's).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster with no memory ordering
// (the arriving thread orders what it must by other means, e.g. completed
// tensor-memory loads); a release at cluster scope costs far more latency.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// try_wait with acquire at cluster scope (the phase may complete by arrivals
// from the other CTA of the pair).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}
__device__ __forceinline__ bool mbar_wait_cluster_warp(uint64_t* bar, uint32_t parity,
                                                       volatile int* abort) {
  bool ok = mbar_try_wait_cluster(bar, parity);
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
      if (mbar_try_wait_cluster(bar, parity)) {
        ok = true;
        break;
      }
      if ((i & 31u) == 0u) {
        if (abort && *abort) break;
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void tmem_alloc2(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Copies a 32-row x 16-byte scale block of each CTA's shared memory into its
// own tensor memory at columns [taddr, taddr+4).
__device__ __forceinline__ void tc_cp2(uint32_t taddr, uint64_t src_desc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc)
               : "memory");
}
// D (both CTAs' tensor memory) (+)= A (128 rows in each CTA) x B (N/2 rows in
// each CTA)^T with per-32 E8M0 scales.
__device__ __forceinline__ void tc_mma_mx2(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
// Arrives once on the mbarrier at the same offset in every CTA of `mask` when
// all tcgen05 operations the thread issued before it have completed.
__device__ __forceinline__ void tc_commit2_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// The kind::mxf4 MMA (both operands packed E2M1, K = 64) over a pair of SMs.
__device__ __forceinline__ void tc_mma_mxf4_2(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem,
                                              uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}


}  // namespace moe
