// CPU oracle for the MXFP4 latent-MoE layer. TEST INFRASTRUCTURE ONLY: the
// test suite, the smoke check and the benchmark's CPU-baseline leg load it; the
// CUDA library never does. The declarations in moe_oracle.h state what each
// function computes and which page section it follows.
//
// Everything is scalar fp64 with per-element table decodes. There is no
// blocking, fusion or reordering beyond the definitions; the only parallelism
// is std::thread over independent tokens in orc_moe_forward.

#include "moe_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Element formats (OCP Microscaling Formats (MX) v1.0, the format the pages
// name: "MXFP4 (one E8M0 scale per 32 values)" in "Kimi K3.1 Pro at a glance").
// Each table is built from the bit-field definition of its format.
// ---------------------------------------------------------------------------

// E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no inf/NaN.
double e2m1_from_fields(unsigned code) {
  const unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  double mag;
  if (e == 0) mag = std::ldexp(m / 2.0, 1 - 1);              // subnormal: 0.m * 2^(1-bias)
  else        mag = std::ldexp(1.0 + m / 2.0, int(e) - 1);   // normal: 1.m * 2^(e-bias)
  return s ? -mag : mag;
}

// E4M3 (the "fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
// S.1111.111 is NaN, no infinities.
double e4m3_from_fields(unsigned code) {
  const unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  double mag;
  if (e == 0) mag = std::ldexp(m / 8.0, 1 - 7);
  else        mag = std::ldexp(1.0 + m / 8.0, int(e) - 7);
  return s ? -mag : mag;
}

// E8M0: an unsigned biased exponent (bias 127), 0xFF is NaN.
double e8m0_from_fields(unsigned code) {
  if (code == 255) return std::numeric_limits<double>::quiet_NaN();
  return std::ldexp(1.0, int(code) - 127);
}

struct Tables {
  double e2m1[16];
  double e4m3[256];
  double e8m0[256];
  Tables() {
    for (unsigned c = 0; c < 16; ++c) e2m1[c] = e2m1_from_fields(c);
    for (unsigned c = 0; c < 256; ++c) e4m3[c] = e4m3_from_fields(c);
    for (unsigned c = 0; c < 256; ++c) e8m0[c] = e8m0_from_fields(c);
  }
};

const Tables& tables() {
  static const Tables t;
  return t;
}

constexpr double kE4M3Max = 448.0;   // largest finite E4M3 magnitude (code 0x7E)
constexpr int kE4M3Emax = 8;         // exponent of the largest E4M3 power of two
constexpr double kE2M1Max = 6.0;     // largest E2M1 magnitude (code 0x7)
constexpr int kE2M1Emax = 2;         // exponent of the largest E2M1 power of two

// MX shared-exponent scale code for a block whose largest magnitude is amax
// and whose element format has largest power of two 2^emax (OCP MX v1.0):
// clamp(floor(log2(amax)) - emax + 127, 0, 254); 0 for an all-zero block.
int mx_scale_code_for(double amax, int emax) {
  if (!(amax > 0.0)) return 0;
  int ex = 0;
  std::frexp(amax, &ex);             // amax = m * 2^ex, m in [0.5, 1)
  const int code = (ex - 1) - emax + 127;
  return std::min(254, std::max(0, code));
}

float bf16_bits_to_float(uint16_t b) {
  uint32_t u = uint32_t(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// One element of a packed E2M1 matrix [rows][K] with scales [rows][K/32].
inline double weight_value(const uint8_t* codes, const uint8_t* scales, int64_t K,
                           int64_t row, int64_t col) {
  const Tables& t = tables();
  const uint8_t byte = codes[row * (K / 2) + col / 2];
  const unsigned nib = (col & 1) ? (byte >> 4) : (byte & 0xF);
  return t.e2m1[nib] * t.e8m0[scales[row * (K / 32) + col / 32]];
}

double sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }

}  // namespace

extern "C" {

double orc_e2m1_value(uint8_t code) { return tables().e2m1[code & 0xF]; }
double orc_e4m3_value(uint8_t code) { return tables().e4m3[code]; }
double orc_e8m0_value(uint8_t code) { return tables().e8m0[code]; }

// Nearest E4M3 value by search over the finite non-negative codes 0x00..0x7E
// (their values increase with the code), ties to the even code, magnitudes
// above 448 saturate to 448. The sign bit follows the sign of v, also for 0.
uint8_t orc_e4m3_encode_rne_sat(double v) {
  const Tables& t = tables();
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  const double a = std::fabs(v);
  if (a >= kE4M3Max) return sign | 0x7E;
  unsigned lo = 0;
  while (lo + 1 <= 0x7E && t.e4m3[lo + 1] <= a) ++lo;
  if (t.e4m3[lo] == a) return sign | uint8_t(lo);
  const unsigned hi = lo + 1;  // a < 448 so hi <= 0x7E
  const double dlo = a - t.e4m3[lo], dhi = t.e4m3[hi] - a;
  unsigned pick;
  if (dlo < dhi) pick = lo;
  else if (dhi < dlo) pick = hi;
  else pick = (lo % 2 == 0) ? lo : hi;
  return sign | uint8_t(pick);
}

// The MX rule (OCP MX v1.0, "conversion to MX"): shared exponent
// floor(log2(amax)) - emax_elem, scale X = 2^shared, elements v/X rounded to
// the element format. floor(log2) is taken exactly from frexp. An all-zero
// block gets scale code 0.
void orc_mx_quant_block(const float* v32, uint8_t* codes32, uint8_t* scale) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(double(v32[i])));
  const int code = mx_scale_code_for(amax, kE4M3Emax);
  const double X = std::ldexp(1.0, code - 127);
  for (int i = 0; i < 32; ++i) codes32[i] = orc_e4m3_encode_rne_sat(double(v32[i]) / X);
  *scale = uint8_t(code);
}

void orc_mx_quant_rows(const float* v, int64_t rows, int64_t K, uint8_t* codes,
                       uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < K / 32; ++b)
      orc_mx_quant_block(v + r * K + b * 32, codes + r * K + b * 32, scales + r * (K / 32) + b);
}

void orc_mx_quant_rows_bf16(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes,
                            uint8_t* scales) {
  std::vector<float> buf(static_cast<size_t>(K));
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c = 0; c < K; ++c) buf[size_t(c)] = bf16_bits_to_float(x[r * K + c]);
    orc_mx_quant_rows(buf.data(), 1, K, codes + r * K, scales + r * (K / 32));
  }
}

// Nearest E2M1 value by search over the non-negative codes 0..7 (their values
// increase with the code), ties to the even code, magnitudes above 6 saturate
// to 6. The sign bit follows the sign of v, also for 0.
uint8_t orc_e2m1_encode_rne_sat(double v) {
  const Tables& t = tables();
  const uint8_t sign = std::signbit(v) ? 0x8 : 0x0;
  const double a = std::fabs(v);
  if (a >= kE2M1Max) return sign | 0x7;
  unsigned lo = 0;
  while (lo + 1 <= 7 && t.e2m1[lo + 1] <= a) ++lo;
  if (t.e2m1[lo] == a) return sign | uint8_t(lo);
  const unsigned hi = lo + 1;  // a < 6 so hi <= 7
  const double dlo = a - t.e2m1[lo], dhi = t.e2m1[hi] - a;
  unsigned pick;
  if (dlo < dhi) pick = lo;
  else if (dhi < dlo) pick = hi;
  else pick = (lo % 2 == 0) ? lo : hi;
  return sign | uint8_t(pick);
}

// The MX rule with E2M1 elements: shared exponent floor(log2(amax)) - 2.
void orc_mxfp4_quant_block(const float* v32, uint8_t* packed16, uint8_t* scale) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(double(v32[i])));
  const int code = mx_scale_code_for(amax, kE2M1Emax);
  const double X = std::ldexp(1.0, code - 127);
  for (int i = 0; i < 16; ++i) {
    const uint8_t lo = orc_e2m1_encode_rne_sat(double(v32[2 * i]) / X);
    const uint8_t hi = orc_e2m1_encode_rne_sat(double(v32[2 * i + 1]) / X);
    packed16[i] = uint8_t(lo | (hi << 4));
  }
  *scale = uint8_t(code);
}

void orc_mxfp4_quant_rows(const float* v, int64_t rows, int64_t K, uint8_t* packed,
                          uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < K / 32; ++b)
      orc_mxfp4_quant_block(v + r * K + b * 32, packed + r * (K / 2) + b * 16,
                            scales + r * (K / 32) + b);
}

void orc_mxfp4_quant_rows_bf16(const uint16_t* x, int64_t rows, int64_t K, uint8_t* packed,
                               uint8_t* scales) {
  std::vector<float> buf(static_cast<size_t>(K));
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c = 0; c < K; ++c) buf[size_t(c)] = bf16_bits_to_float(x[r * K + c]);
    orc_mxfp4_quant_rows(buf.data(), 1, K, packed + r * (K / 2), scales + r * (K / 32));
  }
}

// Sigmoid routing ("896 routed (top-16, sigmoid routing)", "Kimi K3.1 Pro at a
// glance"): a full sort of (logit, id) pairs, logit descending and id
// ascending on equal logits (IEEE comparison, so -0 == +0), the first k kept,
// weights sigmoid(l) / sum over the k of sigmoid(l) in fp64.
void orc_route_topk(const float* logits, int64_t T, int32_t E, int32_t k, int32_t* ids,
                    float* w) {
  std::vector<std::pair<float, int32_t>> row(size_t(E > 0 ? E : 0));
  for (int64_t t = 0; t < T; ++t) {
    for (int32_t e = 0; e < E; ++e) row[size_t(e)] = {logits[t * E + e], e};
    std::sort(row.begin(), row.end(), [](const std::pair<float, int32_t>& a,
                                         const std::pair<float, int32_t>& b) {
      if (a.first > b.first) return true;
      if (a.first < b.first) return false;
      return a.second < b.second;
    });
    double sum = 0.0;
    for (int32_t j = 0; j < k; ++j) sum += sigmoid(double(row[size_t(j)].first));
    for (int32_t j = 0; j < k; ++j) {
      ids[t * k + j] = row[size_t(j)].second;
      w[t * k + j] = float(sigmoid(double(row[size_t(j)].first)) / sum);
    }
  }
}

// Grouping for the grouped-MoE kernel ("The MXFP4 latent MoE on FlyDSL"): a
// counting pass, padded offsets, and a pass over slots in ascending token
// order that hands each expert's rows out in that order.
int32_t orc_permute(const int32_t* ids, int64_t T, int32_t E, int32_t k, int32_t pad_m,
                    int32_t* counts, int32_t* offsets, int32_t* slot_to_row,
                    int32_t* row_to_slot, int64_t rows_capacity) {
  for (int32_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t t = 0; t < T; ++t) {
    for (int32_t j = 0; j < k; ++j) {
      const int32_t e = ids[t * k + j];
      if (e < 0 || e >= E) return -1;
      for (int32_t j2 = 0; j2 < j; ++j2)
        if (ids[t * k + j2] == e) return -1;
      counts[e] += 1;
    }
  }
  offsets[0] = 0;
  for (int32_t e = 0; e < E; ++e) {
    const int32_t padded = (counts[e] + pad_m - 1) / pad_m * pad_m;
    offsets[e + 1] = offsets[e] + padded;
  }
  if (offsets[E] > rows_capacity) return -1;
  for (int32_t e = 0; e < E; ++e)
    for (int32_t r = offsets[e]; r < offsets[e + 1]; ++r) row_to_slot[r] = -1;
  std::vector<int32_t> next(offsets, offsets + E);
  for (int64_t t = 0; t < T; ++t) {
    for (int32_t j = 0; j < k; ++j) {
      const int64_t slot = t * k + j;
      const int32_t e = ids[slot];
      const int32_t row = next[size_t(e)]++;
      slot_to_row[slot] = row;
      row_to_slot[row] = int32_t(slot);
    }
  }
  return 0;
}

// Gate/up projection and GLU of one expert ("3,584->2x3,072" in the page's
// expert row; SwiGLU stand-in for the undefined SiTU-GLU).
static void expert_stage1_dequantised(const std::vector<double>& xd, int32_t d, int32_t I,
                                      const uint8_t* w13_e, const uint8_t* w13s_e, double* h) {
  for (int32_t i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int32_t c = 0; c < d; ++c) {
      g += xd[size_t(c)] * weight_value(w13_e, w13s_e, d, i, c);
      u += xd[size_t(c)] * weight_value(w13_e, w13s_e, d, int64_t(I) + i, c);
    }
    h[i] = g * sigmoid(g) * u;
  }
}

void orc_expert_stage1(const uint8_t* xq, const uint8_t* xs, int32_t d, int32_t I,
                       const uint8_t* w13_e, const uint8_t* w13s_e, double* h) {
  const Tables& t = tables();
  std::vector<double> xd(static_cast<size_t>(d));
  for (int32_t c = 0; c < d; ++c) xd[size_t(c)] = t.e4m3[xq[c]] * t.e8m0[xs[c / 32]];
  expert_stage1_dequantised(xd, d, I, w13_e, w13s_e, h);
}

// The same with MXFP4 activations (the A4W4 stage 1).
void orc_expert_stage1_a4(const uint8_t* xq, const uint8_t* xs, int32_t d, int32_t I,
                          const uint8_t* w13_e, const uint8_t* w13s_e, double* h) {
  std::vector<double> xd(static_cast<size_t>(d));
  for (int32_t c = 0; c < d; ++c) xd[size_t(c)] = weight_value(xq, xs, d, 0, c);
  expert_stage1_dequantised(xd, d, I, w13_e, w13s_e, h);
}

// Down projection of one expert ("3,072->3,584"; the FP8 second stage takes
// the requantised h).
void orc_expert_stage2(const uint8_t* hq, const uint8_t* hs, int32_t I, int32_t d,
                       const uint8_t* w2_e, const uint8_t* w2s_e, double* y) {
  const Tables& t = tables();
  std::vector<double> hd(static_cast<size_t>(I));
  for (int32_t i = 0; i < I; ++i) hd[size_t(i)] = t.e4m3[hq[i]] * t.e8m0[hs[i / 32]];
  for (int32_t o = 0; o < d; ++o) {
    double acc = 0.0;
    for (int32_t i = 0; i < I; ++i) acc += hd[size_t(i)] * weight_value(w2_e, w2s_e, I, o, i);
    y[o] = acc;
  }
}

// Nearest bf16 (8 exponent bits, 7 stored mantissa bits) with ties to even,
// done in one rounding from fp64 (no double rounding through fp32).
uint16_t orc_bf16_rne(double v) {
  if (std::isnan(v)) return 0x7FC0;
  const uint16_t sign = std::signbit(v) ? 0x8000 : 0x0000;
  const double a = std::fabs(v);
  if (a == 0.0) return sign;
  const double max_bf16 = std::ldexp(255.0 / 128.0, 127);
  if (a >= max_bf16 + std::ldexp(1.0, 119) || std::isinf(a)) return sign | 0x7F80;
  int ex = 0;
  std::frexp(a, &ex);
  const int e = ex - 1;                         // a in [2^e, 2^(e+1))
  const int ulp_exp = (e < -126) ? -133 : e - 7;
  const double r = std::nearbyint(std::ldexp(a, -ulp_exp));   // ties to even
  const float f = float(std::ldexp(r, ulp_exp));             // exact in bf16
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return sign | uint16_t(u >> 16);
}

static void moe_forward_impl(bool act_fp4, const uint16_t* x, const float* logits, int64_t n,
                             int32_t d, int32_t E, int32_t k, int32_t I, const uint8_t* w13,
                             const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s,
                             uint16_t* y, int32_t* ids_out, float* w_out, double* y64,
                             int32_t threads) {
  const int64_t w13_stride = int64_t(2) * I * (d / 2), w13s_stride = int64_t(2) * I * (d / 32);
  const int64_t w2_stride = int64_t(d) * (I / 2), w2s_stride = int64_t(d) * (I / 32);

  auto one_token = [&](int64_t t, std::vector<uint8_t>& xq, std::vector<uint8_t>& xs,
                       std::vector<double>& h, std::vector<float>& h32,
                       std::vector<uint8_t>& hq, std::vector<uint8_t>& hs,
                       std::vector<double>& ye, std::vector<double>& acc,
                       std::vector<int32_t>& ids, std::vector<float>& w) {
    if (act_fp4) orc_mxfp4_quant_rows_bf16(x + t * d, 1, d, xq.data(), xs.data());
    else orc_mx_quant_rows_bf16(x + t * d, 1, d, xq.data(), xs.data());
    orc_route_topk(logits + t * E, 1, E, k, ids.data(), w.data());
    std::fill(acc.begin(), acc.end(), 0.0);
    for (int32_t j = 0; j < k; ++j) {
      const int64_t e = ids[size_t(j)];
      if (act_fp4)
        orc_expert_stage1_a4(xq.data(), xs.data(), d, I, w13 + e * w13_stride,
                             w13s + e * w13s_stride, h.data());
      else
        orc_expert_stage1(xq.data(), xs.data(), d, I, w13 + e * w13_stride,
                          w13s + e * w13s_stride, h.data());
      for (int32_t i = 0; i < I; ++i) h32[size_t(i)] = float(h[size_t(i)]);
      orc_mx_quant_rows(h32.data(), 1, I, hq.data(), hs.data());
      orc_expert_stage2(hq.data(), hs.data(), I, d, w2 + e * w2_stride, w2s + e * w2s_stride,
                        ye.data());
      for (int32_t o = 0; o < d; ++o) acc[size_t(o)] += double(w[size_t(j)]) * ye[size_t(o)];
    }
    for (int32_t o = 0; o < d; ++o) {
      y[t * d + o] = orc_bf16_rne(acc[size_t(o)]);
      if (y64) y64[t * d + o] = acc[size_t(o)];
    }
    for (int32_t j = 0; j < k; ++j) {
      if (ids_out) ids_out[t * k + j] = ids[size_t(j)];
      if (w_out) w_out[t * k + j] = w[size_t(j)];
    }
  };

  int nthreads = threads > 0 ? threads : int(std::thread::hardware_concurrency());
  if (nthreads < 1) nthreads = 1;
  if (int64_t(nthreads) > n) nthreads = int(n > 0 ? n : 1);
  std::vector<std::thread> pool;
  for (int tid = 0; tid < nthreads; ++tid) {
    pool.emplace_back([&, tid]() {
      std::vector<uint8_t> xq(static_cast<size_t>(d)), xs(static_cast<size_t>(d / 32)), hq(static_cast<size_t>(I)), hs(static_cast<size_t>(I / 32));
      std::vector<double> h(static_cast<size_t>(I)), ye(static_cast<size_t>(d)), acc(static_cast<size_t>(d));
      std::vector<float> h32(static_cast<size_t>(I)), w(static_cast<size_t>(k > 0 ? k : 1));
      std::vector<int32_t> ids(static_cast<size_t>(k > 0 ? k : 1));
      for (int64_t t = tid; t < n; t += nthreads)
        one_token(t, xq, xs, h, h32, hq, hs, ye, acc, ids, w);
    });
  }
  for (auto& th : pool) th.join();
}

void orc_moe_forward(const uint16_t* x, const float* logits, int64_t n, int32_t d, int32_t E,
                     int32_t k, int32_t I, const uint8_t* w13, const uint8_t* w13s,
                     const uint8_t* w2, const uint8_t* w2s, uint16_t* y, int32_t* ids_out,
                     float* w_out, double* y64, int32_t threads) {
  moe_forward_impl(false, x, logits, n, d, E, k, I, w13, w13s, w2, w2s, y, ids_out, w_out, y64,
                   threads);
}

void orc_moe_forward_a4w4(const uint16_t* x, const float* logits, int64_t n, int32_t d,
                          int32_t E, int32_t k, int32_t I, const uint8_t* w13,
                          const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s,
                          uint16_t* y, int32_t* ids_out, float* w_out, double* y64,
                          int32_t threads) {
  moe_forward_impl(true, x, logits, n, d, E, k, I, w13, w13s, w2, w2s, y, ids_out, w_out, y64,
                   threads);
}

// A dense product of bf16 operands, one fp64 dot product per output.
void orc_gemm_bf16(const uint16_t* a, const uint16_t* b, int64_t M, int64_t N, int64_t K,
                   double* c) {
  std::vector<double> ar(static_cast<size_t>(K));
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t t = 0; t < K; ++t) ar[size_t(t)] = double(bf16_bits_to_float(a[m * K + t]));
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t t = 0; t < K; ++t) acc += ar[size_t(t)] * double(bf16_bits_to_float(b[n * K + t]));
      c[m * N + n] = acc;
    }
  }
}

// The gated MLP step: gate rows [0, Nh) and up rows [Nh, 2 Nh) of B.
void orc_gemm_bf16_swiglu(const uint16_t* a, const uint16_t* b, int64_t M, int64_t Nh,
                          int64_t K, double* h) {
  std::vector<double> gu(static_cast<size_t>(2 * Nh));
  for (int64_t m = 0; m < M; ++m) {
    orc_gemm_bf16(a + m * K, b, 1, 2 * Nh, K, gu.data());
    for (int64_t n = 0; n < Nh; ++n) {
      const double g = gu[size_t(n)], u = gu[size_t(Nh + n)];
      h[m * Nh + n] = g * sigmoid(g) * u;
    }
  }
}

void orc_bf16_rne_n(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_rne(v[i]);
}

int64_t orc_expert_bytes(int32_t d, int32_t I) {
  // Three I x d matrices: d*I/2 bytes of packed E2M1 and d*I/32 scale bytes each.
  return int64_t(3) * (int64_t(d) * I / 2 + int64_t(d) * I / 32);
}

}  // extern "C"
