// moe_oracle.cpp — slow, plain CPU oracle for the NVFP4 routed-expert MoE feed-forward step.
//
// TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline leg
// load this library. The GPU library never links, includes or calls it, and it never calls
// the GPU library.
//
// What it computes follows the model card "Qwen3.8-Flash-Next NVIDIA NVFP4 for Infernix
// (bit-exact)", section "What is bit-exact and what is quantized" (routed experts stored as
// E2M1 codes, one E4M3 scale per 16 weights, an FP32 multiplier and an FP32 activation input
// scale per matrix; router stored BF16; 512 routed experts, top-10), and the Infernix README,
// section "Activation precision" (W4A4 experts with calibrated input scales; a 16-bit
// activation route on the same 4-bit weights). Where the pages are silent (softmax over the
// selected logits, SiLU(gate)*up, the steps of the quantiser, where BF16 roundings happen) the
// plainest reading is taken; each such reading is named at the function that uses it.
//
// Everything is accumulated in FP64. E2M1 and E4M3 are decoded by table. Where a floating-point
// value decides an integer (a quantised code) the decision is taken on FP32 values, computed
// here by exact emulation of IEEE single-precision products and quotients.
//
// Parity status of each function is stated beside it ("pinned by" names the kind of check the
// tests apply; see tests/test_oracle_pins.py).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#include <numeric>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---------------------------------------------------------------------------------------------
// Format tables (OCP 8-bit floating point / OCP microscaling formats, as named on the model
// card: "E2M1 codes, E4M3 scale per 16").
// ---------------------------------------------------------------------------------------------

// E2M1 magnitudes for the three low bits of a code; bit 3 is the sign.
const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

// E4M3 (the "fn" variant: no infinities, S.1111.111 is NaN) magnitudes for bytes 0x00..0x7F,
// row = 4-bit exponent field, column = 3-bit mantissa field. Entry 0x7F is NaN.
const double kE4M3[128] = {
    /* e= 0 */ 0.0, 0.001953125, 0.00390625, 0.005859375, 0.0078125, 0.009765625, 0.01171875, 0.013671875,
    /* e= 1 */ 0.015625, 0.017578125, 0.01953125, 0.021484375, 0.0234375, 0.025390625, 0.02734375, 0.029296875,
    /* e= 2 */ 0.03125, 0.03515625, 0.0390625, 0.04296875, 0.046875, 0.05078125, 0.0546875, 0.05859375,
    /* e= 3 */ 0.0625, 0.0703125, 0.078125, 0.0859375, 0.09375, 0.1015625, 0.109375, 0.1171875,
    /* e= 4 */ 0.125, 0.140625, 0.15625, 0.171875, 0.1875, 0.203125, 0.21875, 0.234375,
    /* e= 5 */ 0.25, 0.28125, 0.3125, 0.34375, 0.375, 0.40625, 0.4375, 0.46875,
    /* e= 6 */ 0.5, 0.5625, 0.625, 0.6875, 0.75, 0.8125, 0.875, 0.9375,
    /* e= 7 */ 1.0, 1.125, 1.25, 1.375, 1.5, 1.625, 1.75, 1.875,
    /* e= 8 */ 2.0, 2.25, 2.5, 2.75, 3.0, 3.25, 3.5, 3.75,
    /* e= 9 */ 4.0, 4.5, 5.0, 5.5, 6.0, 6.5, 7.0, 7.5,
    /* e=10 */ 8.0, 9.0, 10.0, 11.0, 12.0, 13.0, 14.0, 15.0,
    /* e=11 */ 16.0, 18.0, 20.0, 22.0, 24.0, 26.0, 28.0, 30.0,
    /* e=12 */ 32.0, 36.0, 40.0, 44.0, 48.0, 52.0, 56.0, 60.0,
    /* e=13 */ 64.0, 72.0, 80.0, 88.0, 96.0, 104.0, 112.0, 120.0,
    /* e=14 */ 128.0, 144.0, 160.0, 176.0, 192.0, 208.0, 224.0, 240.0,
    /* e=15 */ 256.0, 288.0, 320.0, 352.0, 384.0, 416.0, 448.0, NAN,
};

double e2m1_value(int code) {
  double m = kE2M1[code & 7];
  return (code & 8) ? -m : m;
}

double e4m3_value(int byte) {
  double m = kE4M3[byte & 0x7F];
  return (byte & 0x80) ? -m : m;
}

// Nearest E2M1 code to a finite float, ties to the even code, magnitudes above 6 saturate to 6
// ("satfinite"). The sign bit follows the sign of the input, so negative values that round to
// zero encode as 0x8 (-0).
int e2m1_encode(float v) {
  int sign = std::signbit(v) ? 8 : 0;
  double a = std::fabs((double)v);
  if (std::isnan(v)) return sign | 7;
  if (a >= 6.0) return sign | 7;
  int hi = 1;
  while (kE2M1[hi] < a) ++hi;          // kE2M1[hi] >= a, hi in 1..7
  int lo = hi - 1;
  if (kE2M1[hi] == a) return sign | hi;
  double dlo = a - kE2M1[lo], dhi = kE2M1[hi] - a;
  int c;
  if (dlo < dhi) c = lo;
  else if (dhi < dlo) c = hi;
  else c = (lo % 2 == 0) ? lo : hi;     // tie: even code
  return sign | c;
}

// Nearest non-negative finite E4M3 byte to a non-negative float, ties to the even byte,
// anything above 448 saturates to 448 (0x7E).
int e4m3_encode_nonneg(float v) {
  double a = (double)v;
  if (std::isnan(v)) return 0x7F;
  if (a <= 0.0) return 0;
  if (a >= 448.0) return 0x7E;
  int hi = 1;
  while (kE4M3[hi] < a) ++hi;          // hi in 1..0x7E
  int lo = hi - 1;
  if (kE4M3[hi] == a) return hi;
  double dlo = a - kE4M3[lo], dhi = kE4M3[hi] - a;
  if (dlo < dhi) return lo;
  if (dhi < dlo) return hi;
  return (lo % 2 == 0) ? lo : hi;
}

// Exact emulation of one IEEE single-precision operation with round-to-nearest-even.
// A product of two floats is exact in double (24+24 <= 53 bits), so one rounding to float gives
// the correctly rounded result. For the quotient, double rounding through 53 bits is innocuous
// because 53 >= 2*24+2 (S. A. Figueroa, "When is double rounding innocuous?", 1995).
inline float f32_mul(float a, float b) { return (float)((double)a * (double)b); }
inline float f32_div(float a, float b) { return (float)((double)a / (double)b); }

inline double bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Round a double to the nearest BF16 (8 significant bits, 8-bit exponent), ties to even, in a
// single rounding. Overflow goes to infinity as IEEE round-to-nearest does.
uint16_t double_to_bf16(double v) {
  if (std::isnan(v)) return 0x7FC0;
  if (v == 0.0) return std::signbit(v) ? 0x8000 : 0x0000;
  double a = std::fabs(v);
  int e;
  std::frexp(a, &e);                       // a = f * 2^e, f in [0.5, 1)
  int q_exp = e - 8;                       // 8 significant bits
  if (q_exp < -133) q_exp = -133;          // subnormal spacing 2^-133
  double q = std::ldexp(a, -q_exp);
  double r = std::nearbyint(q);            // default rounding mode: nearest, ties to even
  double rounded = std::ldexp(r, q_exp);
  const double kMax = 3.3895313892515355e38;  // largest finite BF16
  float f;
  if (rounded > kMax) f = INFINITY;
  else f = (float)rounded;                 // exact: rounded has <= 8 significant bits
  if (v < 0) f = -f;
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

// One 16-element NVFP4 block, quantised with per-matrix FP32 scale S.
// Reading of the quantiser steps (the pages name the format but not the steps):
//   inv6S = fl32(1 / fl32(6*S))                 per matrix
//   a     = max |v_i|
//   sf    = E4M3_RNE_satfinite(fl32(a * inv6S))
//   sf == 0  ->  every code +0
//   r     = fl32(1 / fl32(dec(sf) * S))
//   q_i   = E2M1_RNE_satfinite(fl32(v_i * r))
// Decoded value = dec(q_i) * dec(sf) * S.
struct BlockQ {
  uint8_t sf;
  uint8_t q[16];
  float r;
  float t;
};

BlockQ quantize_block(const float* v, int n, float inv6S, float S) {
  BlockQ b;
  float a = 0.0f;
  for (int i = 0; i < n; ++i) a = std::max(a, std::fabs(v[i]));
  b.t = f32_mul(a, inv6S);
  b.sf = (uint8_t)e4m3_encode_nonneg(b.t);
  std::memset(b.q, 0, sizeof(b.q));
  b.r = 0.0f;
  if (kE4M3[b.sf] == 0.0) return b;
  b.r = f32_div(1.0f, f32_mul((float)kE4M3[b.sf], S));
  for (int i = 0; i < n; ++i) b.q[i] = (uint8_t)e2m1_encode(f32_mul(v[i], b.r));
  return b;
}

inline float inv6S_of(float S) { return f32_div(1.0f, f32_mul(6.0f, S)); }

// W4A8 activation quantiser (reading: the pages name an 8-bit expert-activation route but fix
// neither format nor scaling; taken: FP8 E4M3, round to nearest even, saturating at 448, sign
// kept, one FP32 scale per matrix from the same calibration as the NVFP4 input scale S, whose
// calibrated amax maps onto E4M3's largest value 448 instead of 6 * 448):
//   S8 = fl32(6 * S),  r8 = fl32(1 / S8),  q = E4M3_RNE_satfinite(fl32(v * r8)),
//   decoded value = dec(q) * S8.
inline float a8_scale(float S) { return f32_mul(6.0f, S); }
inline float a8_inv(float S) { return f32_div(1.0f, a8_scale(S)); }
int e4m3_encode_signed(float v) {
  return (std::signbit(v) ? 0x80 : 0) | e4m3_encode_nonneg(std::fabs(v));
}
inline int quantize_a8(float v, float r8) { return e4m3_encode_signed(f32_mul(v, r8)); }

// Quantise rows x cols values (cols a multiple of 16) into checkpoint layout:
// codes [rows][cols/2] with the even column in the low nibble, scales [rows][cols/16].
void quantize_rows(const float* v, int64_t rows, int64_t cols, float S, uint8_t* codes,
                   uint8_t* scales) {
  float inv6S = inv6S_of(S);
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < cols / 16; ++b) {
      BlockQ q = quantize_block(v + r * cols + b * 16, 16, inv6S, S);
      scales[r * (cols / 16) + b] = q.sf;
      for (int i = 0; i < 8; ++i)
        codes[r * (cols / 2) + b * 8 + i] = (uint8_t)(q.q[2 * i] | (q.q[2 * i + 1] << 4));
    }
  }
}

// Dequantise an NVFP4 matrix in checkpoint layout to FP64: code * scale * multiplier.
void dequantize_rows(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                     double mult, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      uint8_t byte = codes[r * (cols / 2) + c / 2];
      int code = (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      out[r * cols + c] = e2m1_value(code) * e4m3_value(scales[r * (cols / 16) + c / 16]) * mult;
    }
}

// Ambiguity of the W4A4 h quantiser's decisions, for tests that compare the oracle's codes
// with an FP32 evaluation of h whose values may differ from the oracle's by up to eps times the
// block's max |h| (eps is a tolerance reading: the FP32 evaluation error of h relative to the
// block amax). For one 16-element block v (FP32 h values) with the down input scale S:
//   - the block scale is ambiguous when the scaled amax t = fl32(a * inv6S) and t * (1 -/+ eps)
//     encode to different E4M3 bytes; then block = sum_i |alt_i - dec_i| * colnorm_i, alt_i
//     being element i decoded after Q with the other scale, dec_i with the block's own scale;
//   - element i (block scale unchanged) is ambiguous when its scaled value fl32(v_i * r) moved
//     by -/+ eps * a * r encodes to different E2M1 codes; then elem_i = |dec(alt code) -
//     dec(code)| * dec(sf) * S * colnorm_i, alt code being the code on the other side.
// colnorm_i = ||Wd[:, i]||_2, the factor by which a change of h_i moves the expert's output Y.
// Everything else is 0. Pinned by: hand-built blocks at and around E2M1 and E4M3 rounding
// boundaries against an interval test written independently in FP64, and a brute-force
// perturbation of single elements re-quantised with the (separately pinned) quantiser.
void h_ambiguity(const float* vb, float S, float inv6S, double eps, const double* colnorm,
                 double* elem, double* block) {
  const BlockQ q = quantize_block(vb, 16, inv6S, S);
  const double sfv = kE4M3[q.sf];
  float a = 0.0f;
  for (int i = 0; i < 16; ++i) a = std::max(a, std::fabs(vb[i]));
  double dec[16];
  for (int i = 0; i < 16; ++i) dec[i] = e2m1_value(q.q[i]) * sfv * (double)S;
  *block = 0.0;
  if (eps > 0) {
    const float tlo = (float)((double)q.t * (1.0 - eps));
    const float thi = (float)((double)q.t * (1.0 + eps));
    const int s_lo = e4m3_encode_nonneg(tlo), s_hi = e4m3_encode_nonneg(thi);
    if (s_lo != s_hi) {
      const int alt = (s_lo != q.sf) ? s_lo : s_hi;
      const double altv = kE4M3[alt];
      const float ralt = altv == 0.0 ? 0.0f : f32_div(1.0f, f32_mul((float)altv, S));
      double contrib = 0.0;
      for (int i = 0; i < 16; ++i) {
        const double dalt =
            altv == 0.0 ? 0.0 : e2m1_value(e2m1_encode(f32_mul(vb[i], ralt))) * altv * (double)S;
        contrib += std::fabs(dalt - dec[i]) * colnorm[i];
      }
      *block = contrib;
    }
  }
  for (int i = 0; i < 16; ++i) {
    elem[i] = 0.0;
    if (eps > 0 && q.r != 0.0f) {
      const double xs = (double)f32_mul(vb[i], q.r);
      const double win = eps * (double)a * (double)q.r;
      const int c_lo = e2m1_encode((float)(xs - win)), c_hi = e2m1_encode((float)(xs + win));
      if (c_lo != c_hi) {  // a +0/-0 pair contributes 0 but is still a valid flip
        const int alt = (c_lo != q.q[i]) ? c_lo : c_hi;
        elem[i] = std::fabs(e2m1_value(alt) - e2m1_value(q.q[i])) * sfv * (double)S * colnorm[i];
      }
    }
  }
}

// The same window for the W4A8 h quantiser, element by element (there is no block scale): for a
// 16-element block v of FP32 h values with the down input scale S, element i is ambiguous when
// fl32(v_i * r8) moved by -/+ eps * a * r8 (a = the block's max |h|) encodes to different E4M3
// bytes c_lo, c_hi; the window can span several codes of a small element (E4M3 steps are
// relative to the element), so elem_i = max(|dec(c_lo) - dec(q)|, |dec(c_hi) - dec(q)|) * S8 *
// colnorm_i, the largest move any code in the window makes. Pinned against an interval test.
void h8_ambiguity(const float* vb, float S, double eps, const double* colnorm, double* elem) {
  const float r8 = a8_inv(S);
  const double S8 = (double)a8_scale(S);
  float a = 0.0f;
  for (int i = 0; i < 16; ++i) a = std::max(a, std::fabs(vb[i]));
  for (int i = 0; i < 16; ++i) {
    elem[i] = 0.0;
    if (eps <= 0) continue;
    const int q = quantize_a8(vb[i], r8);
    const double xs = (double)f32_mul(vb[i], r8);
    const double win = eps * (double)a * (double)r8;
    const int c_lo = e4m3_encode_signed((float)(xs - win));
    const int c_hi = e4m3_encode_signed((float)(xs + win));
    if (c_lo != c_hi) {
      const double d = std::max(std::fabs(e4m3_value(c_lo) - e4m3_value(q)),
                                std::fabs(e4m3_value(c_hi) - e4m3_value(q)));
      elem[i] = d * S8 * colnorm[i];
    }
  }
}

}  // namespace

extern "C" {

// ------------------------------- format primitives (pinned: exhaustive decode vs closed form,
// ------------------------------- brute-force nearest search, numpy float32 arithmetic)
double oracle_e2m1_value(int code) { return e2m1_value(code); }
double oracle_e4m3_value(int byte) { return e4m3_value(byte); }
int oracle_e2m1_encode(float v) { return e2m1_encode(v); }
int oracle_e4m3_encode(float v) { return e4m3_encode_nonneg(v); }
float oracle_f32_mul(float a, float b) { return f32_mul(a, b); }
float oracle_f32_div(float a, float b) { return f32_div(a, b); }
uint16_t oracle_double_to_bf16(double v) { return double_to_bf16(v); }

// Quantiser Q over rows of FP32 values (pinned: brute force, round-trip and error invariants).
void oracle_quantize_nvfp4(const float* v, int64_t rows, int64_t cols, float S, uint8_t* codes,
                           uint8_t* scales, int nthreads) {
  (void)nthreads;
#ifdef _OPENMP
  if (nthreads > 1) {
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int64_t r = 0; r < rows; ++r)
      quantize_rows(v + r * cols, 1, cols, S, codes + r * (cols / 2), scales + r * (cols / 16));
    return;
  }
#endif
  quantize_rows(v, rows, cols, S, codes, scales);
}

// The intermediate values of Q for one block, for step-by-step pins.
void oracle_quantize_block_steps(const float* v16, float S, float* inv6S, float* t, int* sf,
                                 float* r, float* scaled16, uint8_t* codes16) {
  float i6 = inv6S_of(S);
  BlockQ q = quantize_block(v16, 16, i6, S);
  *inv6S = i6;
  *t = q.t;
  *sf = q.sf;
  *r = q.r;
  for (int i = 0; i < 16; ++i) {
    scaled16[i] = (q.r == 0.0f) ? 0.0f : f32_mul(v16[i], q.r);
    codes16[i] = q.q[i];
  }
}

// Quantise a BF16 weight matrix as the synthetic checkpoints are made: per-matrix multiplier
// = fl32(fl32(global amax) / 2688), 2688 = 6 * 448, then Q with S = multiplier.
float oracle_quantize_weight_bf16(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* codes,
                                  uint8_t* scales, int nthreads) {
  std::vector<float> v((size_t)(rows * cols));
  float amax = 0.0f;
  for (int64_t i = 0; i < rows * cols; ++i) {
    v[i] = (float)bf16_to_double(w[i]);
    amax = std::max(amax, std::fabs(v[i]));
  }
  float S = f32_div(amax, 2688.0f);
  if (S == 0.0f) S = 1.0f;
  oracle_quantize_nvfp4(v.data(), rows, cols, S, codes, scales, nthreads);
  return S;
}

void oracle_dequantize_nvfp4(const uint8_t* codes, const uint8_t* scales, int64_t rows,
                             int64_t cols, double mult, double* out) {
  dequantize_rows(codes, scales, rows, cols, mult, out);
}

// The W4A8 activation quantiser over n FP32 values with per-matrix scale S (codes: E4M3 bytes).
void oracle_quantize_a8(const float* v, int64_t n, float S, uint8_t* codes) {
  const float r8 = a8_inv(S);
  for (int64_t i = 0; i < n; ++i) codes[i] = (uint8_t)quantize_a8(v[i], r8);
}

// The W4A8 h quantiser's ambiguity for one block (see h8_ambiguity).
void oracle_h8_ambiguity(const float* v16, float S, double eps, const double* colnorm16,
                         double* elem16) {
  h8_ambiguity(v16, S, eps, colnorm16, elem16);
}

// The W4A4 h quantiser's ambiguity for one block (see h_ambiguity; pinned there).
void oracle_h_ambiguity(const float* v16, float S, double eps, const double* colnorm16,
                        double* elem16, double* block) {
  h_ambiguity(v16, S, inv6S_of(S), eps, colnorm16, elem16, block);
}

// ------------------------------- routing
// logits[t][e] = sum_h x[t][h] * Wr[e][h] in FP64 (BF16 products are exact); abssum is
// sum_h |x[t][h] * Wr[e][h]|, the condition of each logit (for near-tie handling in tests).
// Top-k: experts ordered by logit, descending, equal logits -> lower expert index first.
// Weights: softmax over the k selected logits (= the full softmax renormalised over the top-k).
// Histogram/permute: counts[e], offsets = exclusive scan (E+1 entries), perm = token ids grouped
// by expert in ascending expert order, ascending token order inside an expert;
// slot_of[t][j] = the position of (t, idx[t][j]) in perm.
// Pinned by: invariants of top-k on brute force, k=1 and k=E closed forms, permutation checks.
void oracle_route(const uint16_t* x, const uint16_t* wr, int T, int H, int E, int k,
                  double* logits, double* abssum, int32_t* idx, double* w, int32_t* counts,
                  int32_t* offsets, int32_t* perm, int32_t* slot_of, int nthreads) {
  (void)nthreads;
  std::vector<double> xd((size_t)T * H), wd((size_t)E * H);
  for (size_t i = 0; i < xd.size(); ++i) xd[i] = bf16_to_double(x[i]);
  for (size_t i = 0; i < wd.size(); ++i) wd[i] = bf16_to_double(wr[i]);
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(static)
#endif
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0, sa = 0.0;
      for (int h = 0; h < H; ++h) {
        double p = xd[(size_t)t * H + h] * wd[(size_t)e * H + h];
        s += p;
        sa += std::fabs(p);
      }
      logits[(size_t)t * E + e] = s;
      if (abssum) abssum[(size_t)t * E + e] = sa;
    }
  }
  for (int t = 0; t < T; ++t) {
    std::vector<int> order(E);
    std::iota(order.begin(), order.end(), 0);
    const double* l = logits + (size_t)t * E;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return l[a] > l[b]; });
    double lmax = l[order[0]];
    double z = 0.0;
    for (int j = 0; j < k; ++j) z += std::exp(l[order[j]] - lmax);
    for (int j = 0; j < k; ++j) {
      idx[(size_t)t * k + j] = order[j];
      w[(size_t)t * k + j] = std::exp(l[order[j]] - lmax) / z;
    }
  }
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int s = 0; s < T * k; ++s) counts[idx[s]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int> fill(E, 0);
  for (int e = 0; e < E; ++e) {
    for (int t = 0; t < T; ++t) {
      for (int j = 0; j < k; ++j) {
        if (idx[(size_t)t * k + j] == e) {
          int pos = offsets[e] + fill[e]++;
          perm[pos] = t;
          if (slot_of) slot_of[(size_t)t * k + j] = pos;
        }
      }
    }
  }
}

// ------------------------------- the MoE forward
struct OracleMoeInputs {
  int T, H, E, k, I;
  int mode;             // 0 = W4A16, 1 = W4A4, 2 = W4A8
  int y_keep_fp64;      // 1: do not round Y to BF16 (the alternative reading)
  int nthreads;
  double amb_eps;       // W4A4 h-quantiser ambiguity window (relative to the block amax)
  const uint16_t* x;    // [T][H] BF16
  const uint16_t* router;  // [E][H] BF16
  const uint8_t* const* gate_codes;   // [E] -> [I][H/2]
  const uint8_t* const* gate_scales;  // [E] -> [I][H/16]
  const uint8_t* const* up_codes;
  const uint8_t* const* up_scales;
  const uint8_t* const* down_codes;   // [E] -> [H][I/2]
  const uint8_t* const* down_scales;  // [E] -> [H][I/16]
  const float* mult;      // [E][3]: gate, up, down multipliers
  const float* in_scale;  // [E][3]: gate, up, down activation input scales (W4A4)
};

// Every output is optional (null to skip) except out_bf16. "slots" are positions in perm.
struct OracleMoeOutputs {
  uint16_t* out_bf16;     // [T][H]
  double* out64;          // [T][H]  sum_j w_j Y_j before the final BF16 rounding
  double* logits;         // [T][E]
  double* abssum;         // [T][E]
  int32_t* idx;           // [T][k]
  double* w;              // [T][k]
  int32_t* counts;        // [E]
  int32_t* offsets;       // [E+1]
  int32_t* perm;          // [T*k]
  int32_t* slot_of;       // [T][k]
  double* g;              // [T*k][I]
  double* u;              // [T*k][I]
  double* h;              // [T*k][I]  silu(g)*u in FP64
  uint16_t* h_bf16;       // [T*k][I]  W4A16: h rounded to BF16
  uint8_t* hq_codes;      // [T*k][I/2] W4A4: Q(h) codes; W4A8: [T*k][I] E4M3 bytes
  uint8_t* hq_scales;     // [T*k][I/16]
  double* h_amb_elem;     // [T*k][I]   W4A4/W4A8: |dh| * ||Wd[:,i]|| if element i is ambiguous
  double* h_amb_block;    // [T*k][I/16] W4A4: contribution bound if the block scale is ambiguous
  double* y;              // [T*k][H]  Y (after the BF16 rounding unless y_keep_fp64)
  uint8_t* xq_codes;      // [T][H/2]  W4A4: Q(x) with the gate input scale of expert 0;
                          // W4A8: [T][H] E4M3 bytes
  uint8_t* xq_scales;     // [T][H/16]
};

// Steps (reading of the pages plus the stated readings):
//  1-4. routing as oracle_route.
//  5. per slot: g_i = sum_h a_h * Wg[i][h], u_i likewise, with a = x (W4A16), a = dec(Q(x, S))
//     (W4A4) or a = dec(E4M3(x * r8)) * S8 (W4A8), using each matrix's own input scale S;
//     W = code*scale*multiplier. FP64.
//  6. h_i = silu(g_i) * u_i = g_i / (1 + exp(-g_i)) * u_i, FP64.
//  7. h -> BF16 RNE (W4A16), h -> Q(fl32(h), S_down) decoded (W4A4), or h -> E4M3 of
//     fl32(h) under the down matrix's scale, decoded (W4A8).
//  8. Y[r] = sum_i h_i * Wd[r][i] in FP64, then BF16 RNE (unless y_keep_fp64).
//  9. out[t][r] = BF16_RNE( sum_{j=0..k-1} w[t][j] * Y_{slot(t,j)}[r] ), j in rank order.
// Pinned by: one-hot weights (closed form), identical experts, SiLU(0)=0, representable-x
// W4A4==W4A16 before the h rounding, and numpy float64 matmuls of the dequantised matrices.
int oracle_moe_forward(const OracleMoeInputs* in, OracleMoeOutputs* out) {
  const int T = in->T, H = in->H, E = in->E, k = in->k, I = in->I;
  if (T <= 0 || H <= 0 || E <= 0 || k <= 0 || k > E || I <= 0 || H % 16 || I % 16) return 1;
  const int S = T * k;
  std::vector<double> logits((size_t)T * E), wts((size_t)S);
  std::vector<int32_t> idx((size_t)S), counts(E), offsets(E + 1), perm(S), slot_of(S);
  std::vector<double> abssum((size_t)T * E);
  oracle_route(in->x, in->router, T, H, E, k, logits.data(), abssum.data(), idx.data(),
               wts.data(), counts.data(), offsets.data(), perm.data(), slot_of.data(),
               in->nthreads);
  for (int s = 0; s < S; ++s) {
    int e = idx[s];
    if (!in->gate_codes[e] || !in->gate_scales[e] || !in->up_codes[e] || !in->up_scales[e] ||
        !in->down_codes[e] || !in->down_scales[e])
      return 2;  // a selected expert was not supplied
  }
  std::vector<double> xd((size_t)T * H);
  for (size_t i = 0; i < xd.size(); ++i) xd[i] = bf16_to_double(in->x[i]);

  std::vector<double> Y((size_t)S * H);
  std::vector<int> uniq;
  for (int e = 0; e < E; ++e)
    if (counts[e] > 0) uniq.push_back(e);

#ifdef _OPENMP
#pragma omp parallel for num_threads(in->nthreads > 0 ? in->nthreads : 1) schedule(dynamic, 1)
#endif
  for (int ui = 0; ui < (int)uniq.size(); ++ui) {
    const int e = uniq[ui];
    const double mg = in->mult[e * 3 + 0], mu = in->mult[e * 3 + 1], md = in->mult[e * 3 + 2];
    std::vector<double> Wg((size_t)I * H), Wu((size_t)I * H), Wd((size_t)H * I);
    dequantize_rows(in->gate_codes[e], in->gate_scales[e], I, H, mg, Wg.data());
    dequantize_rows(in->up_codes[e], in->up_scales[e], I, H, mu, Wu.data());
    dequantize_rows(in->down_codes[e], in->down_scales[e], H, I, md, Wd.data());
    std::vector<double> colnorm(I, 0.0);
    if (in->mode != 0) {
      for (int i = 0; i < I; ++i) {
        double s2 = 0.0;
        for (int r = 0; r < H; ++r) s2 += Wd[(size_t)r * I + i] * Wd[(size_t)r * I + i];
        colnorm[i] = std::sqrt(s2);
      }
    }
    std::vector<double> ag(H), au(H), hv(I), hdec(I);
    std::vector<float> xf(H), hf(I);
    for (int slot = offsets[e]; slot < offsets[e + 1]; ++slot) {
      const int t = perm[slot];
      const double* xt = xd.data() + (size_t)t * H;
      if (in->mode == 1) {
        // W4A4: the activation is replaced by its NVFP4 quantisation under each matrix's scale.
        for (int hh = 0; hh < H; ++hh) xf[hh] = (float)xt[hh];
        const float Sg = in->in_scale[e * 3 + 0], Su = in->in_scale[e * 3 + 1];
        const float i6g = inv6S_of(Sg), i6u = inv6S_of(Su);
        for (int b = 0; b < H / 16; ++b) {
          BlockQ qg = quantize_block(xf.data() + b * 16, 16, i6g, Sg);
          BlockQ qu = quantize_block(xf.data() + b * 16, 16, i6u, Su);
          for (int i = 0; i < 16; ++i) {
            ag[b * 16 + i] = e2m1_value(qg.q[i]) * kE4M3[qg.sf] * (double)Sg;
            au[b * 16 + i] = e2m1_value(qu.q[i]) * kE4M3[qu.sf] * (double)Su;
          }
        }
      } else if (in->mode == 2) {
        // W4A8: the activation is replaced by its E4M3 quantisation under each matrix's scale.
        const float Sg = in->in_scale[e * 3 + 0], Su = in->in_scale[e * 3 + 1];
        const float rg = a8_inv(Sg), ru = a8_inv(Su);
        const double S8g = a8_scale(Sg), S8u = a8_scale(Su);
        for (int hh = 0; hh < H; ++hh) {
          const float v = (float)xt[hh];
          ag[hh] = e4m3_value(quantize_a8(v, rg)) * S8g;
          au[hh] = e4m3_value(quantize_a8(v, ru)) * S8u;
        }
      } else {
        for (int hh = 0; hh < H; ++hh) ag[hh] = au[hh] = xt[hh];
      }
      for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        const double* wg = Wg.data() + (size_t)i * H;
        const double* wu = Wu.data() + (size_t)i * H;
        for (int hh = 0; hh < H; ++hh) {
          g += ag[hh] * wg[hh];
          u += au[hh] * wu[hh];
        }
        double h = g / (1.0 + std::exp(-g)) * u;
        hv[i] = h;
        if (out->g) out->g[(size_t)slot * I + i] = g;
        if (out->u) out->u[(size_t)slot * I + i] = u;
        if (out->h) out->h[(size_t)slot * I + i] = h;
      }
      if (in->mode == 0) {
        for (int i = 0; i < I; ++i) {
          uint16_t b = double_to_bf16(hv[i]);
          hdec[i] = bf16_to_double(b);
          if (out->h_bf16) out->h_bf16[(size_t)slot * I + i] = b;
        }
      } else if (in->mode == 2) {
        // W4A8: h -> E4M3 with the down matrix's scale, decoded
        const float Sd = in->in_scale[e * 3 + 2];
        const float r8 = a8_inv(Sd);
        const double S8 = a8_scale(Sd);
        for (int i = 0; i < I; ++i) hf[i] = (float)hv[i];
        for (int i = 0; i < I; ++i) {
          const int q = quantize_a8(hf[i], r8);
          hdec[i] = e4m3_value(q) * S8;
          if (out->hq_codes) out->hq_codes[(size_t)slot * I + i] = (uint8_t)q;
        }
        for (int b = 0; b < I / 16; ++b) {
          double amb_e[16];
          h8_ambiguity(hf.data() + b * 16, Sd, in->amb_eps, colnorm.data() + b * 16, amb_e);
          if (out->h_amb_block) out->h_amb_block[(size_t)slot * (I / 16) + b] = 0.0;
          if (out->h_amb_elem)
            for (int i = 0; i < 16; ++i) out->h_amb_elem[(size_t)slot * I + b * 16 + i] = amb_e[i];
        }
      } else {
        const float Sd = in->in_scale[e * 3 + 2];
        const float i6d = inv6S_of(Sd);
        for (int i = 0; i < I; ++i) hf[i] = (float)hv[i];
        for (int b = 0; b < I / 16; ++b) {
          const float* vb = hf.data() + b * 16;
          BlockQ q = quantize_block(vb, 16, i6d, Sd);
          const double sfv = kE4M3[q.sf];
          for (int i = 0; i < 16; ++i) hdec[b * 16 + i] = e2m1_value(q.q[i]) * sfv * (double)Sd;
          if (out->hq_scales) out->hq_scales[(size_t)slot * (I / 16) + b] = q.sf;
          if (out->hq_codes)
            for (int i = 0; i < 8; ++i)
              out->hq_codes[(size_t)slot * (I / 2) + b * 8 + i] =
                  (uint8_t)(q.q[2 * i] | (q.q[2 * i + 1] << 4));
          double amb_e[16], amb_b = 0.0;
          h_ambiguity(vb, Sd, i6d, in->amb_eps, colnorm.data() + b * 16, amb_e, &amb_b);
          if (out->h_amb_block) out->h_amb_block[(size_t)slot * (I / 16) + b] = amb_b;
          if (out->h_amb_elem)
            for (int i = 0; i < 16; ++i) out->h_amb_elem[(size_t)slot * I + b * 16 + i] = amb_e[i];
        }
      }
      for (int r = 0; r < H; ++r) {
        double y = 0.0;
        const double* wd = Wd.data() + (size_t)r * I;
        for (int i = 0; i < I; ++i) y += hdec[i] * wd[i];
        if (!in->y_keep_fp64) y = bf16_to_double(double_to_bf16(y));
        Y[(size_t)slot * H + r] = y;
      }
    }
  }

  for (int t = 0; t < T; ++t) {
    for (int r = 0; r < H; ++r) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += wts[(size_t)t * k + j] * Y[(size_t)slot_of[t * k + j] * H + r];
      out->out_bf16[(size_t)t * H + r] = double_to_bf16(acc);
      if (out->out64) out->out64[(size_t)t * H + r] = acc;
    }
  }

  if (out->logits) std::memcpy(out->logits, logits.data(), sizeof(double) * logits.size());
  if (out->abssum) std::memcpy(out->abssum, abssum.data(), sizeof(double) * abssum.size());
  if (out->idx) std::memcpy(out->idx, idx.data(), sizeof(int32_t) * S);
  if (out->w) std::memcpy(out->w, wts.data(), sizeof(double) * S);
  if (out->counts) std::memcpy(out->counts, counts.data(), sizeof(int32_t) * E);
  if (out->offsets) std::memcpy(out->offsets, offsets.data(), sizeof(int32_t) * (E + 1));
  if (out->perm) std::memcpy(out->perm, perm.data(), sizeof(int32_t) * S);
  if (out->slot_of) std::memcpy(out->slot_of, slot_of.data(), sizeof(int32_t) * S);
  if (out->y) std::memcpy(out->y, Y.data(), sizeof(double) * Y.size());
  if (in->mode == 2 && out->xq_codes) {
    const float r8 = a8_inv(in->in_scale[0]);
    for (size_t i = 0; i < (size_t)T * H; ++i) out->xq_codes[i] = (uint8_t)quantize_a8((float)xd[i], r8);
  }
  if (in->mode == 1 && out->xq_codes && out->xq_scales) {
    std::vector<float> xf(H);
    const float Sg = in->in_scale[0];
    const float i6 = inv6S_of(Sg);
    for (int t = 0; t < T; ++t) {
      for (int hh = 0; hh < H; ++hh) xf[hh] = (float)xd[(size_t)t * H + hh];
      for (int b = 0; b < H / 16; ++b) {
        BlockQ q = quantize_block(xf.data() + b * 16, 16, i6, Sg);
        out->xq_scales[(size_t)t * (H / 16) + b] = q.sf;
        for (int i = 0; i < 8; ++i)
          out->xq_codes[(size_t)t * (H / 2) + b * 8 + i] = (uint8_t)(q.q[2 * i] | (q.q[2 * i + 1] << 4));
      }
    }
  }
  return 0;
}

// ------------------------------- the shared expert
// The model card "Qwen3.8-Flash-Next NVIDIA NVFP4 for Infernix (bit-exact)", section "What is
// bit-exact and what is quantized", lists shared experts among the dense projections stored
// BF16, and a shared-expert gate stored BF16 (the MTP drafter's bullet); it gives neither shape
// nor formula. Reading taken: the Qwen-style shared expert, a dense SwiGLU expert of
// intermediate size Is with BF16 weights, scaled per token by the sigmoid of a BF16 gate
// vector's dot product with x, and added to the routed sum before the final rounding:
//   a_t     = sum_h x[t][h] * gv[h]                                  (FP64; products exact)
//   sigma_t = 1 / (1 + exp(-a_t))
//   g_i     = sum_h x[t][h] * Wgu[i][h],  u_i = sum_h x[t][h] * Wgu[Is + i][h]
//   hs_i    = BF16_RNE( silu(g_i) * u_i )              (as a routed expert's h in W4A16)
//   Ys[t][r] = BF16_RNE( sum_i hs_i * Wd[r][i] )      (FP64 sum, then rounded)
// Ys is rounded to BF16 like a routed expert's output Y: the card stores the shared expert in
// BF16 beside the other BF16 projections, and the reading that rounds the routed Y (each
// expert's output is a BF16 tensor) applies to it in the same way. The shared expert is BF16
// in both modes: W4A4 concerns the NVFP4 routed experts only. Outputs: sigma [T], hs_bf16
// [T][Is], ys [T][H] (the rounded Ys as FP64 values); optional ys64 [T][H] (the sum before its
// rounding) and h64 [T][Is] (silu(g)*u before its rounding).
// Pinned by: equality with a routed expert whose dequantised weights are the shared weights,
// a numpy float64 pipeline, the gate against scipy's logistic function, and closed-form
// combines.
void oracle_shared_expert(const uint16_t* x, int T, int H, int Is, const uint16_t* gate_up,
                          const uint16_t* down, const uint16_t* gate_vec, double* sigma,
                          uint16_t* hs_bf16, double* ys, double* ys64, double* h64,
                          int nthreads) {
  (void)nthreads;
  std::vector<double> gv(H);
  for (int hh = 0; hh < H; ++hh) gv[hh] = bf16_to_double(gate_vec[hh]);
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(static)
#endif
  for (int t = 0; t < T; ++t) {
    std::vector<double> xt(H), hdec(Is);
    for (int hh = 0; hh < H; ++hh) xt[hh] = bf16_to_double(x[(size_t)t * H + hh]);
    double a = 0.0;
    for (int hh = 0; hh < H; ++hh) a += xt[hh] * gv[hh];
    sigma[t] = 1.0 / (1.0 + std::exp(-a));
    for (int i = 0; i < Is; ++i) {
      const uint16_t* wg = gate_up + (size_t)i * H;
      const uint16_t* wu = gate_up + (size_t)(Is + i) * H;
      double g = 0.0, u = 0.0;
      for (int hh = 0; hh < H; ++hh) {
        g += xt[hh] * bf16_to_double(wg[hh]);
        u += xt[hh] * bf16_to_double(wu[hh]);
      }
      const double h = g / (1.0 + std::exp(-g)) * u;
      const uint16_t b = double_to_bf16(h);
      hdec[i] = bf16_to_double(b);
      if (hs_bf16) hs_bf16[(size_t)t * Is + i] = b;
      if (h64) h64[(size_t)t * Is + i] = h;
    }
    for (int r = 0; r < H; ++r) {
      const uint16_t* wd = down + (size_t)r * Is;
      double y = 0.0;
      for (int i = 0; i < Is; ++i) y += hdec[i] * bf16_to_double(wd[i]);
      ys[(size_t)t * H + r] = bf16_to_double(double_to_bf16(y));
      if (ys64) ys64[(size_t)t * H + r] = y;
    }
  }
}

// The MoE step with the shared expert: the routed step of oracle_moe_forward, then
//   out[t][r] = BF16_RNE( sum_{j=0..k-1} w[t][j] * Y_slot(t,j)[r] + sigma_t * Ys[t][r] )
// (Y and Ys both rounded to BF16),
// the shared term added after the routed ones. out->out64 (if given) receives the sum before
// the rounding; the other outputs are those of oracle_moe_forward.
// Pinned by: a zero shared down matrix reproduces the routed step, and k = 1 with every routed
// expert equal to the shared one (down rows exact in BF16 products) gives BF16((1 + sigma_t) Y).
int oracle_moe_forward_shared(const OracleMoeInputs* in, int Is, const uint16_t* gate_up,
                              const uint16_t* down, const uint16_t* gate_vec,
                              OracleMoeOutputs* out, double* sigma, uint16_t* hs_bf16,
                              double* ys, double* ys64, double* h64) {
  if (Is <= 0 || !gate_up || !down || !gate_vec || !sigma || !ys) return 3;
  const int T = in->T, H = in->H;
  std::vector<double> routed((size_t)T * H);
  double* keep = out->out64;
  out->out64 = routed.data();
  const int rc = oracle_moe_forward(in, out);
  out->out64 = keep;
  if (rc != 0) return rc;
  oracle_shared_expert(in->x, T, H, Is, gate_up, down, gate_vec, sigma, hs_bf16, ys, ys64, h64,
                       in->nthreads);
  for (int t = 0; t < T; ++t) {
    for (int r = 0; r < H; ++r) {
      const size_t o = (size_t)t * H + r;
      const double acc = routed[o] + sigma[t] * ys[o];
      out->out_bf16[o] = double_to_bf16(acc);
      if (out->out64) out->out64[o] = acc;
    }
  }
  return 0;
}

int oracle_abi_version(void) { return 1; }

}  // extern "C"
