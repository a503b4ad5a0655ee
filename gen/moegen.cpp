// moegen — seeded, counter-based synthetic inputs for the routed expert layer.
//
// This module produces INPUT DATA only (activations, router weights and bias, FP8 expert
// weights with their per-row scales, forced routes).  It holds none of the layer's own
// arithmetic: no router, no selection, no expert FFN, no combine.  Both the CUDA library
// and the CPU oracle consume what it writes; neither links against the other.
//
// Random numbers: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014; constants as in Vigna's public-domain splitmix64.c).  The i-th
// draw of a stream is the SplitMix64 output function applied to state0 + (i+1)*gamma, so
// any element can be generated independently of the others (counter-based).  The stream
// state0 is derived from (seed, layer, tensor).  Gaussians come from the
// inversion method (one draw per element, see InvNormal).
//
// Weight quantisation recipe (input preparation, the "converted checkpoint"): each output
// row r of a weight matrix is stored as E4M3 codes of w/s_r with s_r = max|w_r| / 448
// (s_r = 1 for an all-zero row), rounded to nearest, ties to even code, saturating at 448.
// The 4-bit checkpoint stores E2M1 codes of w/s_r with s_r = max|w_r| / 6 the same way.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

const uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

inline uint64_t sm64_out(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

inline uint64_t stream_state(uint64_t seed, uint32_t layer, uint32_t tensor) {
  uint64_t s = sm64_out(seed * kGamma + 0x1234567ULL);
  s = sm64_out(s + (uint64_t(layer) + 1) * kGamma);
  s = sm64_out(s ^ ((uint64_t(tensor) + 1) * 0xD1B54A32D192ED03ULL));
  return s;
}

inline uint64_t draw(uint64_t state, uint64_t i) { return sm64_out(state + (i + 1) * kGamma); }

// uniform in (0, 1], 24 bits
inline float u01_open0(uint64_t z) { return float((z >> 40) + 1) * (1.0f / 16777216.0f); }
// uniform in [0, 1), 24 bits
inline float u01(uint64_t z) { return float(z >> 40) * (1.0f / 16777216.0f); }
// uniform in [0, 1), 53 bits
inline double u01d(uint64_t z) { return double(z >> 11) * (1.0 / 9007199254740992.0); }

// Standard normals by inversion: z = Phi^-1(u) for one 32-bit uniform u = (k + 1/2) 2^-32
// per element.  Phi^-1 on v = min(u, 1-u) in (0, 1/2] is tabulated per binary octave
// [2^-(j+1), 2^-j), j = 0..32, at 256 equal steps, and interpolated linearly; the table is
// built once by bisection on Phi(z) = erfc(-z / sqrt 2) / 2 in double precision.
struct InvNormal {
  float t[33][257];
  InvNormal() {
    for (int j = 0; j <= 32; ++j)
      for (int i = 0; i <= 256; ++i) {
        double v = std::ldexp(1.0 + i / 256.0, -j - 1);
        double lo = -40.0, hi = 0.0;
        for (int it = 0; it < 200 && hi - lo > 1e-15; ++it) {
          double mid = 0.5 * (lo + hi);
          if (0.5 * std::erfc(-mid / std::sqrt(2.0)) < v) lo = mid; else hi = mid;
        }
        t[j][i] = float(0.5 * (lo + hi));
      }
  }
};
const InvNormal kInvNormal;

inline float normal_at(uint64_t state, uint64_t i) {
  uint64_t k = draw(state, i) >> 32;
  double u = (double(k) + 0.5) * (1.0 / 4294967296.0);
  double v = u < 0.5 ? u : 1.0 - u;
  uint64_t b;
  std::memcpy(&b, &v, 8);
  int j = 1022 - int((b >> 52) & 0x7FF);           // v in [2^-(j+1), 2^-j)
  uint64_t mant = b & 0xFFFFFFFFFFFFFULL;           // 52 fraction bits
  int idx = int(mant >> 44);                        // top 8 bits
  float frac = float(double(mant & 0xFFFFFFFFFFFULL) * (1.0 / 17592186044416.0));  // low 44 bits
  float z = kInvNormal.t[j][idx] + (kInvNormal.t[j][idx + 1] - kInvNormal.t[j][idx]) * frac;
  return u < 0.5 ? z : -z;
}

// Nearest E4M3 code of v, ties to the even code, saturating at +-448 (finite v).
// Below 2^-6 the E4M3 grid is uniform with step 2^-9, so the code is rint(|v| * 512);
// above it, rounding the fp32 mantissa to 3 bits (round half to even on the bit pattern)
// gives exponent and mantissa fields directly.
inline uint8_t quant_e4m3(float v) {
  uint32_t u;
  std::memcpy(&u, &v, 4);
  uint8_t sign = uint8_t((u >> 24) & 0x80u);
  u &= 0x7FFFFFFFu;
  float a;
  std::memcpy(&a, &u, 4);
  if (!(a == a)) return 0x7F;
  if (a >= 448.0f) return sign | 0x7E;
  if (a < 0.015625f) return sign | uint8_t(int(std::nearbyint(a * 512.0f)));
  uint32_t r = u + 0x7FFFFu + ((u >> 20) & 1u);
  int e = int(r >> 23) - 127;
  int code = ((e + 7) << 3) | int((r >> 20) & 7u);
  if (code > 0x7E) code = 0x7E;
  return sign | uint8_t(code);
}

// Nearest E2M1 code of v (OCP Microscaling v1.0, 4-bit element format E2M1: magnitudes 0,
// 0.5, 1, 1.5, 2, 3, 4, 6 in code order 0..7, sign in bit 3), ties to the code with mantissa
// bit 0, saturating at +-6: brute force over the eight magnitudes in double.
inline uint8_t quant_e2m1(float v) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const uint8_t sign = std::signbit(v) ? 8 : 0;
  const double a = std::fabs(double(v));
  if (!(a == a)) return 0;
  int best = 0;
  double bestd = a;
  for (int c = 1; c < 8; ++c) {
    const double dd = std::fabs(a - mag[c]);
    if (dd < bestd || (dd == bestd && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      bestd = dd;
    }
  }
  return uint8_t(sign | best);
}

inline uint16_t bf16_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return uint16_t((u >> 16) | 0x40);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return uint16_t(u >> 16);
}

template <class F>
void parallel_rows(int64_t rows, int nthreads, F f) {
  if (nthreads <= 1 || rows < 2) { f(int64_t(0), rows); return; }
  nthreads = int(std::min<int64_t>(nthreads, rows));
  std::vector<std::thread> th;
  int64_t per = (rows + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    int64_t a = t * per, b = std::min(rows, a + per);
    if (a >= b) break;
    th.emplace_back([=]() { f(a, b); });
  }
  for (auto& x : th) x.join();
}

}  // namespace

extern "C" {

// out[i] = sqrt(var) * N(0,1) element (start + i) of stream (seed, layer, tensor), fp32.
void moegen_normal_f32(uint64_t seed, uint32_t layer, uint32_t tensor, uint64_t start, int64_t n,
                       double var, float* out, int nthreads) {
  uint64_t st = stream_state(seed, layer, tensor);
  float sd = float(std::sqrt(var));
  parallel_rows(n, nthreads, [&](int64_t a, int64_t b) {
    for (int64_t i = a; i < b; ++i) out[i] = sd * normal_at(st, start + uint64_t(i));
  });
}

// Same values as moegen_normal_f32, stored as bf16 bit patterns (round to nearest even).
void moegen_normal_bf16(uint64_t seed, uint32_t layer, uint32_t tensor, uint64_t start, int64_t n,
                        double var, uint16_t* out, int nthreads) {
  uint64_t st = stream_state(seed, layer, tensor);
  float sd = float(std::sqrt(var));
  parallel_rows(n, nthreads, [&](int64_t a, int64_t b) {
    for (int64_t i = a; i < b; ++i) out[i] = bf16_bits(sd * normal_at(st, start + uint64_t(i)));
  });
}

// Rows [row0, row0 + rows) of a [*, cols] Gaussian matrix (element index = row * cols + col),
// each row quantised to E4M3 with scale = rowabsmax / 448.  codes: [rows, cols], scales: [rows].
void moegen_normal_e4m3_rows(uint64_t seed, uint32_t layer, uint32_t tensor, int64_t row0, int64_t rows,
                             int64_t cols, double var, uint8_t* codes, float* scales, int nthreads) {
  uint64_t st = stream_state(seed, layer, tensor);
  float sd = float(std::sqrt(var));
  parallel_rows(rows, nthreads, [&](int64_t a, int64_t b) {
    std::vector<float> buf(static_cast<size_t>(cols));
    for (int64_t r = a; r < b; ++r) {
      uint64_t base = uint64_t(row0 + r) * uint64_t(cols);
      float amax = 0.0f;
      for (int64_t c = 0; c < cols; ++c) buf[size_t(c)] = sd * normal_at(st, base + uint64_t(c));
      for (int64_t i = 0; i < cols; ++i) amax = std::max(amax, std::fabs(buf[size_t(i)]));
      float s = amax > 0.0f ? amax / 448.0f : 1.0f;
      scales[r] = s;
      uint8_t* dst = codes + r * cols;
      for (int64_t i = 0; i < cols; ++i) dst[i] = quant_e4m3(buf[size_t(i)] / s);
    }
  });
}

// The 4-bit checkpoint: rows [row0, row0 + rows) of the same Gaussian matrix, each row stored
// as E2M1 codes of w/s with s = rowabsmax / 6 (1 for an all-zero row), two codes per byte
// (element 2i in the low nibble of byte i).  codes: [rows, cols / 2], scales: [rows].
void moegen_normal_e2m1_rows(uint64_t seed, uint32_t layer, uint32_t tensor, int64_t row0, int64_t rows,
                             int64_t cols, double var, uint8_t* codes, float* scales, int nthreads) {
  uint64_t st = stream_state(seed, layer, tensor);
  float sd = float(std::sqrt(var));
  parallel_rows(rows, nthreads, [&](int64_t a, int64_t b) {
    std::vector<float> buf(static_cast<size_t>(cols));
    for (int64_t r = a; r < b; ++r) {
      uint64_t base = uint64_t(row0 + r) * uint64_t(cols);
      float amax = 0.0f;
      for (int64_t c = 0; c < cols; ++c) buf[size_t(c)] = sd * normal_at(st, base + uint64_t(c));
      for (int64_t i = 0; i < cols; ++i) amax = std::max(amax, std::fabs(buf[size_t(i)]));
      float s = amax > 0.0f ? amax / 6.0f : 1.0f;
      scales[r] = s;
      uint8_t* dst = codes + r * (cols / 2);
      for (int64_t i = 0; i < cols; i += 2)
        dst[i / 2] = uint8_t(quant_e2m1(buf[size_t(i)] / s) | (quant_e2m1(buf[size_t(i + 1)] / s) << 4));
    }
  });
}

// Codes of single values (for the generator's own tests).
void moegen_quant_e2m1_n(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = quant_e2m1(v[i]);
}

// Quantise caller-supplied fp32 rows with the same recipe (used for hand-built weights).
void moegen_quant_rows_e4m3(const float* w, int64_t rows, int64_t cols, uint8_t* codes, float* scales) {
  for (int64_t r = 0; r < rows; ++r) {
    const float* src = w + r * cols;
    float amax = 0.0f;
    for (int64_t c = 0; c < cols; ++c) amax = std::max(amax, std::fabs(src[c]));
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    scales[r] = s;
    for (int64_t c = 0; c < cols; ++c) codes[r * cols + c] = quant_e4m3(src[c] / s);
  }
}

// Forced routes with Zipf(s) expert popularity: for each token, k distinct experts drawn
// without replacement, P(rank r) proportional to r^-s over the experts still available;
// expert id = rank - 1.  ids: [T, k] in draw order.
void moegen_zipf_ids(uint64_t seed, uint32_t layer, uint32_t tensor, int T, int E, int k, double s,
                     int32_t* ids) {
  uint64_t st = stream_state(seed, layer, tensor);
  std::vector<double> wt(static_cast<size_t>(E));
  for (int r = 0; r < E; ++r) wt[size_t(r)] = std::pow(double(r + 1), -s);
  std::vector<char> used(static_cast<size_t>(E));
  for (int t = 0; t < T; ++t) {
    std::fill(used.begin(), used.end(), 0);
    for (int j = 0; j < k; ++j) {
      double tot = 0.0;
      for (int r = 0; r < E; ++r) if (!used[size_t(r)]) tot += wt[size_t(r)];
      double u = u01d(draw(st, uint64_t(t) * uint64_t(k) + uint64_t(j))) * tot;
      int pick = -1;
      double acc = 0.0;
      for (int r = 0; r < E; ++r) {
        if (used[size_t(r)]) continue;
        pick = r;
        acc += wt[size_t(r)];
        if (u < acc) break;
      }
      used[size_t(pick)] = 1;
      ids[t * k + j] = pick;
    }
  }
}

// Flat-Dirichlet routing weights: k Exp(1) draws per token, divided by their sum.
void moegen_dirichlet_w(uint64_t seed, uint32_t layer, uint32_t tensor, int T, int k, float* w) {
  uint64_t st = stream_state(seed, layer, tensor);
  std::vector<double> g(static_cast<size_t>(k));
  for (int t = 0; t < T; ++t) {
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
      double u = 1.0 - u01d(draw(st, uint64_t(t) * uint64_t(k) + uint64_t(j)));  // (0, 1]
      g[size_t(j)] = -std::log(u);
      sum += g[size_t(j)];
    }
    for (int j = 0; j < k; ++j) w[t * k + j] = float(g[size_t(j)] / sum);
  }
}

// Uniform integers in [0, n) (used to pick sampled token rows for spot checks).
void moegen_uniform_int(uint64_t seed, uint32_t layer, uint32_t tensor, int64_t count, int64_t n, int64_t* out) {
  uint64_t st = stream_state(seed, layer, tensor);
  for (int64_t i = 0; i < count; ++i) out[i] = int64_t(u01d(draw(st, uint64_t(i))) * double(n));
}

}  // extern "C"
