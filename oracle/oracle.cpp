// oracle.cpp — plain, slow, single-threaded fp32 reference of the routed mixture-of-experts
// expert layer (Kolibri-1 style: 384 routed experts, top-6, one shared expert).
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or calls this
// file; only the tests, the package's smoke check and the benchmark's CPU-baseline leg do.
// It shares no code, header, table or helper with the CUDA path.
//
// Sources (page titles, with the section each fact comes from):
//  [P2-gate]  "We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.",
//             section "The gate": every token is scored by a router over 384 experts and
//             sent to the top 6, alongside one shared expert that every token uses; the
//             reference runs in float32; a router computed in bf16 is a planted bug.
//  [P2-1]     same page, section 1 ("Two runs of the same code disagree..."): selection is
//             on the router score plus a per-expert selection bias; forcing replays the
//             expert ids recorded in a free run; passing the forced ids in sorted order
//             changes the summation order of the six expert outputs.
//  [P2-3]     same page, section 3: the expert layer is a SwitchGLU (gated-linear-unit FFN
//             per expert) over quantised weights.
//  [P1-gate]  "We Stopped the Kolibri Benchmark Before Scoring One Answer", section
//             "The gate, forced": run free once, record the choices at every layer and
//             position, then rerun with them forced.
//  [P4]       vllm.cpp Kolibri-1 CPU FP8 dequant-cache pull request: the checkpoint's
//             expert weights are FP8.
// Readings where the pages are silent (the numerical recipe of the layer):
//  - bias added to the logits before the softmax (affects selection and weights);
//  - softmax over all 384, top-6 by probability with the lowest index winning ties,
//    weights renormalised over the selected six, ids ordered by descending probability;
//  - SwiGLU: y = Wd (silu(Wg x) * (Wu x)), silu(z) = z / (1 + exp(-z)), no biases;
//  - FP8 = OCP E4M3FN (bias 7, max 448, no infinities, NaN 0x7F/0xFF, subnormals kept),
//    one fp32 scale per output row;
//  - 4-bit weights (the K4 builds of "We Stopped the Kolibri Benchmark Before Scoring One
//    Answer", section "What this means if you want Kolibri on a Mac"; the pages give no
//    format): OCP E2M1 codes with one fp32 scale per output row, activations as for FP8;
//  - W8A8: activations entering each FP8 contraction are quantised per token (per row)
//    to E4M3 with scale rowabsmax / 448, round to nearest even, saturating;
//  - shared expert: weight 1, same shape and format as a routed expert;
//  - combine: y = y_shared, then y += w_i * y_(id_i) for i = 0..5 in slot order;
//  - stack: r <- bf16_rne(r + y) once per layer.
// Floating point: every sum is a plain sequential fp32 sum in index order; this file
// must be compiled without FMA contraction (-ffp-contract=off) and without fast-math.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- number formats ----------
// E4M3 decode by the format's definition: s eeee mmm, bias 7.
//   e == 0:            (-1)^s * m/8 * 2^-6          (subnormal)
//   e == 15, m == 7:   NaN
//   otherwise:         (-1)^s * (1 + m/8) * 2^(e-7)
float e4m3_value(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  float mag;
  if (e == 15 && m == 7) return std::nanf("");
  if (e == 0) mag = (float(m) / 8.0f) * std::ldexp(1.0f, -6);
  else mag = (1.0f + float(m) / 8.0f) * std::ldexp(1.0f, e - 7);
  return s ? -mag : mag;
}

// E2M1 (the 4-bit element format of the OCP Microscaling specification, v1.0, section
// 5.3.3) decode by the format's definition: s ee m, exponent bias 1, no infinities or NaN.
//   e == 0:   (-1)^s * m/2                 (subnormal: 0 or 0.5)
//   e  > 0:   (-1)^s * (1 + m/2) * 2^(e-1)
// The magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.
float e2m1_value(uint8_t c) {
  int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  float mag = (e == 0) ? float(m) * 0.5f : (1.0f + float(m) * 0.5f) * std::ldexp(1.0f, e - 1);
  return s ? -mag : mag;
}

struct DecodeTable {
  float v[256];
  DecodeTable() { for (int c = 0; c < 256; ++c) v[c] = e4m3_value(uint8_t(c)); }
};
const DecodeTable kDec;

// E4M3 encode: the finite code nearest to v; on a tie, the code whose mantissa LSB is 0
// (round half to even).  There is no infinity, so every value beyond 448 lands on 448
// (saturation).  Brute force over the 127 non-negative finite codes; the distances are
// taken in double, where those to the two neighbouring codes are exact.
uint8_t e4m3_encode(float v) {
  if (v != v) return 0x7F;
  uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  double a = std::fabs(double(v));
  if (a > 448.0) return uint8_t(sign | 0x7E);
  int best = 0;
  double bestd = std::fabs(a - double(kDec.v[0]));
  for (int c = 1; c <= 0x7E; ++c) {
    double dd = std::fabs(a - double(kDec.v[c]));
    if (dd < bestd || (dd == bestd && (c & 1) == 0 && (best & 1) == 1)) { best = c; bestd = dd; }
  }
  return uint8_t(sign | best);
}

float bf16_to_f32(uint16_t h) {
  uint32_t u = uint32_t(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// fp32 -> bf16, round to nearest, ties to even (on the 16 dropped bits); NaN stays NaN.
uint16_t f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if (f != f) return uint16_t((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return uint16_t(u >> 16);
}

float silu(float z) { return z / (1.0f + std::exp(-z)); }

}  // namespace

extern "C" {

// Planted mistakes (mutants) for control tests: each must be caught by a parity check.
enum {
  OR_MUT_NONE = 0,
  OR_MUT_BF16_ROUTER = 1,      // router logits computed from bf16-rounded Wr and rounded to bf16
  OR_MUT_UNBIASED_SELECT = 2,  // experts selected on the score without the bias
  OR_MUT_HIGH_INDEX_TIE = 3,   // ties broken toward the highest index
  OR_MUT_NO_RENORM = 4,        // weights = raw softmax probabilities (no renormalisation)
  OR_MUT_NO_SHARED = 5,        // shared expert dropped
  OR_MUT_SORTED_SUM = 6,       // routed outputs summed in ascending-id order
  OR_MUT_SWAP_GATE_UP = 7,     // silu applied to the up projection instead of the gate
  OR_MUT_SCALE_AXIS = 8,       // weight scale of the neighbouring output row
  OR_MUT_DISPATCH_SHIFT = 9,   // dispatch: each routed group's offset shifted by one row
  OR_MUT_BIASED_WEIGHTS = 10,  // selection-only bias mode, but the weights use the biased score too
};

// How the per-expert bias enters: OR_BIAS_SCORE adds it to the logits (selection and weights);
// OR_BIAS_SELECT adds it to the selection score only, the weights being the renormalised
// softmax of the unbiased logits.
enum { OR_BIAS_SCORE = 0, OR_BIAS_SELECT = 1 };

enum { OR_ACT_W8A8 = 0, OR_ACT_W8A16 = 1 };

typedef struct {
  int d, ffn, E, k;        // d_model, expert hidden width, routed experts, experts per token
  int w_fp8;               // 1: E4M3 codes + per-row fp32 scales; 0: fp32 weights;
                           // 2: E2M1 codes + per-row fp32 scales, two codes per byte (element
                           //    2i in the low nibble of byte i), so a row of K weights is K/2 bytes
  int act_mode;            // OR_ACT_W8A8 (default) or OR_ACT_W8A16 (fp32 activations)
  int mutant;              // OR_MUT_*
  const float* Wr;         // [E, d]
  const float* bias;       // [E] or NULL
  const void* Wgu;         // [E, 2, ffn, d]: gate rows then up rows of each expert
  const float* sgu;        // [E, 2, ffn]
  const void* Wd;          // [E, d, ffn]
  const float* sd;         // [E, d]
  const void* sh_Wgu;      // [2, ffn, d]
  const float* sh_sgu;     // [2, ffn]
  const void* sh_Wd;       // [d, ffn]
  const float* sh_sd;      // [d]
  int bias_mode;           // OR_BIAS_SCORE (default) or OR_BIAS_SELECT
} oracle_layer;

float oracle_e4m3_decode(uint8_t c) { return kDec.v[c]; }
float oracle_e2m1_decode(uint8_t c) { return e2m1_value(uint8_t(c & 15)); }
uint8_t oracle_e4m3_encode(float v) { return e4m3_encode(v); }
uint16_t oracle_bf16_rne(float f) { return f32_to_bf16(f); }
void oracle_e4m3_encode_n(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(v[i]);
}
void oracle_bf16_rne_n(const float* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(v[i]);
}

// ------------------------------------------------------------------- router ---------------
// [P2-gate], [P2-1]: logits[e] = (sum_k x[k] * Wr[e,k]) + b[e], in fp32 (without b in the
// selection-only bias mode: there the bias enters the selection score alone).
void oracle_router_logits(const oracle_layer* L, const float* xf, float* logits) {
  for (int e = 0; e < L->E; ++e) {
    const float* w = L->Wr + size_t(e) * L->d;
    float acc = 0.0f;
    if (L->mutant == OR_MUT_BF16_ROUTER) {
      for (int k = 0; k < L->d; ++k) acc += xf[k] * bf16_to_f32(f32_to_bf16(w[k]));
    } else {
      for (int k = 0; k < L->d; ++k) acc += xf[k] * w[k];
    }
    float b = (L->bias && L->bias_mode == OR_BIAS_SCORE) ? L->bias[e] : 0.0f;
    logits[e] = (L->mutant == OR_MUT_UNBIASED_SELECT) ? acc : acc + b;
    if (L->mutant == OR_MUT_BF16_ROUTER) logits[e] = bf16_to_f32(f32_to_bf16(logits[e]));
  }
}

// p = softmax(logits) with the max subtracted first.
void oracle_softmax(const float* logits, int E, float* p) {
  float m = logits[0];
  for (int e = 1; e < E; ++e) if (logits[e] > m) m = logits[e];
  float s = 0.0f;
  for (int e = 0; e < E; ++e) { p[e] = std::exp(logits[e] - m); s += p[e]; }
  for (int e = 0; e < E; ++e) p[e] = p[e] / s;
}

// k rounds of argmax over p; strict '>' scanning upward keeps the lowest index on ties.
void oracle_topk(const float* p, int E, int k, int mutant, int32_t* ids) {
  std::vector<char> taken(static_cast<size_t>(E), 0);
  for (int i = 0; i < k; ++i) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[size_t(e)]) continue;
      if (best < 0) { best = e; continue; }
      bool better = (mutant == OR_MUT_HIGH_INDEX_TIE) ? (p[e] >= p[best]) : (p[e] > p[best]);
      if (better) best = e;
    }
    taken[size_t(best)] = 1;
    ids[i] = best;
  }
}

// w_i = p[id_i] / sum_j p[id_j]  (sum in slot order).
void oracle_renorm(const float* p, const int32_t* ids, int k, int mutant, float* w) {
  float s = 0.0f;
  for (int i = 0; i < k; ++i) s += p[ids[i]];
  for (int i = 0; i < k; ++i) w[i] = (mutant == OR_MUT_NO_RENORM) ? p[ids[i]] : p[ids[i]] / s;
}

// --------------------------------------------------------------- expert FFN ---------------
// Per-row activation quantisation (W8A8 reading): s = max|v| / 448 (1 if 0), q = E4M3(v / s).
static void quant_row(const float* v, int n, uint8_t* q, float* s_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) { float a = std::fabs(v[i]); if (a > amax) amax = a; }
  float s = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int i = 0; i < n; ++i) q[i] = e4m3_encode(v[i] / s);
  *s_out = s;
}

// One expert (e in [0, E) routed, e == E the shared expert) on one token: ye = FFN_e(xf).
// [P2-3] SwitchGLU: h = silu(gate . x) * (up . x);  ye = down . h.
void oracle_expert(const oracle_layer* L, int e, const float* xf, float* ye) {
  const int d = L->d, F = L->ffn;
  const bool shared = (e == L->E);
  std::vector<float> g(static_cast<size_t>(F)), u(static_cast<size_t>(F)), h(static_cast<size_t>(F));
  if (!L->w_fp8) {
    const float* Wg = shared ? (const float*)L->sh_Wgu : (const float*)L->Wgu + size_t(e) * 2 * F * d;
    const float* Wu = Wg + size_t(F) * d;
    const float* Wd = shared ? (const float*)L->sh_Wd : (const float*)L->Wd + size_t(e) * d * F;
    for (int n = 0; n < F; ++n) {
      float ag = 0.0f, au = 0.0f;
      for (int k = 0; k < d; ++k) ag += xf[k] * Wg[size_t(n) * d + k];
      for (int k = 0; k < d; ++k) au += xf[k] * Wu[size_t(n) * d + k];
      g[size_t(n)] = ag;
      u[size_t(n)] = au;
    }
    for (int n = 0; n < F; ++n) {
      h[size_t(n)] = (L->mutant == OR_MUT_SWAP_GATE_UP) ? silu(u[size_t(n)]) * g[size_t(n)]
                                                        : silu(g[size_t(n)]) * u[size_t(n)];
    }
    for (int m = 0; m < d; ++m) {
      float acc = 0.0f;
      for (int n = 0; n < F; ++n) acc += h[size_t(n)] * Wd[size_t(m) * F + n];
      ye[m] = acc;
    }
    return;
  }
  // quantised weights: E4M3 (one byte per weight) or E2M1 (two weights per byte); a matrix of
  // rows of K weights, the value of weight (row, k) before its row scale
  const bool w4 = (L->w_fp8 == 2);
  auto wval = [&](const uint8_t* W, int row, int k, int K) -> float {
    if (!w4) return kDec.v[W[size_t(row) * K + k]];
    const uint8_t b = W[size_t(row) * (K / 2) + k / 2];
    return e2m1_value(uint8_t((k & 1) ? (b >> 4) : (b & 15)));
  };
  const size_t wdiv = w4 ? 2 : 1;  // weights per byte
  const uint8_t* Wg = shared ? (const uint8_t*)L->sh_Wgu : (const uint8_t*)L->Wgu + size_t(e) * 2 * F * d / wdiv;
  const uint8_t* Wu = Wg + size_t(F) * d / wdiv;
  const uint8_t* Wd = shared ? (const uint8_t*)L->sh_Wd : (const uint8_t*)L->Wd + size_t(e) * d * F / wdiv;
  const float* sg = shared ? L->sh_sgu : L->sgu + size_t(e) * 2 * F;
  const float* su = sg + F;
  const float* sdn = shared ? L->sh_sd : L->sd + size_t(e) * d;
  const bool w8a8 = (L->act_mode == OR_ACT_W8A8);
  auto row_scale = [&](const float* s, int n, int nrows) {
    return (L->mutant == OR_MUT_SCALE_AXIS) ? s[(n + 1) % nrows] : s[n];
  };
  // activations entering the gate/up contraction
  std::vector<float> xa(static_cast<size_t>(d));
  float sx = 1.0f;
  if (w8a8) {
    std::vector<uint8_t> qx(static_cast<size_t>(d));
    quant_row(xf, d, qx.data(), &sx);
    for (int k = 0; k < d; ++k) xa[size_t(k)] = kDec.v[qx[size_t(k)]];
  } else {
    for (int k = 0; k < d; ++k) xa[size_t(k)] = xf[k];
  }
  for (int n = 0; n < F; ++n) {
    float ag = 0.0f, au = 0.0f;
    for (int k = 0; k < d; ++k) ag += xa[size_t(k)] * wval(Wg, n, k, d);
    for (int k = 0; k < d; ++k) au += xa[size_t(k)] * wval(Wu, n, k, d);
    g[size_t(n)] = ag * sx * row_scale(sg, n, F);
    u[size_t(n)] = au * sx * row_scale(su, n, F);
  }
  for (int n = 0; n < F; ++n) {
    h[size_t(n)] = (L->mutant == OR_MUT_SWAP_GATE_UP) ? silu(u[size_t(n)]) * g[size_t(n)]
                                                      : silu(g[size_t(n)]) * u[size_t(n)];
  }
  std::vector<float> ha(static_cast<size_t>(F));
  float sh = 1.0f;
  if (w8a8) {
    std::vector<uint8_t> qh(static_cast<size_t>(F));
    quant_row(h.data(), F, qh.data(), &sh);
    for (int n = 0; n < F; ++n) ha[size_t(n)] = kDec.v[qh[size_t(n)]];
  } else {
    for (int n = 0; n < F; ++n) ha[size_t(n)] = h[size_t(n)];
  }
  for (int m = 0; m < d; ++m) {
    float acc = 0.0f;
    for (int n = 0; n < F; ++n) acc += ha[size_t(n)] * wval(Wd, m, n, F);
    ye[m] = acc * sh * row_scale(sdn, m, d);
  }
}

// ---------------------------------------------------------------- one token ---------------
// Routing of one token.  forced_ids (k ids, in the order given) replaces the selection
// [P1-gate]; forced_w (k weights, used as given) replaces the renormalised softmax.
// logits_out: the router logits (unbiased in the selection-only mode); p_out: the
// probabilities the selection ranks (softmax of logits + bias in that mode).
// Returns 0, or -4 when a forced id is out of range or repeated.
int oracle_route_token(const oracle_layer* L, const float* xf, const int32_t* forced_ids,
                       const float* forced_w, int32_t* ids, float* w, float* logits_out, float* p_out) {
  const int E = L->E, k = L->k;
  std::vector<float> logits(static_cast<size_t>(E)), p(static_cast<size_t>(E));
  if (forced_ids && forced_w) {
    for (int i = 0; i < k; ++i) { ids[i] = forced_ids[i]; w[i] = forced_w[i]; }
  } else {
    oracle_router_logits(L, xf, logits.data());
    oracle_softmax(logits.data(), E, p.data());
    if (forced_ids) {
      for (int i = 0; i < k; ++i) ids[i] = forced_ids[i];
    } else if (L->mutant == OR_MUT_UNBIASED_SELECT && L->bias) {
      // the planted bug selects on the unbiased probabilities but weights with the biased ones
      std::vector<float> lb(static_cast<size_t>(E)), pb(static_cast<size_t>(E));
      for (int e = 0; e < E; ++e) lb[size_t(e)] = logits[size_t(e)] + L->bias[e];
      oracle_softmax(lb.data(), E, pb.data());
      oracle_topk(p.data(), E, k, OR_MUT_NONE, ids);
      p.swap(pb);
      logits.swap(lb);
    } else if (L->bias_mode == OR_BIAS_SELECT && L->bias) {
      // select on softmax(logits + b); weights from softmax(logits) unless the planted bug
      std::vector<float> lb(static_cast<size_t>(E)), pb(static_cast<size_t>(E));
      for (int e = 0; e < E; ++e) lb[size_t(e)] = logits[size_t(e)] + L->bias[e];
      oracle_softmax(lb.data(), E, pb.data());
      oracle_topk(pb.data(), E, k, L->mutant, ids);
      for (int i = 0; i < k; ++i) if (ids[i] < 0 || ids[i] >= E) return -4;
      oracle_renorm(L->mutant == OR_MUT_BIASED_WEIGHTS ? pb.data() : p.data(), ids, k, L->mutant, w);
      if (logits_out) for (int e = 0; e < E; ++e) logits_out[e] = logits[size_t(e)];
      if (p_out) for (int e = 0; e < E; ++e) p_out[e] = pb[size_t(e)];
      for (int i = 0; i < k; ++i)
        for (int j = 0; j < i; ++j) if (ids[j] == ids[i]) return -4;
      return 0;
    } else {
      oracle_topk(p.data(), E, k, L->mutant, ids);
    }
    for (int i = 0; i < k; ++i) if (ids[i] < 0 || ids[i] >= E) return -4;
    oracle_renorm(p.data(), ids, k, L->mutant, w);
    if (logits_out) for (int e = 0; e < E; ++e) logits_out[e] = logits[size_t(e)];
    if (p_out) for (int e = 0; e < E; ++e) p_out[e] = p[size_t(e)];
  }
  for (int i = 0; i < k; ++i) {
    if (ids[i] < 0 || ids[i] >= E) return -4;
    for (int j = 0; j < i; ++j) if (ids[j] == ids[i]) return -4;
  }
  return 0;
}

// The whole layer on one token: y = y_shared + sum_i w_i * y_(id_i), slot order [P2-1].
int oracle_token(const oracle_layer* L, const float* xf, const int32_t* forced_ids, const float* forced_w,
                 int32_t* ids, float* w, float* y, float* logits_out, float* p_out) {
  const int d = L->d, k = L->k;
  int rc = oracle_route_token(L, xf, forced_ids, forced_w, ids, w, logits_out, p_out);
  if (rc) return rc;
  std::vector<float> ye(static_cast<size_t>(d));
  if (L->mutant == OR_MUT_NO_SHARED) {
    for (int m = 0; m < d; ++m) y[m] = 0.0f;
  } else {
    oracle_expert(L, L->E, xf, y);
  }
  int order[64];
  for (int i = 0; i < k; ++i) order[i] = i;
  if (L->mutant == OR_MUT_SORTED_SUM) {
    for (int i = 1; i < k; ++i)
      for (int j = i; j > 0 && ids[order[j]] < ids[order[j - 1]]; --j) { int t = order[j]; order[j] = order[j - 1]; order[j - 1] = t; }
  }
  for (int s = 0; s < k; ++s) {
    int i = order[s];
    oracle_expert(L, ids[i], xf, ye.data());
    for (int m = 0; m < d; ++m) y[m] += w[i] * ye[size_t(m)];
  }
  return 0;
}

static void widen_row(const void* x, int x_bf16, int d, int64_t t, float* xf) {
  if (x_bf16) {
    const uint16_t* xb = (const uint16_t*)x + t * d;
    for (int k = 0; k < d; ++k) xf[k] = bf16_to_f32(xb[k]);
  } else {
    const float* xs = (const float*)x + t * d;
    for (int k = 0; k < d; ++k) xf[k] = xs[k];
  }
}

// Layer over T tokens, one token at a time.  x: [T, d] bf16 bits (x_bf16 = 1) or fp32.
// forced_ids / forced_w: [T, k] or NULL.  Outputs ids/w [T, k], y [T, d] fp32, and
// optionally logits and probabilities [T, E] (free or forced-without-weights routing).
// Tokens [t0, t1) only; nthreads > 1 shards that range across std::threads (same function
// per token, so the result does not depend on the thread count).
int oracle_layer_forward_range(const oracle_layer* L, const void* x, int x_bf16, int64_t t0, int64_t t1,
                               const int32_t* forced_ids, const float* forced_w, int32_t* ids_out,
                               float* w_out, float* y_out, float* logits_out, float* p_out, int nthreads) {
  const int d = L->d, k = L->k, E = L->E;
  auto run = [&](int64_t a, int64_t b, int* rc) {
    std::vector<float> xf(static_cast<size_t>(d));
    for (int64_t t = a; t < b; ++t) {
      widen_row(x, x_bf16, d, t, xf.data());
      int r = oracle_token(L, xf.data(), forced_ids ? forced_ids + t * k : nullptr,
                           forced_w ? forced_w + t * k : nullptr, ids_out + t * k, w_out + t * k,
                           y_out + t * d, logits_out ? logits_out + t * E : nullptr,
                           p_out ? p_out + t * E : nullptr);
      if (r) *rc = r;
    }
  };
  int64_t n = t1 - t0;
  if (nthreads <= 1 || n < 2) { int rc = 0; run(t0, t1, &rc); return rc; }
  if (nthreads > n) nthreads = int(n);
  std::vector<std::thread> th;
  std::vector<int> rcs(static_cast<size_t>(nthreads), 0);
  int64_t per = (n + nthreads - 1) / nthreads;
  for (int i = 0; i < nthreads; ++i) {
    int64_t a = t0 + i * per, b = a + per < t1 ? a + per : t1;
    if (a >= b) break;
    th.emplace_back([&, a, b, i]() { run(a, b, &rcs[size_t(i)]); });
  }
  for (auto& tt : th) tt.join();
  for (int r : rcs) if (r) return r;
  return 0;
}

int oracle_layer_forward(const oracle_layer* L, const void* x, int x_bf16, int64_t T, const int32_t* forced_ids,
                         const float* forced_w, int32_t* ids_out, float* w_out, float* y_out,
                         float* logits_out, float* p_out, int nthreads) {
  return oracle_layer_forward_range(L, x, x_bf16, 0, T, forced_ids, forced_w, ids_out, w_out, y_out,
                                    logits_out, p_out, nthreads);
}

// ------------------------------------------------------------------ stack ------------------
// L layers on a bf16 residual stream: for each layer, y = layer(r); r = bf16_rne(r + y).
// residual: [T, d] bf16 bits, updated in place.  forced_ids: [nL, T, k] or NULL (then the
// routing is free).  ids_out: [nL, T, k] or NULL.
int oracle_stack_forward(const oracle_layer* layers, int nL, uint16_t* residual, int64_t T,
                         const int32_t* forced_ids, int32_t* ids_out, int nthreads) {
  const int d = layers[0].d, k = layers[0].k;
  std::vector<float> y(static_cast<size_t>(T) * d), w(static_cast<size_t>(T) * k);
  std::vector<int32_t> ids(static_cast<size_t>(T) * k);
  for (int l = 0; l < nL; ++l) {
    const int32_t* f = forced_ids ? forced_ids + size_t(l) * T * k : nullptr;
    int rc = oracle_layer_forward(&layers[l], residual, 1, T, f, nullptr, ids.data(), w.data(), y.data(),
                                  nullptr, nullptr, nthreads);
    if (rc) return rc;
    for (int64_t i = 0; i < T * d; ++i)
      residual[i] = f32_to_bf16(bf16_to_f32(residual[i]) + y[size_t(i)]);
    if (ids_out) std::memcpy(ids_out + size_t(l) * T * k, ids.data(), sizeof(int32_t) * size_t(T) * k);
  }
  return 0;
}

// --------------------------------------------------------------- dispatch -----------------
// Grouping of the T*k routed (token, slot) rows by expert, then the shared expert's T rows:
//   counts[e]  = number of rows routed to expert e (e < E); counts[E] = T (shared group)
//   offsets[e] = sum of counts[0..e) (exclusive scan), offsets[E+1] = T*k + T
//   perm[r]    = token of row r; inside each group tokens ascend (stable)
//   pos[t*k+i] = row that holds (token t, slot i)
// Written out as its definition: walk the experts in order, and for each the tokens in
// order.  Ids must be valid (distinct within a token, in [0, E)).
void oracle_dispatch(const int32_t* ids, int64_t T, int E, int k, int mutant, int32_t* counts,
                     int32_t* offsets, int32_t* perm, int32_t* pos) {
  for (int e = 0; e <= E; ++e) counts[e] = 0;
  for (int64_t t = 0; t < T; ++t)
    for (int i = 0; i < k; ++i) counts[ids[t * k + i]] += 1;
  counts[E] = int32_t(T);
  offsets[0] = 0;
  for (int e = 0; e <= E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  for (int e = 0; e < E; ++e) {
    int32_t row = offsets[e] + ((mutant == OR_MUT_DISPATCH_SHIFT && e > 0) ? 1 : 0);
    for (int64_t t = 0; t < T; ++t)
      for (int i = 0; i < k; ++i)
        if (ids[t * k + i] == e) {
          if (row < offsets[E]) perm[row] = int32_t(t);
          pos[t * k + i] = row;
          ++row;
        }
  }
  for (int64_t t = 0; t < T; ++t) perm[offsets[E] + t] = int32_t(t);
}

}  // extern "C"
