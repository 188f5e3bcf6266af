// CPU oracle for the grouped-expert MoE FFN layer.
//
// TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct reference that the
// CUDA path is checked against. Only the tests, the smoke check and the benchmark's
// CPU-baseline leg may load it; the library never does. It shares no code, header,
// table or constant with the CUDA sources.
//
// It computes the layer by its plain definition, one token at a time:
//
//   route:    per token, the top_k largest fp32 logits (ties toward the lowest expert id;
//             slots ordered by logit descending, then id ascending) and a softmax over the
//             selected logits, so the k weights sum to 1 ("top-k softmax routing").
//   quant:    per token s = amax|x| / 127 (fp32), q = round-half-even(x / s), |q| <= 127.
//   expert:   acc_g[i] = sum_h q_x[h] * Wg[e,i,h]  (int32, exact), likewise acc_u;
//             g = (float(acc_g) * s_x) * s_g[e,i], u likewise;
//             h = g / (1 + exp(-g)) * u  ("SiLU(gate) * up"), fp32;
//             requant h per (token, expert) row with the same rule as the activations;
//             acc_d[o] = sum_i q_h[i] * Wd[e,o,i] (int32); d = (float(acc_d) * s_h) * s_d[e,o].
//   combine:  y[t,o] = sum_j w[t,j] * d_j[o] + d_shared[o]   (shared expert weight 1, no gate),
//             summed in slot order in double precision.
//
// The source pages describe this layer without printing formulas: a concatenated-expert
// gate/up GEMM with N = TOP_K x 2 x IM_EXP followed by one GLU region over all experts
// (page "Qwen3.6-35B-A3B Linux v1.0.4: ~2.7s fixed per-request TTFT ...", section "The fix
// (concatenated-expert dispatch)"), and batched decode that deduplicates experts across rows
// and uses an int8 dot (page "[job] Strix Halo: multi-session serving ... #145", section
// "Status", item "Next"). The precise arithmetic above is the layer definition the library
// implements: W8A8 with per-output-channel weight scales, per-token activation scales,
// fp32 scales and an fp32 output.
//
// NVFP4 experts. The same layer with its expert weights (routed and shared) in NVFP4 instead
// of int8: the format the page "[job] Strix Halo: multi-session serving ... #145" keeps for
// the routed experts (its comment of Oct 19, which compares the FP4 formats and keeps NVFP4).
// A weight row is a sequence of 4-bit E2M1 codes, two per byte (element 2j in the
// low nibble), with one E4M3 block scale per 16 consecutive elements and one fp32 scale per
// weight matrix. Dequantised weight = e2m1(code) * e4m3(block scale) * matrix scale. The
// activations stay int8 as above. With w' = e2m1 * e4m3 (the weight without the matrix
// scale), every product q * w' is a multiple of 2^-10 below 2^19 in magnitude, so a row's
// sum over up to 2^13 elements is exact in double; the oracle forms it in double (h
// ascending) and then applies the scales as the int8 layer does:
//   g = (float(acc_g) * s_x) * gs_gate,  u likewise,  d = (float(acc_d) * s_h) * gs_down.
//
// Built with -O2 -ffp-contract=off and no fast-math, so every fp32 operation is a single
// IEEE-rounded operation in the order written.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

extern "C" {

typedef struct {
  int E, k, H, I, Is;                 // Is = 0: no shared expert
  const int8_t* w_gate;               // [E, I, H]
  const int8_t* w_up;                 // [E, I, H]
  const int8_t* w_down;               // [E, H, I]
  const float* s_gate;                // [E, I]
  const float* s_up;                  // [E, I]
  const float* s_down;                // [E, H]
  const int8_t* sh_gate;              // [Is, H]
  const int8_t* sh_up;                // [Is, H]
  const int8_t* sh_down;              // [H, Is]
  const float* sh_s_gate;             // [Is]
  const float* sh_s_up;               // [Is]
  const float* sh_s_down;             // [H]
} oracle_layer;

// Optional intermediates, all indexed by (token, slot); slot j < k is routed slot j,
// slot k is the shared expert. Imax = max(I, Is). Any pointer may be NULL.
typedef struct {
  int8_t* qx;      // [T, H]
  float* sx;       // [T]
  int32_t* acc_gu; // [T, S, 2, Imax]  gate accumulators then up accumulators
  int8_t* hq;      // [T, S, Imax]
  float* sh;       // [T, S]
  int32_t* acc_d;  // [T, S, H]
} oracle_taps;

// NVFP4 layer: codes uint8 [rows, K/2] (two E2M1 codes per byte, element 2j in the low
// nibble), block scales uint8 E4M3 [rows, K/16], one fp32 scale per matrix.
typedef struct {
  int E, k, H, I, Is;
  const uint8_t* w_gate;              // [E, I, H/2]
  const uint8_t* w_up;                // [E, I, H/2]
  const uint8_t* w_down;              // [E, H, I/2]
  const uint8_t* b_gate;              // [E, I, H/16]
  const uint8_t* b_up;                // [E, I, H/16]
  const uint8_t* b_down;              // [E, H, I/16]
  const float* g_gate;                // [E]
  const float* g_up;                  // [E]
  const float* g_down;                // [E]
  const uint8_t* sh_gate;             // [Is, H/2]
  const uint8_t* sh_up;               // [Is, H/2]
  const uint8_t* sh_down;             // [H, Is/2]
  const uint8_t* sh_b_gate;           // [Is, H/16]
  const uint8_t* sh_b_up;             // [Is, H/16]
  const uint8_t* sh_b_down;           // [H, Is/16]
  const float* sh_g;                  // [3]: gate, up, down matrix scales
} oracle_layer_nvfp4;

// Intermediates of the NVFP4 layer; the accumulators are the exact sums of q * w' (double).
typedef struct {
  int8_t* qx;      // [T, H]
  float* sx;       // [T]
  double* acc_gu;  // [T, S, 2, Imax]
  int8_t* hq;      // [T, S, Imax]
  float* sh;       // [T, S]
  double* acc_d;   // [T, S, H]
} oracle_taps_nvfp4;

}  // extern "C"

namespace {

float bf16_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Per-row symmetric int8 quantisation: s = amax / 127, q = rne(v / s), clamp +-127.
void quantize_row(const float* v, int n, int8_t* q, float* s_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(v[i]));
  const float s = amax / 127.0f;
  for (int i = 0; i < n; ++i) {
    if (s == 0.0f) {
      q[i] = 0;
      continue;
    }
    float r = std::nearbyint(v[i] / s);  // default rounding mode: to nearest, ties to even
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q[i] = static_cast<int8_t>(r);
  }
  *s_out = s;
}

// One expert applied to one quantised token row. Weight rows are row-major with the
// reduction dimension contiguous. Writes d[H] (fp32) and, optionally, intermediates.
void expert_ffn(const int8_t* qx, float sx, int H, int I,
                const int8_t* Wg, const int8_t* Wu, const int8_t* Wd,
                const float* sg, const float* su, const float* sd,
                float* d, int32_t* acc_gu_tap, int8_t* hq_tap, float* sh_tap,
                int32_t* acc_d_tap, int Imax) {
  std::vector<float> h(I);
  for (int i = 0; i < I; ++i) {
    int32_t ag = 0, au = 0;
    for (int c = 0; c < H; ++c) {
      ag += static_cast<int32_t>(qx[c]) * static_cast<int32_t>(Wg[(size_t)i * H + c]);
      au += static_cast<int32_t>(qx[c]) * static_cast<int32_t>(Wu[(size_t)i * H + c]);
    }
    if (acc_gu_tap) {
      acc_gu_tap[i] = ag;
      acc_gu_tap[Imax + i] = au;
    }
    const float g = (static_cast<float>(ag) * sx) * sg[i];
    const float u = (static_cast<float>(au) * sx) * su[i];
    const float silu = g / (1.0f + std::exp(-g));
    h[i] = silu * u;
  }
  std::vector<int8_t> hq(I);
  float sh = 0.0f;
  quantize_row(h.data(), I, hq.data(), &sh);
  if (hq_tap) std::memcpy(hq_tap, hq.data(), I);
  if (sh_tap) *sh_tap = sh;
  for (int o = 0; o < H; ++o) {
    int32_t ad = 0;
    for (int i = 0; i < I; ++i)
      ad += static_cast<int32_t>(hq[i]) * static_cast<int32_t>(Wd[(size_t)o * I + i]);
    if (acc_d_tap) acc_d_tap[o] = ad;
    d[o] = (static_cast<float>(ad) * sh) * sd[o];
  }
}

// E2M1 (OCP Microscaling Formats v1.0, FP4): bit 3 sign, bits 2-1 exponent with bias 1,
// bit 0 mantissa; exponent 0 encodes the subnormals 0 and 0.5.
double e2m1_value(unsigned code) {
  const unsigned sgn = (code >> 3) & 1u, ex = (code >> 1) & 3u, man = code & 1u;
  const double mag = ex == 0 ? 0.5 * man : std::ldexp(1.0 + 0.5 * man, (int)ex - 1);
  return sgn ? -mag : mag;
}

// E4M3 (OCP FP8, the "fn" variant without infinities): bit 7 sign, bits 6-3 exponent with
// bias 7, bits 2-0 mantissa; exponent 0 encodes subnormals f/8 * 2^-6; S.1111.111 is NaN.
double e4m3_value(unsigned b) {
  const unsigned sgn = (b >> 7) & 1u, ex = (b >> 3) & 15u, man = b & 7u;
  if (ex == 15 && man == 7) return std::nan("");
  const double mag = ex == 0 ? std::ldexp(man / 8.0, -6) : std::ldexp(1.0 + man / 8.0, (int)ex - 7);
  return sgn ? -mag : mag;
}

// Element j of an NVFP4 row without the matrix scale: e2m1(code j) * e4m3(block scale j/16).
double nvfp4_element(const uint8_t* codes, const uint8_t* bscale, int j) {
  const unsigned code = (codes[j / 2] >> (4 * (j % 2))) & 15u;
  return e2m1_value(code) * e4m3_value(bscale[j / 16]);
}

// A block scale must be a finite, non-negative E4M3 value.
bool block_scales_valid(const uint8_t* b, size_t n) {
  for (size_t i = 0; i < n; ++i)
    if (b[i] >= 0x7f) return false;
  return true;
}

// One expert with NVFP4 weights applied to one quantised token row (the int8 expert_ffn with
// each weight row read through nvfp4_element and the sums formed exactly in double).
void expert_ffn_nvfp4(const int8_t* qx, float sx, int H, int I, const uint8_t* Wg,
                      const uint8_t* Wu, const uint8_t* Wd, const uint8_t* Bg, const uint8_t* Bu,
                      const uint8_t* Bd, float gg, float gu, float gd, float* d,
                      double* acc_gu_tap, int8_t* hq_tap, float* sh_tap, double* acc_d_tap,
                      int Imax) {
  std::vector<float> h(I);
  for (int i = 0; i < I; ++i) {
    double ag = 0.0, au = 0.0;
    for (int hh = 0; hh < H; ++hh) {
      ag += qx[hh] * nvfp4_element(Wg + (size_t)i * (H / 2), Bg + (size_t)i * (H / 16), hh);
      au += qx[hh] * nvfp4_element(Wu + (size_t)i * (H / 2), Bu + (size_t)i * (H / 16), hh);
    }
    if (acc_gu_tap) {
      acc_gu_tap[i] = ag;
      acc_gu_tap[Imax + i] = au;
    }
    const float g4 = (static_cast<float>(ag) * sx) * gg;
    const float u4 = (static_cast<float>(au) * sx) * gu;
    h[i] = g4 / (1.0f + std::exp(-g4)) * u4;
  }
  std::vector<int8_t> hq(I);
  float sh = 0.0f;
  quantize_row(h.data(), I, hq.data(), &sh);
  if (hq_tap) std::memcpy(hq_tap, hq.data(), I);
  if (sh_tap) *sh_tap = sh;
  for (int o = 0; o < H; ++o) {
    double ad = 0.0;
    for (int j = 0; j < I; ++j)
      ad += hq[j] * nvfp4_element(Wd + (size_t)o * (I / 2), Bd + (size_t)o * (I / 16), j);
    if (acc_d_tap) acc_d_tap[o] = ad;
    d[o] = (static_cast<float>(ad) * sh) * gd;
  }
}

// fp32 -> bf16, round to nearest even (finite inputs).
uint16_t float_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

int check_layer(const oracle_layer* L) {
  if (!L || L->E <= 0 || L->k <= 0 || L->k > L->E || L->H <= 0 || L->I <= 0 || L->Is < 0)
    return -1;
  return 0;
}

template <class F>
void parallel_tokens(int T, int nthreads, F f) {
  if (nthreads <= 1 || T <= 1) {
    for (int t = 0; t < T; ++t) f(t);
    return;
  }
  nthreads = std::min(nthreads, T);
  std::vector<std::thread> th;
  th.reserve(nthreads);
  for (int w = 0; w < nthreads; ++w) {
    th.emplace_back([=]() {
      for (int t = w; t < T; t += nthreads) f(t);
    });
  }
  for (auto& x : th) x.join();
}

}  // namespace

extern "C" {

// Top-k routing of fp32 logits [T, E] -> idx int32 [T, k], w fp32 [T, k].
// Selection compares logits (strictly greater wins, so ties go to the lowest id);
// the weights are a softmax over the k selected logits, computed in double.
int oracle_route(const float* logits, int T, int E, int k, int32_t* idx, float* w) {
  if (T < 0 || E <= 0 || k <= 0 || k > E) return -1;
  std::vector<char> taken(E);
  std::vector<double> ex(k);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) {
      if (!std::isfinite(l[e])) return -2;
      taken[e] = 0;
    }
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
      taken[best] = 1;
      idx[(size_t)t * k + j] = best;
    }
    const double m = l[idx[(size_t)t * k]];
    double z = 0.0;
    for (int j = 0; j < k; ++j) {
      ex[j] = std::exp(static_cast<double>(l[idx[(size_t)t * k + j]]) - m);
      z += ex[j];
    }
    for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = static_cast<float>(ex[j] / z);
  }
  return 0;
}

// Per-token activation quantisation of bf16 x [T, H] -> q int8 [T, H], s fp32 [T].
int oracle_quant_rows(const uint16_t* x, int T, int H, int8_t* q, float* s) {
  std::vector<float> v(H);
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < H; ++c) v[c] = bf16_to_float(x[(size_t)t * H + c]);
    quantize_row(v.data(), H, q + (size_t)t * H, s + t);
  }
  return 0;
}

// Token-by-expert permutation. counts[e] = number of (t, j) with idx[t,j] = e;
// offsets = exclusive prefix sum (E + 1 entries); perm lists the flat slot t*k + j of every
// assignment, grouped by expert in id order and, inside an expert, by (t, j) ascending.
int oracle_permute(const int32_t* idx, int T, int k, int E, int32_t* counts,
                   int32_t* offsets, int32_t* perm) {
  const long R = (long)T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long r = 0; r < R; ++r) {
    if (idx[r] < 0 || idx[r] >= E) return -1;
    counts[idx[r]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  long pos = 0;
  for (int e = 0; e < E; ++e)
    for (long r = 0; r < R; ++r)
      if (idx[r] == e) perm[pos++] = (int32_t)r;
  return 0;
}

// The whole layer, token by token (see the file header). y is double [T, H].
int oracle_forward(const oracle_layer* L, const uint16_t* x, int T, const int32_t* idx,
                   const float* w, double* y, const oracle_taps* taps, int nthreads) {
  if (check_layer(L)) return -1;
  const int H = L->H, I = L->I, Is = L->Is, k = L->k, E = L->E;
  const int S = k + (Is > 0 ? 1 : 0);
  const int Imax = std::max(I, Is);
  for (long r = 0; r < (long)T * k; ++r)
    if (idx[r] < 0 || idx[r] >= E) return -2;
  parallel_tokens(T, nthreads, [&](int t) {
    std::vector<float> xf(H), d(H);
    std::vector<int8_t> qx(H);
    for (int c = 0; c < H; ++c) xf[c] = bf16_to_float(x[(size_t)t * H + c]);
    float sx = 0.0f;
    quantize_row(xf.data(), H, qx.data(), &sx);
    if (taps && taps->qx) std::memcpy(taps->qx + (size_t)t * H, qx.data(), H);
    if (taps && taps->sx) taps->sx[t] = sx;
    double* yt = y + (size_t)t * H;
    for (int o = 0; o < H; ++o) yt[o] = 0.0;
    for (int s = 0; s < S; ++s) {
      const bool shared = (s == k);
      const int e = shared ? -1 : idx[(size_t)t * k + s];
      const int Ie = shared ? Is : I;
      const size_t slot = (size_t)t * S + s;
      int32_t* agu = (taps && taps->acc_gu) ? taps->acc_gu + slot * 2 * Imax : nullptr;
      int8_t* hq = (taps && taps->hq) ? taps->hq + slot * Imax : nullptr;
      float* sh = (taps && taps->sh) ? taps->sh + slot : nullptr;
      int32_t* ad = (taps && taps->acc_d) ? taps->acc_d + slot * H : nullptr;
      if (shared) {
        expert_ffn(qx.data(), sx, H, Is, L->sh_gate, L->sh_up, L->sh_down, L->sh_s_gate,
                   L->sh_s_up, L->sh_s_down, d.data(), agu, hq, sh, ad, Imax);
      } else {
        expert_ffn(qx.data(), sx, H, I, L->w_gate + (size_t)e * I * H,
                   L->w_up + (size_t)e * I * H, L->w_down + (size_t)e * H * I,
                   L->s_gate + (size_t)e * I, L->s_up + (size_t)e * I,
                   L->s_down + (size_t)e * H, d.data(), agu, hq, sh, ad, Imax);
      }
      const double wt = shared ? 1.0 : static_cast<double>(w[(size_t)t * k + s]);
      for (int o = 0; o < H; ++o) yt[o] += wt * static_cast<double>(d[o]);
      (void)Ie;
    }
  });
  return 0;
}

// Brute force: every routed expert applied to every token, each weighted by its routing
// weight (0 when the token did not select it), summed in expert-id order, plus the shared
// expert. Equal to oracle_forward up to the order of the double additions.
int oracle_dense(const oracle_layer* L, const uint16_t* x, int T, const int32_t* idx,
                 const float* w, double* y, int nthreads) {
  if (check_layer(L)) return -1;
  const int H = L->H, I = L->I, Is = L->Is, k = L->k, E = L->E;
  parallel_tokens(T, nthreads, [&](int t) {
    std::vector<float> xf(H), d(H);
    std::vector<int8_t> qx(H);
    for (int c = 0; c < H; ++c) xf[c] = bf16_to_float(x[(size_t)t * H + c]);
    float sx = 0.0f;
    quantize_row(xf.data(), H, qx.data(), &sx);
    std::vector<double> mask(E, 0.0);
    for (int j = 0; j < k; ++j) mask[idx[(size_t)t * k + j]] += w[(size_t)t * k + j];
    double* yt = y + (size_t)t * H;
    for (int o = 0; o < H; ++o) yt[o] = 0.0;
    for (int e = 0; e < E; ++e) {
      expert_ffn(qx.data(), sx, H, I, L->w_gate + (size_t)e * I * H,
                 L->w_up + (size_t)e * I * H, L->w_down + (size_t)e * H * I,
                 L->s_gate + (size_t)e * I, L->s_up + (size_t)e * I, L->s_down + (size_t)e * H,
                 d.data(), nullptr, nullptr, nullptr, nullptr, I);
      for (int o = 0; o < H; ++o) yt[o] += mask[e] * static_cast<double>(d[o]);
    }
    if (Is > 0) {
      expert_ffn(qx.data(), sx, H, Is, L->sh_gate, L->sh_up, L->sh_down, L->sh_s_gate,
                 L->sh_s_up, L->sh_s_down, d.data(), nullptr, nullptr, nullptr, nullptr, Is);
      for (int o = 0; o < H; ++o) yt[o] += static_cast<double>(d[o]);
    }
  });
  return 0;
}

// Input of one layer of the stacked prefill. When y is given, first the residual update
// x <- bf16(float(x) + float(y)) (fp32 add, round to nearest even); then the parameter-free RMS
// pre-norm x_in = bf16(x / sqrt(mean(x^2) + 1e-6)), evaluated in double.
int oracle_rmsnorm_residual(uint16_t* x, const double* y, uint16_t* x_in, int T, int H) {
  for (int t = 0; t < T; ++t) {
    uint16_t* xr = x + (size_t)t * H;
    if (y) {
      for (int h = 0; h < H; ++h)
        xr[h] = float_to_bf16(bf16_to_float(xr[h]) + static_cast<float>(y[(size_t)t * H + h]));
    }
    double ss = 0.0;
    for (int h = 0; h < H; ++h) {
      const double v = bf16_to_float(xr[h]);
      ss += v * v;
    }
    const double rms = std::sqrt(ss / H + 1e-6);
    for (int h = 0; h < H; ++h)
      x_in[(size_t)t * H + h] = float_to_bf16(static_cast<float>(bf16_to_float(xr[h]) / rms));
  }
  return 0;
}

// Router projection of the stacked-prefill workload: logits[t,e] = sum_h x[t,h] * Wr[h,e],
// x bf16 [T, H], Wr fp32 [H, E], summed in double (h ascending). Output double [T, E].
int oracle_router_logits(const uint16_t* x, const float* Wr, int T, int H, int E,
                         double* logits, int nthreads) {
  parallel_tokens(T, nthreads, [&](int t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += static_cast<double>(bf16_to_float(x[(size_t)t * H + h])) *
               static_cast<double>(Wr[(size_t)h * E + e]);
      logits[(size_t)t * E + e] = acc;
    }
  });
  return 0;
}

// Value of one E2M1 code (0..15) and of one E4M3 byte (0..255; NaN for the NaN encodings).
double oracle_e2m1_value(int code) { return e2m1_value((unsigned)code & 15u); }
double oracle_e4m3_value(int byte) { return e4m3_value((unsigned)byte & 255u); }

// The layer with NVFP4 expert weights (see the file header). Same arguments as
// oracle_forward; returns -3 when a block scale is negative or NaN.
int oracle_forward_nvfp4(const oracle_layer_nvfp4* L, const uint16_t* x, int T,
                         const int32_t* idx, const float* w, double* y,
                         const oracle_taps_nvfp4* taps, int nthreads) {
  if (!L || L->E <= 0 || L->k <= 0 || L->k > L->E || L->H <= 0 || L->I <= 0 || L->Is < 0 ||
      L->H % 16 || L->I % 16 || L->Is % 16)
    return -1;
  const int H = L->H, I = L->I, Is = L->Is, k = L->k, E = L->E;
  const int S = Is > 0 ? k + 1 : k;
  const int Imax = std::max(I, Is);
  for (long r = 0; r < (long)T * k; ++r)
    if (idx[r] < 0 || idx[r] >= E) return -2;
  if (!block_scales_valid(L->b_gate, (size_t)E * I * (H / 16)) ||
      !block_scales_valid(L->b_up, (size_t)E * I * (H / 16)) ||
      !block_scales_valid(L->b_down, (size_t)E * H * (I / 16)))
    return -3;
  if (Is > 0 && (!block_scales_valid(L->sh_b_gate, (size_t)Is * (H / 16)) ||
                 !block_scales_valid(L->sh_b_up, (size_t)Is * (H / 16)) ||
                 !block_scales_valid(L->sh_b_down, (size_t)H * (Is / 16))))
    return -3;
  parallel_tokens(T, nthreads, [&](int t) {
    std::vector<float> xf(H), d(H);
    std::vector<int8_t> qx(H);
    for (int c = 0; c < H; ++c) xf[c] = bf16_to_float(x[(size_t)t * H + c]);
    float sx = 0.0f;
    quantize_row(xf.data(), H, qx.data(), &sx);
    if (taps && taps->qx) std::memcpy(taps->qx + (size_t)t * H, qx.data(), H);
    if (taps && taps->sx) taps->sx[t] = sx;
    double* yt = y + (size_t)t * H;
    for (int o = 0; o < H; ++o) yt[o] = 0.0;
    for (int s = 0; s < S; ++s) {
      const bool shared = (s == k);
      const size_t slot = (size_t)t * S + s;
      double* agu = (taps && taps->acc_gu) ? taps->acc_gu + slot * 2 * Imax : nullptr;
      int8_t* hq = (taps && taps->hq) ? taps->hq + slot * Imax : nullptr;
      float* sh = (taps && taps->sh) ? taps->sh + slot : nullptr;
      double* ad = (taps && taps->acc_d) ? taps->acc_d + slot * H : nullptr;
      if (shared) {
        expert_ffn_nvfp4(qx.data(), sx, H, Is, L->sh_gate, L->sh_up, L->sh_down, L->sh_b_gate,
                         L->sh_b_up, L->sh_b_down, L->sh_g[0], L->sh_g[1], L->sh_g[2], d.data(),
                         agu, hq, sh, ad, Imax);
      } else {
        const int e = idx[(size_t)t * k + s];
        expert_ffn_nvfp4(qx.data(), sx, H, I, L->w_gate + (size_t)e * I * (H / 2),
                         L->w_up + (size_t)e * I * (H / 2), L->w_down + (size_t)e * H * (I / 2),
                         L->b_gate + (size_t)e * I * (H / 16), L->b_up + (size_t)e * I * (H / 16),
                         L->b_down + (size_t)e * H * (I / 16), L->g_gate[e], L->g_up[e],
                         L->g_down[e], d.data(), agu, hq, sh, ad, Imax);
      }
      const double wt4 = shared ? 1.0 : static_cast<double>(w[(size_t)t * k + s]);
      for (int o = 0; o < H; ++o) yt[o] += wt4 * static_cast<double>(d[o]);
    }
  });
  return 0;
}

}  // extern "C"
