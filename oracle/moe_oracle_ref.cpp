// Second CPU oracle of the FP4 routed mixture-of-experts layer, in plain C++
// loops (test infrastructure only).
//
// This file is test infrastructure.  Tests may load it (through ctypes); the
// product path never does, and it shares no code with the CUDA path or with
// the numpy oracle beside it: it restates the layer's definition on its own,
// so that two independent programs of the definition can be held against each
// other and against the hand-worked fixtures.
//
// What it computes follows "DeepSeek-V4-Flash on AMD gfx90a: Correctness
// Recovery and Inference Performance Engineering" (abstract: FP4 routed MoE,
// expert sorting, the routed-expert W2 layout), the MXFP4 MoE path of the vLLM
// MI300X write-up ("MXFP4 MoE"), and the routing rules of the MI250
// correctness blog (section 4.1 table: top-k compared in FP32 with a fixed
// tie-break; section 4.2: ties go to the lower expert id).  Where the pages
// are silent, the readings are the same as the numpy oracle's:
//   - MXFP4: E2M1 codes (sign bit 3, exponent bits 2..1, mantissa bit 0), two
//     per byte along K, the low nibble holding the even K element; one E8M0
//     byte s per 32 K elements meaning 2^(s - 127) (0xFF: NaN);
//   - W13 rows [0, I) gate, [I, 2I) up; W2 row n is output feature n;
//   - routing: experts ordered by (logit descending, index ascending), the
//     first k kept; weights softmax over the k kept, shifted by the slot-0
//     logit, the normaliser summed in slot order;
//   - stable counting sort of the flat slots t*k + j by expert;
//   - h = bf16(silu(g) * u), silu(z) = z / (1 + e^-z), nearest-even;
//   - out[t] = sum over j in slot order of w[t, j] * y[slot t*k + j].
// Arithmetic is fp64 throughout except the one rounding point the layer fixes
// (h to bf16).  Sums run in index order.  Experts run on worker threads (each
// output row is written by one thread only), so the result does not depend on
// the thread count.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// E2M1 value of a 4-bit code (OCP Microscaling v1.0, FP4 E2M1): exponent bits
// e = (code >> 1) & 3, mantissa bit m = code & 1; e = 0 is subnormal
// (m * 0.5), otherwise 2^(e - 1) * (1 + m / 2); bit 3 is the sign.
double e2m1_value(unsigned code) {
  const unsigned e = (code >> 1) & 3u, m = code & 1u;
  const double mag = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, (int)e - 1);
  return (code & 8u) ? -mag : mag;
}

double e8m0_value(unsigned s) { return s == 255 ? std::nan("") : std::ldexp(1.0, (int)s - 127); }

// Element k of a packed MXFP4 row (K elements: K/2 code bytes, K/32 scales).
double mx_element(const uint8_t* row_codes, const uint8_t* row_scales, int k) {
  const uint8_t byte = row_codes[k / 2];
  const unsigned code = (k & 1) ? (byte >> 4) : (byte & 15u);
  return e2m1_value(code) * e8m0_value(row_scales[k / 32]);
}

double bf16_bits_value(uint16_t bits) {
  const uint32_t u = (uint32_t)bits << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Nearest bf16 value (ties to even) of a real v: bf16 keeps 8 significant
// bits with binary32's exponent range, so numbers in [2^e, 2^(e+1)) are spaced
// 2^(e - 7) for e >= -126 and 2^-133 below; values at or past 2^128 after
// rounding overflow to infinity.
double bf16_round(double v) {
  if (v == 0.0 || !std::isfinite(v)) return v;
  const double a = std::fabs(v);
  int ex;
  std::frexp(a, &ex);  // a = f * 2^ex, f in [0.5, 1)
  int e = ex - 1;
  if (e < -126) e = -126;
  const double ulp = std::ldexp(1.0, e - 7);
  double q = std::nearbyint(a / ulp) * ulp;  // the default rounding mode: nearest, ties to even
  if (q >= std::ldexp(1.0, 128)) q = INFINITY;
  return std::copysign(q, v);
}

double silu(double z) { return z / (1.0 + std::exp(-z)); }

// Top-k of one token: k times the best remaining expert, "best" being the
// larger fp32 logit (+0 and -0 equal) or, on equal logits, the lower index.
void route_token(const float* logits, int E, int k, int32_t* ids, double* w) {
  std::vector<char> taken(E, 0);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || logits[e] > logits[best]) best = e;  // equal logits keep the lower index
    }
    taken[best] = 1;
    ids[j] = best;
  }
  const double l0 = (double)logits[ids[0]];
  double tot = 0.0;
  for (int j = 0; j < k; ++j) {
    w[j] = std::exp((double)logits[ids[j]] - l0);
    tot += w[j];
  }
  for (int j = 0; j < k; ++j) w[j] /= tot;
}

}  // namespace

extern "C" {

// Routing of T tokens: ids int32 [T, k], weights fp64 [T, k].  0 on success.
int oracle_ref_route(int T, int E, int k, const float* logits, int32_t* ids, double* w) {
  if (T < 1 || E < 1 || k < 1 || k > E || !logits || !ids || !w) return -1;
  for (int t = 0; t < T; ++t) route_token(logits + (size_t)t * E, E, k, ids + (size_t)t * k, w + (size_t)t * k);
  return 0;
}

// Stable counting sort of the S = T*k flat slots by expert: offsets [E+1]
// (slots routed to experts below e), sorted_slot [S] (flat slot of each sorted
// position, increasing within an expert), slot_pos [S] (its inverse).
int oracle_ref_sort(int T, int E, int k, const int32_t* ids, int32_t* offsets, int32_t* sorted_slot,
                    int32_t* slot_pos) {
  const long long S = (long long)T * k;
  if (T < 1 || E < 1 || k < 1 || !ids || !offsets || !sorted_slot || !slot_pos) return -1;
  std::vector<long long> count(E, 0);
  for (long long f = 0; f < S; ++f) {
    if (ids[f] < 0 || ids[f] >= E) return -1;
    ++count[ids[f]];
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = (int32_t)(offsets[e] + count[e]);
  std::vector<long long> next(offsets, offsets + E);
  for (long long f = 0; f < S; ++f) {
    const long long pos = next[ids[f]]++;
    sorted_slot[pos] = (int32_t)f;
    slot_pos[f] = (int32_t)pos;
  }
  return 0;
}

// The whole layer.  x bf16 bits [T, d]; logits fp32 [T, E]; w13 [E, 2I, d/2]
// and scales [E, 2I, d/32]; w2 [E, d, I/2] and scales [E, d, I/32].  Outputs:
// ids [T, k], w [T, k], offsets [E+1], sorted_slot [S], h fp64 [S, I] (bf16
// values, sorted order), out fp64 [T, d].  n_threads workers (>= 1) take
// experts in turn.  0 on success.
int oracle_ref_forward(int T, int d, int I, int E, int k, const uint16_t* x, const float* logits,
                       const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s, int32_t* ids,
                       double* w, int32_t* offsets, int32_t* sorted_slot, double* h, double* out, int n_threads) {
  if (T < 1 || d < 32 || I < 32 || d % 32 || I % 32 || !x || !h || !out) return -1;
  if (oracle_ref_route(T, E, k, logits, ids, w) != 0) return -1;
  const long long S = (long long)T * k;
  std::vector<int32_t> slot_pos(S);
  if (oracle_ref_sort(T, E, k, ids, offsets, sorted_slot, slot_pos.data()) != 0) return -1;
  std::vector<double> y((size_t)S * d, 0.0);
  auto expert = [&](int e) {
    const uint8_t* g_codes = w13 + (size_t)e * 2 * I * (d / 2);
    const uint8_t* g_scales = w13s + (size_t)e * 2 * I * (d / 32);
    const uint8_t* d_codes = w2 + (size_t)e * d * (I / 2);
    const uint8_t* d_scales = w2s + (size_t)e * d * (I / 32);
    for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
      const int t = sorted_slot[r] / k;
      const uint16_t* xr = x + (size_t)t * d;
      double* hr = h + (size_t)r * I;
      for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        const uint8_t* gc = g_codes + (size_t)i * (d / 2);
        const uint8_t* gs = g_scales + (size_t)i * (d / 32);
        const uint8_t* uc = g_codes + (size_t)(I + i) * (d / 2);
        const uint8_t* us = g_scales + (size_t)(I + i) * (d / 32);
        for (int kk = 0; kk < d; ++kk) {
          const double xv = bf16_bits_value(xr[kk]);
          g += xv * mx_element(gc, gs, kk);
          u += xv * mx_element(uc, us, kk);
        }
        hr[i] = bf16_round(silu(g) * u);
      }
      double* yr = y.data() + (size_t)r * d;
      for (int n = 0; n < d; ++n) {
        const uint8_t* dc = d_codes + (size_t)n * (I / 2);
        const uint8_t* ds = d_scales + (size_t)n * (I / 32);
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += hr[i] * mx_element(dc, ds, i);
        yr[n] = acc;
      }
    }
  };
  const int nt = n_threads < 1 ? 1 : n_threads;
  std::vector<std::thread> pool;
  for (int p = 0; p < nt; ++p)
    pool.emplace_back([&, p] {
      for (int e = p; e < E; e += nt) expert(e);
    });
  for (auto& th : pool) th.join();
  for (int t = 0; t < T; ++t)
    for (int n = 0; n < d; ++n) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += w[(size_t)t * k + j] * y[(size_t)slot_pos[(size_t)t * k + j] * d + n];
      out[(size_t)t * d + n] = acc;
    }
  return 0;
}

}  // extern "C"
