// Plain CPU C++ oracle of the DeepSeekMoE layer forward (see moe_oracle.h).
//
// TEST INFRASTRUCTURE: loaded only by tests/, __graft_entry__.smoke() and the
// CPU legs of bench.py. Every function below is the definition of one step of
// the layer written out with loops; sums run in index order in double.
#include "moe_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>
#include <thread>
#include <vector>

namespace {

int workers(int threads) {
  if (threads > 0) return threads;
  const unsigned h = std::thread::hardware_concurrency();
  return h == 0 ? 1 : (int)h;
}

// body(i) for every i in [0, n), the range cut into one contiguous piece per
// worker. Callers only write to rows owned by i, so the split cannot change a
// result.
template <class F>
void parallel_for(int64_t n, int threads, const F& body) {
  const int64_t w = std::min<int64_t>(workers(threads), std::max<int64_t>(n, 1));
  if (w <= 1) {
    for (int64_t i = 0; i < n; ++i) body(i);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve((size_t)w);
  for (int64_t k = 0; k < w; ++k) {
    const int64_t lo = n * k / w, hi = n * (k + 1) / w;
    pool.emplace_back([lo, hi, &body] {
      for (int64_t i = lo; i < hi; ++i) body(i);
    });
  }
  for (auto& t : pool) t.join();
}

// sum_i a[i] * b[i], in double, i ascending.
double dot(const float* a, const float* b, int n) {
  double acc = 0.0;
  for (int i = 0; i < n; ++i) acc += (double)a[i] * (double)b[i];
  return acc;
}

double silu(double z) { return z / (1.0 + std::exp(-z)); }

// ---------------------------------------------------------------- routing
// [digest-2.2], [resmic-moe]

// The group scores of one token: for group g, its members' biased
// affinities sorted in descending order, the first group_topk of them added
// largest first in fp32.
void token_group_scores(const float* sp, int E, int G, int gk, float* gs) {
  const int gsz = E / G;
  std::vector<float> members((size_t)gsz);
  for (int g = 0; g < G; ++g) {
    for (int j = 0; j < gsz; ++j) members[(size_t)j] = sp[g * gsz + j];
    std::sort(members.begin(), members.end(), [](float a, float b) { return a > b; });
    float acc = members[0];
    for (int j = 1; j < gk; ++j) acc = acc + members[(size_t)j];
    gs[g] = acc;
  }
}

// Routing of one token: s' = s + b; the M groups with the largest group
// score (equal scores: lower group first); among their experts the K with
// the largest s' (equal values: lower index first), in that order; gate_k =
// s_{e_k} / sum_j s_{e_j} over the chosen experts, the sum and quotient in
// double, the bias not involved.
void route_token(const float* s, const float* bias, int E, int G, int K, int M, int gk, int32_t* idx,
                 float* gate) {
  std::vector<float> sp((size_t)E);
  for (int e = 0; e < E; ++e) sp[(size_t)e] = s[e] + bias[e];
  std::vector<float> gs((size_t)G);
  token_group_scores(sp.data(), E, G, gk, gs.data());
  std::vector<int> groups((size_t)G);
  std::iota(groups.begin(), groups.end(), 0);
  std::stable_sort(groups.begin(), groups.end(), [&](int a, int b) { return gs[(size_t)a] > gs[(size_t)b]; });
  std::vector<char> kept((size_t)G, 0);
  for (int i = 0; i < M; ++i) kept[(size_t)groups[(size_t)i]] = 1;
  const int gsz = E / G;
  std::vector<int> cand;
  for (int e = 0; e < E; ++e)
    if (kept[(size_t)(e / gsz)]) cand.push_back(e);
  std::stable_sort(cand.begin(), cand.end(), [&](int a, int b) { return sp[(size_t)a] > sp[(size_t)b]; });
  double sum = 0.0;
  for (int k = 0; k < K; ++k) sum += (double)s[cand[(size_t)k]];
  for (int k = 0; k < K; ++k) {
    idx[k] = cand[(size_t)k];
    gate[k] = (float)((double)s[cand[(size_t)k]] / sum);
  }
}

// ---------------------------------------------------------------- FP8
// [digest-3.1]

constexpr double kE4m3Max = 448.0;

// e4m3 value nearest to v: magnitudes in binade 2^e (e >= -6; smaller ones
// share the subnormal binade -6) are multiples of 2^(e-3); ties to even;
// anything above 448 becomes 448.
double e4m3_value(float v) {
  const double a = std::fabs((double)v);
  double q = 0.0;
  if (a > 0.0) {
    int ex = 0;
    std::frexp(a, &ex);  // a = m * 2^ex, m in [0.5, 1)
    const int e = std::max(ex - 1, -6);
    const double quantum = std::ldexp(1.0, e - 3);
    q = std::nearbyint(a / quantum) * quantum;
    if (q > kE4m3Max) q = kE4m3Max;
  }
  return std::signbit(v) ? -q : q;
}

float tile_scale(float amax, bool ue8m0) {
  if (!(amax > 0.0f)) return 1.0f;
  if (!ue8m0) return amax / 448.0f;  // one IEEE fp32 division
  // smallest power of two 2^e with 2^e >= amax / 448, e in [-127, 127]:
  // r = m * 2^ex with m in [0.5, 1) gives ceil(log2 r) = ex, or ex - 1 when
  // r is itself a power of two (m == 0.5). The double quotient is exact when
  // r is a power of two and otherwise cannot round onto one.
  const double r = (double)amax / kE4m3Max;
  int ex = 0;
  const double m = std::frexp(r, &ex);
  int e = (m == 0.5) ? ex - 1 : ex;
  e = std::min(127, std::max(-127, e));
  return (float)std::ldexp(1.0, e);
}

// q = e4m3(v / scale) per 1x128 tile of each row, the division in fp32.
void quantize_rows(const float* v, int64_t n, int k, bool ue8m0, double* q, float* scales) {
  const int nb = (k + 127) / 128;
  for (int64_t r = 0; r < n; ++r) {
    const float* row = v + r * k;
    for (int b = 0; b < nb; ++b) {
      const int c0 = b * 128, c1 = std::min(k, c0 + 128);
      float amax = 0.0f;
      for (int c = c0; c < c1; ++c) amax = std::max(amax, std::fabs(row[c]));
      const float sc = tile_scale(amax, ue8m0);
      scales[r * nb + b] = sc;
      for (int c = c0; c < c1; ++c) q[r * k + c] = e4m3_value(row[c] / sc);
    }
  }
}

// 128x128 blocks of w [n, k]: one scale per block from its largest magnitude.
void quantize_blocks(const float* w, int64_t n, int k, bool ue8m0, int threads, double* q, float* scales) {
  const int64_t nbn = (n + 127) / 128;
  const int nbk = (k + 127) / 128;
  parallel_for(nbn * nbk, threads, [&](int64_t blk) {
    const int64_t bn = blk / nbk;
    const int bk = (int)(blk % nbk);
    const int64_t r0 = bn * 128, r1 = std::min<int64_t>(n, r0 + 128);
    const int c0 = bk * 128, c1 = std::min(k, c0 + 128);
    float amax = 0.0f;
    for (int64_t r = r0; r < r1; ++r)
      for (int c = c0; c < c1; ++c) amax = std::max(amax, std::fabs(w[r * k + c]));
    const float sc = tile_scale(amax, ue8m0);
    scales[bn * nbk + bk] = sc;
    for (int64_t r = r0; r < r1; ++r)
      for (int c = c0; c < c1; ++c) q[r * k + c] = e4m3_value(w[r * k + c] / sc);
  });
}

// One output element of the FP8 GEMM: sum over K blocks b of the block's
// product sum, times the row scale of A and the block scale of W.
double fp8_dot(const double* qa_row, const float* sa_row, const double* qw_row, const float* sw_rowblock, int k) {
  const int nb = (k + 127) / 128;
  double out = 0.0;
  for (int b = 0; b < nb; ++b) {
    double part = 0.0;
    for (int i = b * 128; i < std::min(k, b * 128 + 128); ++i) part += qa_row[i] * qw_row[i];
    out += part * (double)sa_row[b] * (double)sw_rowblock[b];
  }
  return out;
}

// An expert's master weights quantised in 128x128 blocks.
struct QuantExpert {
  std::vector<double> q13, q2;
  std::vector<float> s13, s2;
  int d = 0, I = 0;
};

void quantize_expert(const float* w13, const float* w2, int d, int I, bool ue8m0, int threads, QuantExpert& qe) {
  qe.d = d;
  qe.I = I;
  qe.q13.assign((size_t)2 * I * d, 0.0);
  qe.s13.assign((size_t)((2 * I + 127) / 128) * ((d + 127) / 128), 0.0f);
  qe.q2.assign((size_t)d * I, 0.0);
  qe.s2.assign((size_t)((d + 127) / 128) * ((I + 127) / 128), 0.0f);
  quantize_blocks(w13, 2 * I, d, ue8m0, threads, qe.q13.data(), qe.s13.data());
  quantize_blocks(w2, d, I, ue8m0, threads, qe.q2.data(), qe.s2.data());
}

// One token through an FP8 expert: x row quantised 1x128 along d, GEMM1,
// SwiGLU in double with h rounded to fp32, h quantised 1x128 along I, GEMM2.
void ffn_row_fp8(const float* xrow, const QuantExpert& qe, bool ue8m0, double* y) {
  const int d = qe.d, I = qe.I;
  const int nbd = (d + 127) / 128, nbi = (I + 127) / 128;
  std::vector<double> qx((size_t)d);
  std::vector<float> sx((size_t)nbd);
  quantize_rows(xrow, 1, d, ue8m0, qx.data(), sx.data());
  std::vector<float> h((size_t)I);
  for (int j = 0; j < I; ++j) {
    const double a = fp8_dot(qx.data(), sx.data(), &qe.q13[(size_t)j * d], &qe.s13[(size_t)(j / 128) * nbd], d);
    const double b =
        fp8_dot(qx.data(), sx.data(), &qe.q13[(size_t)(I + j) * d], &qe.s13[(size_t)((I + j) / 128) * nbd], d);
    h[(size_t)j] = (float)(silu(a) * b);
  }
  std::vector<double> qh((size_t)I);
  std::vector<float> sh((size_t)nbi);
  quantize_rows(h.data(), 1, I, ue8m0, qh.data(), sh.data());
  for (int c = 0; c < d; ++c)
    y[c] = fp8_dot(qh.data(), sh.data(), &qe.q2[(size_t)c * I], &qe.s2[(size_t)(c / 128) * nbi], I);
}

// One token through a bf16 / fp32 expert, double throughout:
// y = W2 (silu(W1 v) * (W3 v)).
void ffn_row(const float* v, int d, int I, const float* w13, const float* w2, double* y) {
  std::vector<double> h((size_t)I);
  for (int j = 0; j < I; ++j) {
    const double a = dot(v, w13 + (size_t)j * d, d);
    const double b = dot(v, w13 + (size_t)(I + j) * d, d);
    h[(size_t)j] = silu(a) * b;
  }
  for (int c = 0; c < d; ++c) {
    const float* wrow = w2 + (size_t)c * I;
    double acc = 0.0;
    for (int j = 0; j < I; ++j) acc += h[(size_t)j] * (double)wrow[j];
    y[c] = acc;
  }
}

}  // namespace

extern "C" {

int mo_hardware_threads(void) { return workers(0); }

void mo_router_scores(const float* x, int64_t T, int d, const float* w_router, int E, int threads, float* s) {
  parallel_for(T, threads, [&](int64_t t) {
    for (int e = 0; e < E; ++e) {
      const float u = (float)dot(x + t * d, w_router + (size_t)e * d, d);
      s[t * E + e] = (float)(1.0 / (1.0 + std::exp(-(double)u)));
    }
  });
}

void mo_select_experts(const float* s, const float* bias, int64_t T, int E, int G, int K, int M, int group_topk,
                       int threads, int32_t* idx, float* gate) {
  parallel_for(T, threads, [&](int64_t t) {
    route_token(s + t * E, bias, E, G, K, M, group_topk, idx + t * K, gate + t * K);
  });
}

void mo_group_scores(const float* s, const float* bias, int64_t T, int E, int G, int group_topk, float* gs) {
  std::vector<float> sp((size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) sp[(size_t)e] = s[t * E + e] + bias[e];
    token_group_scores(sp.data(), E, G, group_topk, gs + t * G);
  }
}

void mo_expert_counts(const int32_t* idx, int64_t T, int K, int E, int32_t* counts) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < T * K; ++i) counts[idx[i]] += 1;
}

void mo_exclusive_offsets(const int32_t* counts, int E, int32_t* offsets) {
  int64_t run = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = (int32_t)run;
    run += counts[e];
  }
  offsets[E] = (int32_t)run;
}

void mo_permutation(const int32_t* idx, int64_t T, int K, int E, int32_t* sorted_tok, int32_t* slot_pos) {
  // experts in ascending order; inside an expert, its tokens in ascending
  // order; every (token, slot) pair gets a place (dropless [digest-2.2])
  int64_t p = 0;
  for (int e = 0; e < E; ++e) {
    for (int64_t t = 0; t < T; ++t) {
      for (int k = 0; k < K; ++k) {
        if (idx[t * K + k] == e) {
          sorted_tok[p] = (int32_t)t;
          slot_pos[t * K + k] = (int32_t)p;
          ++p;
        }
      }
    }
  }
}

void mo_bias_update(const int32_t* counts, int E, int64_t T, int K, float gamma, float* bias) {
  // load counts_e against the mean load T*K/E, compared as counts_e * E vs T * K
  const int64_t target = T * (int64_t)K;
  for (int e = 0; e < E; ++e) {
    const int64_t load = (int64_t)counts[e] * E;
    if (load > target) {
      bias[e] = bias[e] - gamma;  // overloaded
    } else if (load < target) {
      bias[e] = bias[e] + gamma;  // underloaded
    }
  }
}

float mo_load_max_over_mean(const int32_t* counts, int E, int64_t T, int K) {
  int32_t mx = 0;
  for (int e = 0; e < E; ++e) mx = std::max(mx, counts[e]);
  return (float)((double)mx * E / ((double)T * K));
}

void mo_bias_balancing_loop(const float* s, const float* bias0, int64_t T, int E, int G, int K, int M,
                            int group_topk, int steps, float gamma, int threads, float* biases, int32_t* idx,
                            float* loads) {
  std::vector<float> b(bias0, bias0 + E);
  std::vector<float> gate((size_t)(T * K));
  std::vector<int32_t> counts((size_t)E);
  for (int step = 0; step < steps; ++step) {
    int32_t* ix = idx + (int64_t)step * T * K;
    mo_select_experts(s, b.data(), T, E, G, K, M, group_topk, threads, ix, gate.data());
    mo_expert_counts(ix, T, K, E, counts.data());
    loads[step] = mo_load_max_over_mean(counts.data(), E, T, K);
    mo_bias_update(counts.data(), E, T, K, gamma, b.data());
    std::memcpy(biases + (int64_t)step * E, b.data(), sizeof(float) * (size_t)E);
  }
}

void mo_swiglu_ffn(const float* v, int64_t n, int d, int I, const float* w13, const float* w2, int threads,
                   double* y) {
  parallel_for(n, threads, [&](int64_t r) { ffn_row(v + r * d, d, I, w13, w2, y + r * d); });
}

void mo_expert_accumulate(const float* x, int d, const int64_t* rows, int64_t n, int I, const float* w13,
                          const float* w2, const float* g, int threads, double* acc) {
  parallel_for(n, threads, [&](int64_t i) {
    std::vector<double> y((size_t)d);
    ffn_row(x + rows[i] * d, d, I, w13, w2, y.data());
    const double gi = g ? (double)g[i] : 1.0;
    double* out = acc + rows[i] * d;
    for (int c = 0; c < d; ++c) out[c] += gi * y[(size_t)c];
  });
}

void mo_layer_forward(const float* x, int64_t T, int d, int E, int G, int K, int M, int group_topk, int I, int S,
                      const float* w_router, const float* w13, const float* w2, const float* ws13,
                      const float* ws2, const float* bias, const float* scores_in, int threads, float* scores,
                      int32_t* idx, float* gate, double* out) {
  if (scores_in != nullptr) {
    std::memcpy(scores, scores_in, sizeof(float) * (size_t)(T * E));
  } else {
    mo_router_scores(x, T, d, w_router, E, threads, scores);
  }
  mo_select_experts(scores, bias, T, E, G, K, M, group_topk, threads, idx, gate);
  const size_t w13_sz = (size_t)2 * I * d, w2_sz = (size_t)d * I;
  // [resmic-moe]: output = sum of the shared experts + gate-weighted routed sum
  parallel_for(T, threads, [&](int64_t t) {
    std::vector<double> y((size_t)d);
    double* o = out + t * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int sh = 0; sh < S; ++sh) {
      ffn_row(x + t * d, d, I, ws13 + sh * w13_sz, ws2 + sh * w2_sz, y.data());
      for (int c = 0; c < d; ++c) o[c] += y[(size_t)c];
    }
    for (int k = 0; k < K; ++k) {
      const int e = idx[t * K + k];
      ffn_row(x + t * d, d, I, w13 + e * w13_sz, w2 + e * w2_sz, y.data());
      for (int c = 0; c < d; ++c) o[c] += (double)gate[t * K + k] * y[(size_t)c];
    }
  });
}

double mo_e4m3_value(float v) { return e4m3_value(v); }

uint8_t mo_e4m3_code(float v) {
  const double q = e4m3_value(v);
  const uint8_t sign = std::signbit(q) ? 0x80 : 0x00;
  const double a = std::fabs(q);
  if (a == 0.0) return sign;
  int ex = 0;
  std::frexp(a, &ex);
  const int e = ex - 1;
  if (e >= -6) {  // normal: 1.mmm * 2^e, exponent field e + 7
    const int mant = (int)std::nearbyint((a / std::ldexp(1.0, e) - 1.0) * 8.0);
    return (uint8_t)(sign | ((e + 7) << 3) | mant);
  }
  // subnormal: m * 2^-9 with m in 1..7, exponent field 0
  return (uint8_t)(sign | (int)std::nearbyint(a / std::ldexp(1.0, -9)));
}

double mo_e4m3_decode(uint8_t c) {
  const double sign = (c & 0x80) ? -1.0 : 1.0;
  const int ef = (c >> 3) & 0xF, mf = c & 0x7;
  if (ef == 0xF && mf == 0x7) return std::nan("");
  if (ef == 0) return sign * (mf / 8.0) * std::ldexp(1.0, -6);
  return sign * (1.0 + mf / 8.0) * std::ldexp(1.0, ef - 7);
}

float mo_tile_scale(float amax, int ue8m0) { return tile_scale(amax, ue8m0 != 0); }

void mo_quantize_rows_1x128(const float* v, int64_t n, int k, int ue8m0, double* q, float* scales) {
  quantize_rows(v, n, k, ue8m0 != 0, q, scales);
}

void mo_quantize_blocks_128x128(const float* w, int64_t n, int k, int ue8m0, double* q, float* scales) {
  quantize_blocks(w, n, k, ue8m0 != 0, 1, q, scales);
}

void mo_fp8_gemm(const double* qa, const float* sa, int64_t n, int k, const double* qw, const float* sw, int64_t m,
                 int threads, double* out) {
  const int nb = (k + 127) / 128;
  parallel_for(n, threads, [&](int64_t r) {
    for (int64_t c = 0; c < m; ++c)
      out[r * m + c] = fp8_dot(qa + r * k, sa + r * nb, qw + c * k, sw + (c / 128) * nb, k);
  });
}

void mo_expert_accumulate_fp8(const float* x, int d, const int64_t* rows, int64_t n, int I, const float* w13,
                              const float* w2, const float* g, int ue8m0, int threads, double* acc) {
  QuantExpert qe;
  quantize_expert(w13, w2, d, I, ue8m0 != 0, threads, qe);
  parallel_for(n, threads, [&](int64_t i) {
    std::vector<double> y((size_t)d);
    ffn_row_fp8(x + rows[i] * d, qe, ue8m0 != 0, y.data());
    const double gi = g ? (double)g[i] : 1.0;
    double* out = acc + rows[i] * d;
    for (int c = 0; c < d; ++c) out[c] += gi * y[(size_t)c];
  });
}

void mo_layer_forward_fp8(const float* x, int64_t T, int d, int E, int G, int K, int M, int group_topk, int I,
                          int S, const float* w_router, const float* w13, const float* w2, const float* ws13,
                          const float* ws2, const float* bias, int ue8m0, int threads, float* scores, int32_t* idx,
                          float* gate, double* out) {
  mo_router_scores(x, T, d, w_router, E, threads, scores);
  mo_select_experts(scores, bias, T, E, G, K, M, group_topk, threads, idx, gate);
  const size_t w13_sz = (size_t)2 * I * d, w2_sz = (size_t)d * I;
  std::vector<QuantExpert> routed((size_t)E), shared((size_t)S);
  for (int e = 0; e < E; ++e) quantize_expert(w13 + e * w13_sz, w2 + e * w2_sz, d, I, ue8m0 != 0, threads, routed[e]);
  for (int s = 0; s < S; ++s) quantize_expert(ws13 + s * w13_sz, ws2 + s * w2_sz, d, I, ue8m0 != 0, threads, shared[s]);
  parallel_for(T, threads, [&](int64_t t) {
    std::vector<double> y((size_t)d);
    double* o = out + t * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int s = 0; s < S; ++s) {
      ffn_row_fp8(x + t * d, shared[(size_t)s], ue8m0 != 0, y.data());
      for (int c = 0; c < d; ++c) o[c] += y[(size_t)c];
    }
    for (int k = 0; k < K; ++k) {
      ffn_row_fp8(x + t * d, routed[(size_t)idx[t * K + k]], ue8m0 != 0, y.data());
      for (int c = 0; c < d; ++c) o[c] += (double)gate[t * K + k] * y[(size_t)c];
    }
  });
}

void mo_sequence_balance(const float* s, const int32_t* idx, int64_t T, int E, int K, int seq_len, double alpha,
                         double* loss, double* f, double* P) {
  // per run of seq_len tokens (the last may be shorter), L its length:
  // f_i = E / (K L) * #choices of i, P_i = (1/L) sum_t s_it / sum_j s_jt,
  // loss = alpha * sum_i f_i P_i  [digest-2.2; the report's definition]
  const int64_t n_seq = (T + seq_len - 1) / seq_len;
  std::vector<double> fq((size_t)E), pq((size_t)E);
  for (int64_t q = 0; q < n_seq; ++q) {
    const int64_t t0 = q * seq_len, t1 = std::min<int64_t>(T, t0 + seq_len);
    const double L = (double)(t1 - t0);
    std::fill(fq.begin(), fq.end(), 0.0);
    std::fill(pq.begin(), pq.end(), 0.0);
    for (int64_t t = t0; t < t1; ++t) {
      for (int k = 0; k < K; ++k) fq[(size_t)idx[t * K + k]] += 1.0;
      double row = 0.0;
      for (int e = 0; e < E; ++e) row += (double)s[t * E + e];
      for (int e = 0; e < E; ++e) pq[(size_t)e] += (double)s[t * E + e] / row;
    }
    double acc = 0.0;
    for (int e = 0; e < E; ++e) {
      fq[(size_t)e] = (double)E / ((double)K * L) * fq[(size_t)e];
      pq[(size_t)e] = pq[(size_t)e] / L;
      acc += fq[(size_t)e] * pq[(size_t)e];
      if (f) f[q * E + e] = fq[(size_t)e];
      if (P) P[q * E + e] = pq[(size_t)e];
    }
    loss[q] = alpha * acc;
  }
}

}  // extern "C"
