// Plain CPU oracle for decode-phase grouped-query attention (scaled dot-product attention of
// one new query token per sequence against that sequence's key/value cache).
//
// TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's CPU legs may
// load or call this library. The CUDA path never does, and this file shares no code, header,
// table or helper with it.
//
// What it computes (HiNa-MoE arXiv 2610.05123, §6.1 and Figure 9):
//  * Each sequence b has one query token, split into h_q heads of length d. Its keys and
//    values are split into h_kv heads, each an l_seq x d matrix (l_seq = seq_lens[b]).
//  * GQA: a group of G = h_q / h_kv query heads shares one key/value head. Reading taken
//    (the pages do not say which query heads form a group): consecutive query heads share,
//    i.e. query head hq uses key/value head hq / G.
//  * For query head hq and key/value head j = hq / G:
//        s_i = scale * sum_c q[b,hq,c] * K[b,j,i,c]              for i < l_seq
//        p_i = exp(s_i - max_i s_i) / sum_i exp(s_i - max_i s_i)
//        o_c = sum_i p_i * V[b,j,i,c]
//    which is softmax(scale * q K^T) V, the scaled dot-product attention of one query.
//    The pages fix neither the scale nor the precision; the caller passes the scale
//    (1/sqrt(d) in the pages' models) and this oracle computes every sum in float64, in
//    index order, from the bf16 inputs widened exactly.
//  * Output: o rounded once to bf16, round to nearest even; the float64 value is returned too.
//  * An empty sequence (l_seq = 0) has no keys to attend to; reading taken: its output is 0.
//
// Layouts (row-major, the reading of "the framework's native tensor layouts" in §6.1):
//   q   [B, h_q, d]          bf16 bits
//   K,V [B, h_kv, L_cap, d]  bf16 bits; rows i >= seq_lens[b] are never read
//   out [B, h_q, d]          bf16 bits (+ float64 copy)
//
// Parity pins (tests/test_oracle_gqa_pins.py): a hand-worked fixture, a library routine
// (torch's scaled_dot_product_attention in float64 on the CPU), closed forms (one key, equal
// keys, a zero query, a dominating key), invariants (key permutation, contents past the
// sequence length, the query-head to key/value-head mapping).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

double bf16_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// float64 -> bf16 bits, round to nearest, ties to even, in one rounding step (no detour
// through float, which could round twice). bf16 keeps 8 significant bits; its smallest
// quantum (subnormals) is 2^-133; values past the largest finite bf16 round to infinity.
uint16_t double_to_bf16_bits(double x) {
  if (std::isnan(x)) return 0x7fc0;
  if (x == 0.0 || std::isinf(x)) {
    float f = static_cast<float>(x);
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return static_cast<uint16_t>(u >> 16);
  }
  int e = 0;
  std::frexp(x, &e);                      // |x| = m * 2^e, 0.5 <= m < 1
  int qexp = e - 8;                       // quantum of an 8-significant-bit value
  if (qexp < -133) qexp = -133;
  double r = std::nearbyint(std::ldexp(x, -qexp));  // default rounding mode: to nearest even
  double v = std::ldexp(r, qexp);
  const double max_bf16 = std::ldexp(255.0, 120);   // 0x7f7f
  if (std::fabs(v) > max_bf16) v = std::copysign(INFINITY, x);
  float f = static_cast<float>(v);        // exact: v has at most 8 significant bits
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return static_cast<uint16_t>(u >> 16);
}

}  // namespace

extern "C" {

// Decode-phase GQA attention, definition above. Returns 0, or -1 on bad sizes or a sequence
// length outside [0, L_cap].
int oracle_gqa_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* seq_lens,
                      int B, int h_q, int h_kv, int d, int L_cap, float scale, uint16_t* out,
                      double* out_f64) {
  if (B < 0 || h_q < 1 || h_kv < 1 || d < 1 || L_cap < 0 || h_q % h_kv) return -1;
  for (int b = 0; b < B; ++b)
    if (seq_lens[b] < 0 || seq_lens[b] > L_cap) return -1;
  const int G = h_q / h_kv;
  const double sc = static_cast<double>(scale);
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < B; ++b) {
    for (int hq = 0; hq < h_q; ++hq) {
      const int j = hq / G;
      const int n = seq_lens[b];
      const uint16_t* qv = q + (static_cast<long>(b) * h_q + hq) * d;
      const uint16_t* kh = k + (static_cast<long>(b) * h_kv + j) * L_cap * d;
      const uint16_t* vh = v + (static_cast<long>(b) * h_kv + j) * L_cap * d;
      uint16_t* ob = out + (static_cast<long>(b) * h_q + hq) * d;
      double* of = out_f64 ? out_f64 + (static_cast<long>(b) * h_q + hq) * d : nullptr;
      std::vector<double> s(n), o(d, 0.0);
      double m = -INFINITY;
      for (int i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += bf16_to_double(qv[c]) * bf16_to_double(kh[static_cast<long>(i) * d + c]);
        s[i] = sc * acc;
        if (s[i] > m) m = s[i];
      }
      double z = 0.0;
      for (int i = 0; i < n; ++i) {
        s[i] = std::exp(s[i] - m);
        z += s[i];
      }
      for (int i = 0; i < n; ++i)
        for (int c = 0; c < d; ++c) o[c] += s[i] * bf16_to_double(vh[static_cast<long>(i) * d + c]);
      for (int c = 0; c < d; ++c) {
        const double val = n > 0 ? o[c] / z : 0.0;
        ob[c] = double_to_bf16_bits(val);
        if (of) of[c] = val;
      }
    }
  }
  return 0;
}

// float64 -> bf16 bits (RNE, one rounding); tests use it to state expected values.
void oracle_f64_to_bf16(const double* in, long n, uint16_t* out) {
  for (long i = 0; i < n; ++i) out[i] = double_to_bf16_bits(in[i]);
}

}  // extern "C"
