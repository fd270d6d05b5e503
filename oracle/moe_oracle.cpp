// Plain CPU oracle for the routed-expert MoE FFN (decode regime).
//
// TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's
// CPU-baseline leg may load or call this library. The CUDA path never does, and
// this file shares no code, header, table or helper with it.
//
// What it computes, step by step, with the passage each step follows:
//
//  * Routing (HiNa-MoE arXiv 2610.05123, §2.1: a gating function sends each token
//    to a small subset of experts; §8.1 Table 3: Top-2 / Top-8). The pages give no
//    formula. Reading taken: softmax over all E router logits, keep the top-k,
//    renormalise over the kept k. That equals w_j = exp(l_j - m) / sum_sel exp(l_i - m)
//    with m the largest kept logit. Order: descending logit, ties to the lower
//    expert id. Slot j is the j-th largest.
//  * Token gathering into the intermediate matrix I (§4.1, Figure 5): the tokens
//    routed to expert e, in ascending token order ("stable" counting sort:
//    offsets[e] = sum of counts of experts before e).
//  * Expert FFN (§4.1, the FFN equation): FFN(I) = SiLU(I x W_gate) (.) (I x W_up) x W_down,
//    with bf16 inputs and fp32 accumulation (§4.2.1: "Each AMX FMA consumes BF16
//    inputs and accumulates into FP32"). Weights are stored one output row per line
//    with the reduction contiguous (§2.2 Figure 3 "general layout"; Algorithm 1
//    indexes W(n, k)). The intermediate h = SiLU(g) * u is rounded to bf16
//    (round-to-nearest-even) before the down projection; SiLU(g) = g / (1 + exp(-g)).
//  * INT8 variant (§8.1, Figure 11: symmetric group-wise quantisation): the weight
//    is dequantised as w = float(q) * scale[row][k / 128] in fp32, then used as above.
//  * Residual-split variant (RapidMoE, arXiv 2610.01265, "Residual-Split Representation" and
//    "GLU Architecture Adoption"): gate and up are held as a low-precision part W^Q and the
//    quantised residual W^R of W - W^Q, both symmetric group-128 INT8 here (the pages name no
//    bit width), and the high-precision weight is W^H = W^Q + W^R, dequantised as
//    w = float(qQ) * sQ + float(qR) * sR in fp32; gate and up preactivations are therefore
//    W^Q x + W^R x. Down keeps one separately quantised INT8 copy (the pages' "dual
//    quantization" of down_proj, which is not split).
//  * Combine: out[t] = sum over slots j (in slot order) of w_j * y_j, fp32, then
//    rounded once to bf16. The pages leave the combine to the framework (§4.1 ends at
//    "write the output back in the standard row-major layout").
//
// All sums run sequentially in index order in fp32 (the build passes
// -ffp-contract=off so no multiply-add is fused). OpenMP splits only the
// independent outputs (rows) across threads; it never splits a sum.
//
// Parity pins (tests/test_oracle_pins.py): fp64 brute force over all experts with
// masked weights, identity-weight closed form, x = 0, top_k = 1 and top_k = E closed
// forms, identical-expert and token-permutation invariants, power-of-two-scale INT8
// equivalence, hand-worked routing fixtures; residual split (tests/test_oracle_residual_pins.py):
// a zero residual reduces to the INT8 oracle, a zero low part to the BF16 oracle, and gate/up
// preactivations are the sum of the two parts' (linearity).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

namespace {

float bf16_bits_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// float -> bf16, round to nearest, ties to even (NaN stays a quiet NaN).
uint16_t float_to_bf16_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

// One weight element W[row][k] of an expert, as fp32.
//  wtype 0: bf16 bits; wtype 1: int8 with fp32 group scales [rows][K/128].
float weight_at(const void* W, const float* scales, int wtype, int K, long row, long k) {
  if (wtype == 0) {
    const uint16_t* w = static_cast<const uint16_t*>(W);
    return bf16_bits_to_float(w[row * K + k]);
  }
  const int8_t* q = static_cast<const int8_t*>(W);
  float s = scales[row * (K / 128) + k / 128];
  return static_cast<float>(q[row * K + k]) * s;
}

// sum_k a[k] * W[row][k], sequential fp32
float dot_row(const float* a, const void* W, const float* scales, int wtype, int K, long row) {
  float acc = 0.0f;
  for (long k = 0; k < K; ++k) acc += a[k] * weight_at(W, scales, wtype, K, row, k);
  return acc;
}

// Residual-split weight W^H[row][k] = float(qQ) * sQ + float(qR) * sR (int8, group-128 scales).
float residual_weight_at(const int8_t* qQ, const float* sQ, const int8_t* qR, const float* sR, int K, long row,
                         long k) {
  const long g = row * (K / 128) + k / 128;
  return static_cast<float>(qQ[row * K + k]) * sQ[g] + static_cast<float>(qR[row * K + k]) * sR[g];
}

float dot_row_residual(const float* a, const int8_t* qQ, const float* sQ, const int8_t* qR, const float* sR,
                       int K, long row) {
  float acc = 0.0f;
  for (long k = 0; k < K; ++k) acc += a[k] * residual_weight_at(qQ, sQ, qR, sR, K, row, k);
  return acc;
}

float silu(float g) { return g / (1.0f + std::exp(-g)); }

size_t weight_elem_bytes(int wtype) { return wtype == 0 ? 2 : 1; }

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Routing: top-k selection + renormalised softmax weights + counting sort.
//   logits [T,E] f32 -> ids [T,k], w [T,k], counts [E], offsets [E+1],
//   sorted_token [T*k], inv_pos [T,k], active [E] (first *num_active used).
// Returns 0, or -1 on bad sizes.
int oracle_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                 int32_t* counts, int32_t* offsets, int32_t* sorted_token, int32_t* inv_pos,
                 int32_t* active, int32_t* num_active) {
  if (T < 0 || E < 1 || k < 1 || k > E) return -1;
  std::vector<int> order(E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + static_cast<long>(t) * E;
    std::iota(order.begin(), order.end(), 0);
    // descending logit; stable, so equal logits keep ascending expert id
    std::stable_sort(order.begin(), order.end(), [l](int a, int b) { return l[a] > l[b]; });
    float m = l[order[0]];
    float denom = 0.0f;
    for (int j = 0; j < k; ++j) denom += std::exp(l[order[j]] - m);
    for (int j = 0; j < k; ++j) {
      ids[t * k + j] = order[j];
      w[t * k + j] = std::exp(l[order[j]] - m) / denom;
    }
  }
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long a = 0; a < static_cast<long>(T) * k; ++a) counts[ids[a]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> cursor(offsets, offsets + E);
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      int e = ids[t * k + j];
      int p = cursor[e]++;
      sorted_token[p] = t;
      inv_pos[t * k + j] = p;
    }
  }
  int n = 0;
  for (int e = 0; e < E; ++e)
    if (counts[e] > 0) active[n++] = e;
  *num_active = n;
  return 0;
}

// ---------------------------------------------------------------------------
// Gate/up projection of one token through one expert:
//   g_i = sum_c x[c] * Wg[i][c],  u_i = sum_c x[c] * Wu[i][c]   (fp32)
//   h_i = bf16(SiLU(g_i) * u_i)
// x: H bf16 bits. Wg/Wu: that expert's [I,H] weights. sg/su: its [I,H/128] scales
// (int8 only). h_out: I bf16 bits. g_out/u_out (optional): fp32 g, u.
void oracle_gateup_token(const uint16_t* x, const void* Wg, const void* Wu, const float* sg,
                         const float* su, int wtype, int H, int I, uint16_t* h_out,
                         float* g_out, float* u_out) {
  std::vector<float> xf(H);
  for (int c = 0; c < H; ++c) xf[c] = bf16_bits_to_float(x[c]);
#pragma omp parallel for schedule(static)
  for (int i = 0; i < I; ++i) {
    float g = dot_row(xf.data(), Wg, sg, wtype, H, i);
    float u = dot_row(xf.data(), Wu, su, wtype, H, i);
    h_out[i] = float_to_bf16_bits(silu(g) * u);
    if (g_out) g_out[i] = g;
    if (u_out) u_out[i] = u;
  }
}

// Down projection of one token's intermediate through one expert:
//   y_r = sum_i h[i] * Wd[r][i]   (fp32)
// h: I bf16 bits. Wd: that expert's [H,I] weights. sd: its [H,I/128] scales.
void oracle_down_token(const uint16_t* h, const void* Wd, const float* sd, int wtype, int H,
                       int I, float* y_out) {
  std::vector<float> hf(I);
  for (int i = 0; i < I; ++i) hf[i] = bf16_bits_to_float(h[i]);
#pragma omp parallel for schedule(static)
  for (int r = 0; r < H; ++r) y_out[r] = dot_row(hf.data(), Wd, sd, wtype, I, r);
}

// Combine of one token: out[r] = bf16(sum_j w[j] * y[j][r]) in slot order (fp32).
// y: k rows of H fp32. out_f32 (optional): the fp32 sum before rounding.
void oracle_combine_token(const float* y, const float* w, int k, int H, uint16_t* out,
                          float* out_f32) {
  for (int r = 0; r < H; ++r) {
    float acc = 0.0f;
    for (int j = 0; j < k; ++j) acc += w[j] * y[static_cast<long>(j) * H + r];
    out[r] = float_to_bf16_bits(acc);
    if (out_f32) out_f32[r] = acc;
  }
}

// ---------------------------------------------------------------------------
// Whole routed-expert FFN for T tokens.
//   x [T,H] bf16, logits [T,E] f32, Wg/Wu [E,I,H], Wd [E,H,I] (bf16 bits or int8),
//   sg/su [E,I,H/128], sd [E,H,I/128] (int8 only) -> out [T,H] bf16 (+ fp32 copy).
// Optional intermediates (may be null): ids/w [T,k]; h [T,k,I] bf16; y [T,k,H] f32.
int oracle_forward(const uint16_t* x, const float* logits, const void* Wg, const void* Wu,
                   const void* Wd, const float* sg, const float* su, const float* sd, int wtype,
                   int T, int H, int I, int E, int k, uint16_t* out, float* out_f32,
                   int32_t* ids_out, float* w_out, uint16_t* h_out, float* y_out) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1 || k > E) return -1;
  if (wtype != 0 && wtype != 1) return -1;
  if (wtype == 1 && (H % 128 || I % 128)) return -1;
  if (T == 0) return 0;
  const long P = static_cast<long>(T) * k;
  std::vector<int32_t> ids(P), counts(E), offsets(E + 1), sorted_token(P), inv_pos(P), active(E);
  std::vector<float> w(P);
  int32_t num_active = 0;
  oracle_route(logits, T, E, k, ids.data(), w.data(), counts.data(), offsets.data(),
               sorted_token.data(), inv_pos.data(), active.data(), &num_active);
  const size_t eb = weight_elem_bytes(wtype);
  const size_t w_expert = static_cast<size_t>(I) * H * eb;  // bytes of one expert's matrix
  const size_t s_gu = static_cast<size_t>(I) * (H / 128);   // scales per expert, gate/up
  const size_t s_d = static_cast<size_t>(H) * (I / 128);    // scales per expert, down
  std::vector<uint16_t> h(I);
  std::vector<float> y(static_cast<size_t>(k) * H);
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      const int e = ids[t * k + j];
      const char* wg = static_cast<const char*>(Wg) + e * w_expert;
      const char* wu = static_cast<const char*>(Wu) + e * w_expert;
      const char* wd = static_cast<const char*>(Wd) + e * w_expert;
      oracle_gateup_token(x + static_cast<long>(t) * H, wg, wu, wtype ? sg + e * s_gu : nullptr,
                          wtype ? su + e * s_gu : nullptr, wtype, H, I, h.data(), nullptr,
                          nullptr);
      oracle_down_token(h.data(), wd, wtype ? sd + e * s_d : nullptr, wtype, H, I,
                        y.data() + static_cast<size_t>(j) * H);
      if (h_out) std::memcpy(h_out + (static_cast<size_t>(t) * k + j) * I, h.data(), I * 2);
    }
    if (y_out) std::memcpy(y_out + static_cast<size_t>(t) * k * H, y.data(), y.size() * 4);
    oracle_combine_token(y.data(), w.data() + static_cast<long>(t) * k, k, H,
                         out + static_cast<long>(t) * H,
                         out_f32 ? out_f32 + static_cast<long>(t) * H : nullptr);
  }
  if (ids_out) std::memcpy(ids_out, ids.data(), P * 4);
  if (w_out) std::memcpy(w_out, w.data(), P * 4);
  return 0;
}

// ---------------------------------------------------------------------------
// Residual-split gate/up of one token through one expert (definition at the top):
//   g_i = sum_c x[c] * (qQg * sQg + qRg * sRg)[i][c], u likewise, h_i = bf16(SiLU(g_i) * u_i).
// qQ*/qR*: that expert's [I,H] int8 parts; sQ*/sR*: their [I,H/128] scales.
void oracle_gateup_token_residual(const uint16_t* x, const int8_t* qQg, const float* sQg, const int8_t* qRg,
                                  const float* sRg, const int8_t* qQu, const float* sQu, const int8_t* qRu,
                                  const float* sRu, int H, int I, uint16_t* h_out, float* g_out, float* u_out) {
  std::vector<float> xf(H);
  for (int c = 0; c < H; ++c) xf[c] = bf16_bits_to_float(x[c]);
#pragma omp parallel for schedule(static)
  for (int i = 0; i < I; ++i) {
    float g = dot_row_residual(xf.data(), qQg, sQg, qRg, sRg, H, i);
    float u = dot_row_residual(xf.data(), qQu, sQu, qRu, sRu, H, i);
    h_out[i] = float_to_bf16_bits(silu(g) * u);
    if (g_out) g_out[i] = g;
    if (u_out) u_out[i] = u;
  }
}

// Whole routed-expert FFN with residual-split gate/up (INT8 + INT8 residual) and INT8 down:
// routing, gather and combine as in oracle_forward; W_gate/W_up [E,I,H] int8 with their residual
// parts Wr_gate/Wr_up and scales [E,I,H/128] each; W_down [E,H,I] int8, s_down [E,H,I/128].
int oracle_forward_residual(const uint16_t* x, const float* logits, const int8_t* Wg, const float* sg,
                            const int8_t* Wgr, const float* sgr, const int8_t* Wu, const float* su,
                            const int8_t* Wur, const float* sur, const int8_t* Wd, const float* sd, int T, int H,
                            int I, int E, int k, uint16_t* out, float* out_f32) {
  if (T < 0 || H < 128 || I < 128 || E < 1 || k < 1 || k > E || H % 128 || I % 128) return -1;
  if (T == 0) return 0;
  const long P = static_cast<long>(T) * k;
  std::vector<int32_t> ids(P), counts(E), offsets(E + 1), sorted_token(P), inv_pos(P), active(E);
  std::vector<float> w(P);
  int32_t num_active = 0;
  oracle_route(logits, T, E, k, ids.data(), w.data(), counts.data(), offsets.data(), sorted_token.data(),
               inv_pos.data(), active.data(), &num_active);
  const size_t n_e = static_cast<size_t>(I) * H;          // elements of one expert's matrix
  const size_t s_gu = static_cast<size_t>(I) * (H / 128);  // scales per expert, gate/up
  const size_t s_d = static_cast<size_t>(H) * (I / 128);   // scales per expert, down
  std::vector<uint16_t> h(I);
  std::vector<float> y(static_cast<size_t>(k) * H);
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      const int e = ids[t * k + j];
      oracle_gateup_token_residual(x + static_cast<long>(t) * H, Wg + e * n_e, sg + e * s_gu, Wgr + e * n_e,
                                   sgr + e * s_gu, Wu + e * n_e, su + e * s_gu, Wur + e * n_e, sur + e * s_gu, H,
                                   I, h.data(), nullptr, nullptr);
      oracle_down_token(h.data(), Wd + e * n_e, sd + e * s_d, 1, H, I, y.data() + static_cast<size_t>(j) * H);
    }
    oracle_combine_token(y.data(), w.data() + static_cast<long>(t) * k, k, H, out + static_cast<long>(t) * H,
                         out_f32 ? out_f32 + static_cast<long>(t) * H : nullptr);
  }
  return 0;
}

// Round fp32 values to bf16 bits (RNE); used by tests to state expected values.
void oracle_f32_to_bf16(const float* in, long n, uint16_t* out) {
  for (long i = 0; i < n; ++i) out[i] = float_to_bf16_bits(in[i]);
}

}  // extern "C"
