// Warp-level top-k with renormalised softmax weights (HiNa-MoE, arXiv 2610.05123, §2.1 and §8.1
// Table 3; the reading implemented is softmax over the E logits, top-k, renormalised over the kept
// k: w_j = exp(l_j - m) / sum_kept exp(l_i - m), m the largest kept logit; slot j is the j-th largest
// logit and equal logits go to the lower expert id). Used by the routing kernels and by the fused
// decode-step kernel, which routes its batch in every CTA.
#pragma once

#include <cuda_runtime.h>
#include <math.h>

#include <cstdint>

namespace moe {

__device__ __forceinline__ bool route_better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Order-preserving 32-bit image of a logit (NaN already mapped to -inf; -0 and +0 share +0's image,
// as they compare equal): a larger logit has a larger key. key_value inverts it (-0 comes back as +0).
__device__ __forceinline__ uint32_t ordered_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of kNT tokens by the calling warp: tokens tok0 + t * tok_step (t < kNT; those at or past T
// are skipped). Each lane holds kPer logits of a token (experts lane, lane + 32, ...; kPer = 4 covers
// E <= 128, 8 covers E <= 256) and sorts them once, best first (odd-even merge networks: 5
// compare-exchanges for 4, 19 for 8); every round two warp reductions over the lanes' heads leave the
// winner in all lanes, and the winning lane drops its head. Past E a lane holds
// (-inf, none), which loses to every real expert. Round j's winner of token t goes to
// sel_v[t * sel_step + j] / sel_i[...] (shared memory): per-lane arrays indexed by the round would
// live in local memory. With kNT = 2 the two tokens' dependent reduction chains interleave.
template <int kPer, int kNT>
__device__ __forceinline__ void topk_tokens(const float* __restrict__ logits, int tok0, int tok_step, int T, int E,
                                            int k, int32_t* ids, float* w, float* sel_v, int* sel_i,
                                            int sel_step) {
  static_assert(kPer == 4 || kPer == 8, "4 or 8 logits per lane");
  const int lane = threadIdx.x & 31;
  constexpr int kNone = 0x7fffffff;
  float cv[kNT][kPer];
  int ci[kNT][kPer];
  bool valid[kNT];
#pragma unroll
  for (int t = 0; t < kNT; ++t) {
    const int tok = tok0 + t * tok_step;
    valid[t] = tok < T;  // the same for the whole warp
    const float* l = logits + static_cast<int64_t>(valid[t] ? tok : 0) * E;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = lane + 32 * q;
      const float x = (valid[t] && e < E) ? l[e] : -INFINITY;
      cv[t][q] = (x != x) ? -INFINITY : x;  // NaN orders as -inf (documented: unspecified routing)
      ci[t][q] = e < E ? e : kNone;
    }
  }
  auto cx = [&](float& va, int& ia, float& vb, int& ib) {  // (a, b) in route order
    if (route_better(vb, ib, va, ia)) {
      const float tv = va;
      const int ti = ia;
      va = vb;
      ia = ib;
      vb = tv;
      ib = ti;
    }
  };
#pragma unroll
  for (int t = 0; t < kNT; ++t) {
#define MOE_CX(a, b) cx(cv[t][a], ci[t][a], cv[t][b], ci[t][b])
    if constexpr (kPer == 4) {
      MOE_CX(0, 1); MOE_CX(2, 3);
      MOE_CX(0, 2); MOE_CX(1, 3);
      MOE_CX(1, 2);
    } else {
      MOE_CX(0, 1); MOE_CX(2, 3); MOE_CX(4, 5); MOE_CX(6, 7);
      MOE_CX(0, 2); MOE_CX(1, 3); MOE_CX(4, 6); MOE_CX(5, 7);
      MOE_CX(1, 2); MOE_CX(5, 6);
      MOE_CX(0, 4); MOE_CX(1, 5); MOE_CX(2, 6); MOE_CX(3, 7);
      MOE_CX(2, 4); MOE_CX(3, 5);
      MOE_CX(1, 2); MOE_CX(3, 4); MOE_CX(5, 6);
    }
#undef MOE_CX
  }
  float m[kNT];  // the largest kept logit of each token
  for (int j = 0; j < k; ++j) {
    float bv[kNT];
    int bi[kNT];
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
      // the round's winner over the lanes' heads in two warp reductions: the largest key (an
      // order-preserving 32-bit image of the logit), then the lowest expert id among the heads that
      // hold it (equal logits go to the lower id)
      const uint32_t key = ordered_key(cv[t][0]);
      const uint32_t mk = __reduce_max_sync(0xffffffffu, key);
      const uint32_t wi = __reduce_min_sync(0xffffffffu, key == mk ? static_cast<uint32_t>(ci[t][0]) : 0xffffffffu);
      bv[t] = key_value(mk);
      bi[t] = static_cast<int>(wi);
    }
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
      if ((bi[t] & 31) == lane) {  // the winner was this lane's head
#pragma unroll
        for (int q = 0; q < kPer - 1; ++q) {
          cv[t][q] = cv[t][q + 1];
          ci[t][q] = ci[t][q + 1];
        }
        cv[t][kPer - 1] = -INFINITY;
        ci[t][kPer - 1] = kNone;
      }
      if (j == 0) m[t] = bv[t];
      if (lane == 0 && valid[t]) {
        sel_v[t * sel_step + j] = bv[t];
        sel_i[t * sel_step + j] = bi[t];
      }
    }
  }
  __syncwarp();
  // renormalised softmax over the kept logits: exp(l_j - m) / sum of them
#pragma unroll
  for (int t = 0; t < kNT; ++t) {
    if (!valid[t]) continue;
    const int tok = tok0 + t * tok_step;
    const float* sv = sel_v + t * sel_step;
    const int* si = sel_i + t * sel_step;
    float ex[8];
    float part = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = lane + 32 * q;
      ex[q] = j < k ? expf(__fsub_rn(sv[j], m[t])) : 0.0f;
      part = __fadd_rn(part, ex[q]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, o));
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = lane + 32 * q;
      if (j < k) {
        ids[static_cast<int64_t>(tok) * k + j] = si[j];
        w[static_cast<int64_t>(tok) * k + j] = __fdiv_rn(ex[q], part);
      }
    }
  }
}

}  // namespace moe
