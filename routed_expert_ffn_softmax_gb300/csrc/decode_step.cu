// The whole routed-expert FFN of a decode step in one persistent launch, for batches whose experts
// see few tokens each (about one or two).
//
// HiNa-MoE (arXiv 2610.05123): routing (§2.1; Top-k of §8.1 Table 3, read as softmax over the E
// logits, top-k, renormalised over the kept k), the per-expert token block (§4.1, Figure 5), the FFN
// equation of §4.1, FFN(I) = SiLU(I x W_gate) (.) (I x W_up) x W_down, with bf16 inputs and fp32
// accumulation (§4.2.1), h rounded to bf16 before the down projection, and the routing-weighted
// combine back to row-major token order. INT8 weights: symmetric group-128 quantisation (§8.1,
// Figure 11), w = q * s.
//
// At one or two tokens per expert the FFN is a matrix-vector product: every weight is used once
// per token, so the tensor cores have nothing to amortise and the kernel's job is to move the
// active experts' weights through HBM once, at full rate, with as little fixed cost per step as
// possible. The usual sequence (routing, gather, gate+up, down, combine, each its own launch)
// costs a launch boundary and a start-up per kernel, which at one token per expert is most of the
// step. Here one launch does all of it:
//   1. every CTA routes the whole batch itself (top-k per token by a warp, counts, offsets, the
//      stable expert-major order), so no CTA waits for another to learn the routing;
//   2. gate+up: the (expert pass, 128-row block, 128-byte reduction slice) tiles of all active
//      experts are cut into equal contiguous ranges per CTA (stream-K); a unit split between CTAs
//      is finished by its last-arriving CTA in a fixed order;
//   3. one grid-wide barrier (h complete): while waiting, the producer already streams the CTA's
//      first down-projection weight tiles, which do not depend on h;
//   4. down, cut the same way, row-block-major; the CTA that completes the last unit of a 128-row
//      block of the output writes that block's combine (fixed slot order, no atomics on data).
// Per CTA (one per SM; a cooperative launch, so all CTAs are resident for the barrier):
//   warps 0..15  compute: thread = (weight row r of the tile, quarter q of its 128-byte slice);
//                mixed-precision FMAs (fma.rn.f32.bf16 / .f16: exact products, fp32 sums) read
//                the weights straight from the TMA-filled tile and the tokens from the slot;
//   warp 16      producer: TMA tensor loads of the weight tiles (and INT8 scale boxes), bulk
//                copies of the tokens' slices (x for gate+up, h for down) into the same slot.
// INT8 weights become exact fp16 values (one logic op, two byte permutes, two fp16x2 subtractions
// per four weights); the tokens are fp16 copies of the bf16 values, scaled by a power of two (a row
// scale for x, a scale per 128-element group for h) that the epilogue multiplies back.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <atomic>
#include <cstdint>
#include <type_traits>

#include "decode_device.cuh"
#include "moe_launch.h"
#include "route_topk.cuh"

namespace moe {
namespace dec {

constexpr int kNE = 8;                                // tokens per pass of an expert
constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = 32 * kComputeWarps;  // 128 rows x 4 quarters
constexpr int kProducerWarp = kComputeWarps;
constexpr int kThreads = kComputeThreads + 32;
constexpr int kRec = 272;  // INT8 h record: 128 fp16 values, the fp32 group scale, padding to 16 B

template <bool kInt8>
struct Geo {
  static constexpr int kKt = kInt8 ? 128 : 64;          // reduction elements per 128-byte tile row
  static constexpr int kWBytes = 32768;                 // two 128-row x 128-byte weight boxes
  static constexpr int kScaleBytes = kInt8 ? 4096 : 0;  // INT8: two {4 groups x 128 rows} fp32 boxes
  static constexpr int kSliceGU = kInt8 ? 256 : 128;    // token bytes per slot, gate+up (x)
  static constexpr int kSliceDN = kInt8 ? 2 * kRec : 256;  // and down (h: two reduction slices)
  static constexpr int kSliceMax = kSliceGU > kSliceDN ? kSliceGU : kSliceDN;
  static constexpr int kTokOff = kWBytes + kScaleBytes;
  static constexpr int kSlot = (kTokOff + kNE * kSliceMax + 1023) / 1024 * 1024;
  static constexpr int kStages = kInt8 ? 5 : 6;
  static_assert(kSlot % 1024 == 0, "slots keep the 1024-byte alignment of the 128B swizzle");
};

struct Shared {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t gbar_arrived;  // compute -> producer: this CTA has arrived at the grid barrier
  int gbar_epoch;         // the barrier's release word as read before arriving
  int flag;               // broadcast word of the epilogues
  float xs[kDecodeMaxT];  // INT8: the power of two each token's fp16 copy was divided by
  uint32_t need;          // INT8: tokens this CTA converts (bit t)
  int A;                  // active experts
  int ids[kDecodeMaxP];   // token t's experts at t * k .. t * k + k - 1 (slot order)
  float w[kDecodeMaxP];
  int inv[kDecodeMaxP];
  int sorted[kDecodeMaxP];
  float selv[kDecodeMaxP];
  int seli[kDecodeMaxP];
  int cnt[256];
  int off[257];
  uint32_t tokmask[256];
  int act_e[256];
  int pp[257];            // prefix sums of the passes of the active experts
  float red[2][kComputeWarps][kNE];
};

template <bool kInt8>
constexpr int smem_bytes() {
  return Geo<kInt8>::kStages * Geo<kInt8>::kSlot + static_cast<int>(sizeof(Shared));
}
static_assert(smem_bytes<false>() <= 232448 && smem_bytes<true>() <= 232448, "dynamic shared memory per CTA");

// One unit: pass `np` of the a-th active expert (tokens at sorted positions p0 .. p0 + n - 1) and a
// 128-row block of the output rows.
struct Unit {
  int e, p0, n, rb;
};

__device__ __forceinline__ Unit unit_of(const Shared& S, int q, int rb) {
  int lo = 0, hi = S.A - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.pp[mid] <= q) lo = mid; else hi = mid - 1;
  }
  Unit u;
  u.e = S.act_e[lo];
  const int np = q - S.pp[lo];
  u.p0 = S.off[u.e] + np * kNE;
  const int left = S.cnt[u.e] - np * kNE;
  u.n = left < kNE ? left : kNE;
  u.rb = rb;
  return u;
}

// Grid barrier that leaves itself reset: the CTA reads the release word, arrives on the counter, and
// the last arriver zeroes the counter and advances the release word. Returns the word read (a waiter
// spins, bounded, while the release word still holds it).
__device__ __forceinline__ int grid_arrive(int32_t* gbar, int nctas) {
  const int e = ld_relaxed_gpu(gbar + 1);
  __threadfence();
  const int old = atomicAdd(gbar, 1);
  if (old == nctas - 1) {
    atomicExch(gbar, 0);
    __threadfence();
    st_release_gpu(gbar + 1, e + 1);
  }
  return e;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Largest |v| over the 32 lanes (v >= 0).
__device__ __forceinline__ float warp_max_abs(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// k with max * 2^-k in [2^14, 2^15) (fp16 keeps every bf16 value from max down to max * 2^-29 exactly),
// clamped so that 2^k and 2^-k are normal fp32 numbers; 0 for an all-zero or non-finite group.
__device__ __forceinline__ int f16_exponent(float m) {
  int k = 0;
  if (m > 0.0f && m <= 3.0e38f) {
    int e = 0;
    frexpf(m, &e);
    k = e - 15;
    k = k < -100 ? -100 : (k > 127 ? 127 : k);
  }
  return k;
}

template <bool kInt8>
__global__ void __launch_bounds__(kThreads, 1)
    decode_step_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmU,
                       const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmSG,
                       const __grid_constant__ CUtensorMap tmSU, const __grid_constant__ CUtensorMap tmSD,
                       const DecodeArgs a) {
  using G = Geo<kInt8>;
  extern __shared__ __align__(1024) uint8_t smem[];
  Shared& S = *reinterpret_cast<Shared*>(smem + G::kStages * G::kSlot);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int T = a.T, E = a.E, k = a.k, H = a.H, I = a.I;
  const int P = T * k;
  const int N = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);

  if (tid == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(&S.full[s], 1);               // producer's expect_tx
      mbar_init(&S.empty[s], kComputeWarps);  // one arrival per compute warp
    }
    mbar_init(&S.gbar_arrived, 1);
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmG);
    tma_prefetch_desc(&tmU);
    tma_prefetch_desc(&tmD);
    if (kInt8) {
      tma_prefetch_desc(&tmSG);
      tma_prefetch_desc(&tmSU);
      tma_prefetch_desc(&tmSD);
    }
  }
  // warm the logits in L2 (a line still being written by the predecessor is updated there)
  for (int i = tid; i * 32 < T * E; i += kThreads)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.logits + i * 32));
  for (int i = tid; i < 256; i += kThreads) {
    S.cnt[i] = 0;
    S.tokmask[i] = 0u;
  }
  pdl_wait_predecessor();
  pdl_allow_successor();
  // the status word starts each call at 0 (a wait gives up only after kWaitLimitNs, long after every
  // CTA of this cooperative launch has passed this point)
  if (cta == 0 && tid == 0) *a.status = 0;
  __syncthreads();

  // ============================ 1. routing (every CTA) ============================
  if (warp < kComputeWarps) {
    for (int tok = warp; tok < T; tok += kComputeWarps) {
      if (E <= 128)
        topk_tokens<4, 1>(a.logits, tok, 0, T, E, k, S.ids, S.w, S.selv + tok * k, S.seli + tok * k, 0);
      else
        topk_tokens<8, 1>(a.logits, tok, 0, T, E, k, S.ids, S.w, S.selv + tok * k, S.seli + tok * k, 0);
    }
  }
  __syncthreads();
  for (int i = tid; i < P; i += kThreads) {
    const int e = S.ids[i];
    atomicAdd(&S.cnt[e], 1);
    atomicOr(&S.tokmask[e], 1u << (i / k));
  }
  __syncthreads();
  if (warp == 0) {  // exclusive offsets, active list and pass counts, 32 experts at a time
    int run = 0, nact = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int c = e < E ? S.cnt[e] : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      const uint32_t act = __ballot_sync(0xffffffffu, c > 0);
      if (e < E) {
        S.off[e] = run + incl - c;
        if (c > 0) {
          const int ai = nact + __popc(act & ((1u << lane) - 1u));
          S.act_e[ai] = e;
          S.pp[ai + 1] = (c + kNE - 1) / kNE;
        }
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      nact += __popc(act);
    }
    if (lane == 0) {
      S.off[E] = run;
      S.A = nact;
      S.pp[0] = 0;
      for (int i = 1; i <= nact; ++i) S.pp[i] += S.pp[i - 1];
    }
  }
  __syncthreads();
  for (int i = tid; i < P; i += kThreads) {  // stable expert-major order
    const int t = i / k;
    const int e = S.ids[i];
    const int p = S.off[e] + __popc(S.tokmask[e] & ((1u << t) - 1u));
    S.sorted[p] = t;
    S.inv[i] = p;
  }
  __syncthreads();
  const int A = S.A;
  const int NU = S.pp[A];  // (expert, pass) pairs
  if (cta == 0) {          // the routing tables, for callers that read them from the workspace
    for (int i = tid; i < P; i += kThreads) {
      a.ids[i] = S.ids[i];
      a.w[i] = S.w[i];
      a.inv_pos[i] = S.inv[i];
      a.sorted_token[i] = S.sorted[i];
    }
    for (int e = tid; e < E; e += kThreads) {
      a.counts[e] = S.cnt[e];
      a.offsets[e] = S.off[e];
    }
    for (int i = tid; i < A; i += kThreads) a.active[i] = S.act_e[i];
    if (tid == 0) {
      a.offsets[E] = S.off[E];
      *a.num_active = A;
    }
  }

  // ============================ schedule ============================
  const int RBg = I / 128, KIg = H / G::kKt;        // gate+up: rows of I, reduction H
  const int RBd = H / 128, KId = I / (2 * G::kKt);  // down: rows of H, reduction I (two slices per slot)
  const int64_t Wg = static_cast<int64_t>(NU) * RBg * KIg;
  const int64_t Wd = static_cast<int64_t>(NU) * RBd * KId;
  const int64_t NCg = Wg < N ? Wg : N, NCd = Wd < N ? Wd : N;
  const int64_t g_beg = cta < NCg ? cta * Wg / NCg : 0, g_end = cta < NCg ? (cta + 1) * Wg / NCg : 0;
  const int64_t d_beg = cta < NCd ? cta * Wd / NCd : 0, d_end = cta < NCd ? (cta + 1) * Wd / NCd : 0;
  // gate+up units are pass-major (q * RBg + rb): a CTA's range touches few experts' tokens;
  // down units are row-block-major (rb * NU + q): a row block's combine becomes ready as soon as
  // its last unit is done, spread over the step instead of all at its end.
  auto gu_unit = [&](int64_t u) { return unit_of(S, static_cast<int>(u / RBg), static_cast<int>(u % RBg)); };
  auto dn_unit = [&](int64_t u) { return unit_of(S, static_cast<int>(u % NU), static_cast<int>(u / NU)); };

  // INT8: fp16 copies of the token rows this CTA's gate+up tiles read, each divided by a power of
  // two that brings its largest value into [2^14, 2^15). CTAs that share a token write the same
  // bytes; each CTA reads only rows it has written itself.
  if (kInt8) {
    if (tid == 0) {
      uint32_t need = 0u;
      if (g_beg < g_end) {
        const int q0 = static_cast<int>((g_beg / KIg) / RBg), q1 = static_cast<int>(((g_end - 1) / KIg) / RBg);
        const Unit u0 = unit_of(S, q0, 0), u1 = unit_of(S, q1, 0);
        for (int p = u0.p0; p < u1.p0 + u1.n; ++p) need |= 1u << S.sorted[p];
      }
      S.need = need;
    }
    __syncthreads();
    if (warp < kComputeWarps) {
      const uint32_t need = S.need;
      const int nn = __popc(need);
      for (int j = warp; j < nn; j += kComputeWarps) {
        uint32_t m = need;
        for (int z = 0; z < j; ++z) m &= m - 1u;
        const int t = __ffs(m) - 1;
        const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t) * H);
        float mx = 0.0f;
        for (int c = lane; c < H / 8; c += 32) {
          const uint4 v = src[c];
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            mx = fmaxf(mx, fabsf(__uint_as_float(wv[i] << 16)));
            mx = fmaxf(mx, fabsf(__uint_as_float(wv[i] & 0xffff0000u)));
          }
        }
        mx = warp_max_abs(mx);
        const int kx = f16_exponent(mx);
        const float down = ldexpf(1.0f, -kx);
        uint4* dst = reinterpret_cast<uint4*>(a.x16 + static_cast<int64_t>(t) * H);
        for (int c = lane; c < H / 8; c += 32) {
          const uint4 v = src[c];
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 h2 = __floats2half2_rn(__uint_as_float(wv[i] << 16) * down,
                                                 __uint_as_float(wv[i] & 0xffff0000u) * down);
            o[i] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (lane == 0) S.xs[t] = ldexpf(1.0f, kx);
      }
      fence_proxy_async_global();  // the producer's bulk copies of these rows come after the barrier
    }
    named_bar_sync(1, kThreads);
  }

  if (warp == kProducerWarp) {
    // ================================ producer ================================
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      uint8_t* const slots = smem;
      int slot = 0;
      uint32_t ph = 0;
      int64_t used = 0;
      bool ok = true;
      auto advance = [&]() {
        ++used;
        if (++slot == G::kStages) {
          slot = 0;
          ph ^= 1u;
        }
      };
      // ---- gate+up tiles
      for (int64_t i = g_beg; i < g_end && ok; ++i) {
        const int64_t u = i / KIg;
        const int kk = static_cast<int>(i - u * KIg);
        const Unit un = gu_unit(u);
        if (!mbar_wait(&S.empty[slot], ph ^ 1u)) {
          ok = false;
          atomicExch(a.status, kStatusWaitEmptyTimeout);
          break;
        }
        uint8_t* st = slots + slot * G::kSlot;
        mbar_arrive_expect_tx(&S.full[slot], G::kWBytes + G::kScaleBytes + un.n * G::kSliceGU);
        tma_load_3d(st, &tmG, &S.full[slot], kk * G::kKt, un.rb * 128, un.e, pol);
        tma_load_3d(st + 16384, &tmU, &S.full[slot], kk * G::kKt, un.rb * 128, un.e, pol);
        if (kInt8) {
          tma_load_3d_plain(st + G::kWBytes, &tmSG, &S.full[slot], kk & ~3, un.rb * 128, un.e);
          tma_load_3d_plain(st + G::kWBytes + 2048, &tmSU, &S.full[slot], kk & ~3, un.rb * 128, un.e);
        }
        for (int t = 0; t < un.n; ++t) {
          const int tok = S.sorted[un.p0 + t];
          const uint16_t* src = (kInt8 ? a.x16 : a.x) + static_cast<int64_t>(tok) * H + kk * G::kKt;
          bulk_g2s(st + G::kTokOff + t * G::kSliceGU, src, G::kSliceGU, &S.full[slot]);
        }
        advance();
      }
      // ---- down tiles: weights as slots free up; the h slices once the grid barrier is passed
      int pend_slot[8];
      int64_t pend_i[8];
      int npend = 0;
      bool passed = false;
      auto issue_h = [&](int sl, int64_t i) {
        const int64_t u = i / KId;
        const int kk2 = static_cast<int>(i - u * KId);
        const Unit un = dn_unit(u);
        uint8_t* st = slots + sl * G::kSlot;
        for (int t = 0; t < un.n; ++t) {
          const int p = un.p0 + t;
          const void* src;
          if (kInt8)
            src = static_cast<const uint8_t*>(a.h) + (static_cast<int64_t>(p) * (I / 128) + 2 * kk2) * kRec;
          else
            src = static_cast<const uint16_t*>(a.h) + static_cast<int64_t>(p) * I + kk2 * 128;
          bulk_g2s(st + G::kTokOff + t * G::kSliceDN, src, G::kSliceDN, &S.full[sl]);
        }
      };
      // the grid barrier has been passed: every CTA's h is written (acquire, then order the async
      // proxy's later reads after it)
      auto barrier_ready = [&]() -> bool {
        if (!mbar_try_wait(&S.gbar_arrived, 0)) return false;
        return ld_acquire_gpu(a.gbar + 1) != *reinterpret_cast<volatile int*>(&S.gbar_epoch);
      };
      auto release_pending = [&]() {
        fence_proxy_async_global();
        passed = true;
        for (int j = 0; j < npend; ++j) issue_h(pend_slot[j], pend_i[j]);
        npend = 0;
      };
      // wait for a free slot, issuing the pending h slices as soon as the barrier opens (the slots
      // they complete are the ones the compute warps wait for)
      auto wait_slot = [&]() -> bool {
        const uint64_t t0 = global_timer_ns();
        uint64_t tb = t0;
        for (;;) {
          if (mbar_try_wait(&S.empty[slot], ph ^ 1u)) return true;
          if (!passed && npend > 0) {
            if (barrier_ready()) {
              release_pending();
              tb = global_timer_ns();
              continue;
            }
            if (global_timer_ns() - tb > a.grid_wait_ns) {  // the barrier never opened: go on without it
              atomicExch(a.status, kStatusGridTimeout);
              release_pending();
              tb = global_timer_ns();
              continue;
            }
          }
          if ((passed || npend == 0) && global_timer_ns() - t0 > 2 * kWaitLimitNs) return false;
        }
      };
      for (int64_t i = d_beg; i < d_end && ok; ++i) {
        if (!wait_slot()) {
          ok = false;
          atomicExch(a.status, kStatusWaitEmptyTimeout);
          break;
        }
        const int64_t u = i / KId;
        const int kk2 = static_cast<int>(i - u * KId);
        const Unit un = dn_unit(u);
        uint8_t* st = slots + slot * G::kSlot;
        mbar_arrive_expect_tx(&S.full[slot], G::kWBytes + (kInt8 ? 2048 : 0) + un.n * G::kSliceDN);
        tma_load_3d(st, &tmD, &S.full[slot], 2 * kk2 * G::kKt, un.rb * 128, un.e, pol);
        tma_load_3d(st + 16384, &tmD, &S.full[slot], (2 * kk2 + 1) * G::kKt, un.rb * 128, un.e, pol);
        if (kInt8) tma_load_3d_plain(st + G::kWBytes, &tmSD, &S.full[slot], (2 * kk2) & ~3, un.rb * 128, un.e);
        if (passed) {
          issue_h(slot, i);
        } else {
          pend_slot[npend] = slot;
          pend_i[npend] = i;
          ++npend;
        }
        advance();
      }
      if (!passed && npend > 0) {
        const uint64_t t0 = global_timer_ns();
        while (!barrier_ready()) {
          if (global_timer_ns() - t0 > a.grid_wait_ns) {
            atomicExch(a.status, kStatusGridTimeout);
            break;
          }
        }
        release_pending();
      }
      // never leave copies in flight: wait for the last uses of every slot to land
      const int64_t n = used < G::kStages ? used : G::kStages;
      int s = slot;
      uint32_t p2 = ph;
      for (int64_t j = 0; j < n; ++j) {
        if (--s < 0) {
          s = G::kStages - 1;
          p2 ^= 1u;
        }
        if (!mbar_wait(&S.full[s], p2)) {
          atomicExch(a.status, kStatusDrainTimeout);
          break;
        }
      }
    }
    __syncwarp();
  } else {
    // ================================ compute ================================
    const int r = tid >> 2;  // weight row of the tile
    const int q = tid & 3;   // quarter of the row's 128-byte slice
    const int x7 = r & 7;
    const uint32_t sbase = smem_addr(smem);
    int slot = 0;
    uint32_t ph = 0;
    bool ok = true;
    int red_buf = 0;
    auto take = [&]() -> uint32_t {  // wait for the next slot; its shared-memory address
      if (ok && !mbar_wait(&S.full[slot], ph)) {
        ok = false;
        atomicExch(a.status, kStatusWaitFullTimeout);
      }
      return sbase + slot * G::kSlot;
    };
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      if (++slot == G::kStages) {
        slot = 0;
        ph ^= 1u;
      }
    };
    auto cta_of = [](int64_t i, int64_t W, int64_t NC) -> int64_t { return ((i + 1) * NC - 1) / W; };

    // Split-unit hand-off: publish this CTA's partial sums (vals[t][m], m < kM) and let the last of
    // the unit's CTAs sum all pieces in CTA order. Returns true in the CTA that must finish the unit
    // (vals then holds the full sums in its quarter-0 threads).
    auto split_unit = [&](auto& vals, auto kMc, int64_t ub, int64_t ue, int64_t beg, int64_t W, int64_t NC,
                          int64_t KI) -> bool {
      constexpr int kM = decltype(kMc)::value;
      const int64_t c_first = cta_of(ub, W, NC), c_last = cta_of(ue - 1, W, NC);
      const int sl = (ub / KI == beg / KI) ? 0 : 1;
      float* mine = a.partials + (static_cast<int64_t>(cta) * 2 + sl) * kPartialSlotFloats;
      if (q == 0) {
#pragma unroll
        for (int t = 0; t < kNE; ++t)
#pragma unroll
          for (int m = 0; m < kM; ++m) mine[(t * 2 + m) * 128 + r] = vals[t][m];
      }
      __threadfence();
      named_bar_sync(2, kComputeThreads);
      if (tid == 0) {
        __threadfence();
        const int old = atomicAdd(&a.counters[c_first], 1);
        const int last = old == static_cast<int>(c_last - c_first);
        if (last) a.counters[c_first] = 0;
        S.flag = last;
      }
      named_bar_sync(2, kComputeThreads);
      const bool last = S.flag != 0;
      named_bar_sync(2, kComputeThreads);  // S.flag is reused by the next hand-off
      if (!last) return false;
      __threadfence();
      if (q == 0) {
#pragma unroll
        for (int t = 0; t < kNE; ++t)
#pragma unroll
          for (int m = 0; m < kM; ++m) vals[t][m] = 0.0f;
        for (int64_t c = c_first; c <= c_last; ++c) {
          const int cs = (ub / KI == (c * W / NC) / KI) ? 0 : 1;
          const float* src = a.partials + (c * 2 + cs) * kPartialSlotFloats;
#pragma unroll
          for (int t = 0; t < kNE; ++t)
#pragma unroll
            for (int m = 0; m < kM; ++m) vals[t][m] += __ldcg(src + (t * 2 + m) * 128 + r);
        }
      }
      return true;
    };

    // ---------------------------- gate+up ----------------------------
    for (int64_t i = g_beg; i < g_end;) {
      const int64_t u = i / KIg;
      const int64_t ub = u * KIg, ue = ub + KIg;
      const int64_t pe = ue < g_end ? ue : g_end;
      const Unit un = gu_unit(u);
      float acc[kNE][2];  // gate, up (INT8: sums of scaled group sums)
#pragma unroll
      for (int t = 0; t < kNE; ++t) acc[t][0] = acc[t][1] = 0.0f;
      for (; i < pe; ++i) {
        const uint32_t st = take();
        const uint32_t rowg = st + r * 128, rowu = rowg + 16384;
        const uint32_t c0 = ((2 * q) ^ x7) << 4, c1 = ((2 * q + 1) ^ x7) << 4;
        const uint4 g0 = lds128(rowg + c0), g1 = lds128(rowg + c1);
        const uint4 u0 = lds128(rowu + c0), u1 = lds128(rowu + c1);
        if constexpr (!kInt8) {
          const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          const uint32_t uw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          const uint32_t tb = st + G::kTokOff + q * 32;
#pragma unroll
          for (int t = 0; t < kNE; ++t) {
            if (t < un.n) {
              const uint4 xa = lds128(tb + t * G::kSliceGU), xb = lds128(tb + t * G::kSliceGU + 16);
              const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
              float ga = acc[t][0], gb = 0.0f, ua = acc[t][1], ubb = 0.0f;
#pragma unroll
              for (int j = 0; j < 8; j += 2) {
                ga = fma2_bf16(gw[j], xw[j], ga);
                gb = fma2_bf16(gw[j + 1], xw[j + 1], gb);
                ua = fma2_bf16(uw[j], xw[j], ua);
                ubb = fma2_bf16(uw[j + 1], xw[j + 1], ubb);
              }
              acc[t][0] = ga + gb;
              acc[t][1] = ua + ubb;
            }
          }
        } else {
          const uint32_t gq[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          const uint32_t uq[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          uint32_t gh[16], uh[16];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            int8x4_to_f16x2x2(gq[j], gh[2 * j], gh[2 * j + 1]);
            int8x4_to_f16x2x2(uq[j], uh[2 * j], uh[2 * j + 1]);
          }
          const int kk = static_cast<int>(i - ub);
          const float sg = lds_f32(st + G::kWBytes + r * 16 + (kk & 3) * 4);
          const float su = lds_f32(st + G::kWBytes + 2048 + r * 16 + (kk & 3) * 4);
          const uint32_t tb = st + G::kTokOff + q * 64;
#pragma unroll
          for (int t = 0; t < kNE; ++t) {
            if (t < un.n) {
              float ga = 0.0f, gb = 0.0f, ua = 0.0f, ubb = 0.0f;
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const uint4 xv = lds128(tb + t * G::kSliceGU + h * 16);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                  ga = fma2_f16(gh[4 * h + j], xw[j], ga);
                  gb = fma2_f16(gh[4 * h + j + 1], xw[j + 1], gb);
                  ua = fma2_f16(uh[4 * h + j], xw[j], ua);
                  ubb = fma2_f16(uh[4 * h + j + 1], xw[j + 1], ubb);
                }
              }
              acc[t][0] = fmaf(ga + gb, sg, acc[t][0]);
              acc[t][1] = fmaf(ua + ubb, su, acc[t][1]);
            }
          }
        }
        release();
      }
      // the four quarters of a row hold partial sums over their quarter of every slice
#pragma unroll
      for (int t = 0; t < kNE; ++t)
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          acc[t][m] += __shfl_xor_sync(0xffffffffu, acc[t][m], 1);
          acc[t][m] += __shfl_xor_sync(0xffffffffu, acc[t][m], 2);
        }
      bool finish = true;
      if (!(ub >= g_beg && ue <= g_end)) finish = split_unit(acc, std::integral_constant<int, 2>{}, ub, ue, g_beg, Wg, NCg, KIg);
      if (finish) {
        const int i_row = un.rb * 128 + r;
        if constexpr (!kInt8) {
          if (q == 0) {
            __nv_bfloat16* h = static_cast<__nv_bfloat16*>(a.h);
#pragma unroll
            for (int t = 0; t < kNE; ++t)
              if (t < un.n)
                h[static_cast<int64_t>(un.p0 + t) * I + i_row] = __float2bfloat16_rn(silu_mul(acc[t][0], acc[t][1]));
          }
        } else {
          // h rounded to bf16, then its fp16 record: this unit's 128 rows are one scale group of the
          // down projection's reduction, so the group's largest |h| sets the record's power of two
          float hv[kNE];
#pragma unroll
          for (int t = 0; t < kNE; ++t) {
            float m = 0.0f;  // only quarter 0 holds the full sums after a split unit's hand-off
            if (t < un.n) {
              const float xsc = S.xs[S.sorted[un.p0 + t]];
              hv[t] = __bfloat162float(__float2bfloat16_rn(silu_mul(acc[t][0] * xsc, acc[t][1] * xsc)));
              if (q == 0) m = fabsf(hv[t]);
            } else {
              hv[t] = 0.0f;
            }
            m = warp_max_abs(m);
            if (lane == 0) S.red[red_buf][warp][t] = m;
          }
          named_bar_sync(2, kComputeThreads);
          if (q == 0) {
#pragma unroll
            for (int t = 0; t < kNE; ++t) {
              if (t < un.n) {
                float m = 0.0f;
#pragma unroll
                for (int w = 0; w < kComputeWarps; ++w) m = fmaxf(m, S.red[red_buf][w][t]);
                const int kh = f16_exponent(m);
                uint8_t* rec = static_cast<uint8_t*>(a.h) +
                               (static_cast<int64_t>(un.p0 + t) * (I / 128) + un.rb) * kRec;
                reinterpret_cast<__half*>(rec)[r] = __float2half_rn(hv[t] * ldexpf(1.0f, -kh));
                if (r == 0) *reinterpret_cast<float*>(rec + 256) = ldexpf(1.0f, kh);
              }
            }
          }
          red_buf ^= 1;
        }
      }
    }

    // ---- grid barrier: every CTA's h is written (this CTA's writes are ordered before the arrival)
    named_bar_sync(2, kComputeThreads);
    if (tid == 0) {
      S.gbar_epoch = grid_arrive(a.gbar, N + a.grid_extra);
      mbar_arrive(&S.gbar_arrived);
    }

    // ---------------------------- down ----------------------------
    for (int64_t i = d_beg; i < d_end;) {
      const int64_t u = i / KId;
      const int64_t ub = u * KId, ue = ub + KId;
      const int64_t pe = ue < d_end ? ue : d_end;
      const Unit un = dn_unit(u);
      float acc[kNE][1];
#pragma unroll
      for (int t = 0; t < kNE; ++t) acc[t][0] = 0.0f;
      const int box = q >> 1;  // quarters 0, 1 read the slot's first slice, 2, 3 its second
      for (; i < pe; ++i) {
        const uint32_t st = take();
        const uint32_t row = st + box * 16384 + r * 128;
        const int cb = 4 * (q & 1);
        const uint4 w0 = lds128(row + (((cb + 0) ^ x7) << 4)), w1 = lds128(row + (((cb + 1) ^ x7) << 4));
        const uint4 w2 = lds128(row + (((cb + 2) ^ x7) << 4)), w3 = lds128(row + (((cb + 3) ^ x7) << 4));
        const uint32_t wq[16] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w,
                                 w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
        if constexpr (!kInt8) {
          const uint32_t tb = st + G::kTokOff + q * 64;
#pragma unroll
          for (int t = 0; t < kNE; ++t) {
            if (t < un.n) {
              float ya = acc[t][0], yb = 0.0f;
#pragma unroll
              for (int hq = 0; hq < 4; ++hq) {
                const uint4 xv = lds128(tb + t * G::kSliceDN + hq * 16);
                ya = fma2_bf16(wq[4 * hq + 0], xv.x, ya);
                yb = fma2_bf16(wq[4 * hq + 1], xv.y, yb);
                ya = fma2_bf16(wq[4 * hq + 2], xv.z, ya);
                yb = fma2_bf16(wq[4 * hq + 3], xv.w, yb);
              }
              acc[t][0] = ya + yb;
            }
          }
        } else {
          uint32_t wh[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) int8x4_to_f16x2x2(wq[j], wh[2 * j], wh[2 * j + 1]);
          const int kk2 = static_cast<int>(i - ub);
          const float sd = lds_f32(st + G::kWBytes + r * 16 + ((2 * kk2 + box) & 3) * 4);
          const uint32_t tb = st + G::kTokOff + box * kRec;
#pragma unroll
          for (int t = 0; t < kNE; ++t) {
            if (t < un.n) {
              const uint32_t rec = tb + t * G::kSliceDN;
              float ya = 0.0f, yb = 0.0f;
#pragma unroll
              for (int hq = 0; hq < 8; ++hq) {
                const uint4 xv = lds128(rec + (q & 1) * 128 + hq * 16);
                ya = fma2_f16(wh[4 * hq + 0], xv.x, ya);
                yb = fma2_f16(wh[4 * hq + 1], xv.y, yb);
                ya = fma2_f16(wh[4 * hq + 2], xv.z, ya);
                yb = fma2_f16(wh[4 * hq + 3], xv.w, yb);
              }
              acc[t][0] = fmaf(ya + yb, sd * lds_f32(rec + 256), acc[t][0]);
            }
          }
        }
        release();
      }
#pragma unroll
      for (int t = 0; t < kNE; ++t) {
        acc[t][0] += __shfl_xor_sync(0xffffffffu, acc[t][0], 1);
        acc[t][0] += __shfl_xor_sync(0xffffffffu, acc[t][0], 2);
      }
      bool finish = true;
      if (!(ub >= d_beg && ue <= d_end)) finish = split_unit(acc, std::integral_constant<int, 1>{}, ub, ue, d_beg, Wd, NCd, KId);
      if (!finish) continue;
      const int h_row = un.rb * 128 + r;
      if (q == 0) {
#pragma unroll
        for (int t = 0; t < kNE; ++t)
          if (t < un.n) a.Y[static_cast<int64_t>(un.p0 + t) * H + h_row] = acc[t][0];
      }
      // this unit's Y rows are final: count it toward its row block, and let the row block's last
      // unit write the combine out[t, rows] = bf16(sum_j w[t, j] * Y[inv_pos[t, j], rows]) in slot order
      __threadfence();
      named_bar_sync(2, kComputeThreads);
      if (tid == 0) {
        __threadfence();
        const int old = atomicAdd(&a.ccount[un.rb], 1);
        const int last = old == NU - 1;
        if (last) a.ccount[un.rb] = 0;
        S.flag = last;
      }
      named_bar_sync(2, kComputeThreads);
      const bool last = S.flag != 0;
      named_bar_sync(2, kComputeThreads);
      if (last) {
        __threadfence();
        for (int idx = tid; idx < T * 128; idx += kComputeThreads) {
          const int t = idx >> 7;
          const int row = un.rb * 128 + (idx & 127);
          float acc2 = 0.0f;
          for (int j = 0; j < k; ++j) {
            const float y = __ldcg(a.Y + static_cast<int64_t>(S.inv[t * k + j]) * H + row);
            acc2 = __fadd_rn(acc2, __fmul_rn(S.w[t * k + j], y));
          }
          a.out[static_cast<int64_t>(t) * H + row] = __bfloat16_as_ushort(__float2bfloat16_rn(acc2));
        }
      }
    }
  }
  __syncthreads();
}

template <bool kInt8>
cudaError_t prepare(int* max_ctas) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDev) {
    const int c = cache[dev].load(std::memory_order_acquire);
    if (c > 0) {
      *max_ctas = c;
      return cudaSuccess;
    }
  }
  e = cudaFuncSetAttribute(decode_step_kernel<kInt8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem_bytes<kInt8>());
  if (e != cudaSuccess) return e;
  int per_sm = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_step_kernel<kInt8>, kThreads,
                                                    smem_bytes<kInt8>());
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorNotSupported;
  const int n = sms;  // one CTA per SM
  if (dev < kMaxDev) cache[dev].store(n, std::memory_order_release);
  *max_ctas = n;
  return cudaSuccess;
}

// Scale tensor map {groups (contiguous), rows, E} fp32, box = 4 groups x 128 rows.
bool encode_scales(CUtensorMap* map, const float* s, int groups, int rows, int E) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(groups), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(E)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(groups) * 4, static_cast<cuuint64_t>(groups) * rows * 4};
  cuuint32_t box[3] = {4, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return tensor_map_encoder()(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(s), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kInt8>
cudaError_t launch(const DecodePlan& p, cudaStream_t stream) {
  CUtensorMap tg, tu, td, tsg, tsu, tsd;
  if (!tensor_map_encoder()) return cudaErrorNotSupported;
  if (!encode_weights(&tg, p.W_gate, kInt8, p.H, p.I, p.E, 128) ||
      !encode_weights(&tu, p.W_up, kInt8, p.H, p.I, p.E, 128) ||
      !encode_weights(&td, p.W_down, kInt8, p.I, p.H, p.E, 128))
    return cudaErrorInvalidValue;
  tsg = tg;
  tsu = tu;
  tsd = td;
  if (kInt8 && (!encode_scales(&tsg, p.s_gate, p.H / 128, p.I, p.E) ||
                !encode_scales(&tsu, p.s_up, p.H / 128, p.I, p.E) ||
                !encode_scales(&tsd, p.s_down, p.I / 128, p.H, p.E)))
    return cudaErrorInvalidValue;
  int max_ctas = 0;
  cudaError_t e = prepare<kInt8>(&max_ctas);
  if (e != cudaSuccess) return e;
  const int ctas = max_ctas < p.max_ctas ? max_ctas : p.max_ctas;
  // cooperative (all CTAs resident: the grid barrier waits on every CTA) and, where the driver
  // accepts the combination, with programmatic dependent launch (the next launch's start-up overlaps
  // this one's tail; every CTA waits for the predecessor before reading its inputs)
  static std::atomic<int> pdl_ok{1};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes<kInt8>();
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_ok.load(std::memory_order_relaxed) ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, decode_step_kernel<kInt8>, tg, tu, td, tsg, tsu, tsd, p.args);
  if (e != cudaSuccess && cfg.numAttrs == 2) {
    cudaGetLastError();  // clear the launch error, then launch cooperatively alone
    pdl_ok.store(0, std::memory_order_relaxed);
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_step_kernel<kInt8>, tg, tu, td, tsg, tsu, tsd, p.args);
  }
  return e;
}

}  // namespace dec

bool decode_step_supported(int T, int H, int I, int E, int k, bool int8) {
  if (T < 1 || T > kDecodeMaxT || static_cast<int64_t>(T) * k > kDecodeMaxP || E > 256) return false;
  if (H % 128 || I % 128) return false;
  if (int8 && (H % 512 || I % 512)) return false;  // scale boxes of 4 groups; two groups per down slot
  return true;
}

cudaError_t launch_decode_step(const DecodePlan& plan, cudaStream_t stream) {
  return plan.int8 ? dec::launch<true>(plan, stream) : dec::launch<false>(plan, stream);
}

}  // namespace moe
