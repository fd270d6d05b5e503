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
//      is finished by its head, the CTA holding its first tiles, which adds the later pieces'
//      partial sums in CTA order (stored with a tag, gathered while it works on its own part);
//   3. one grid-wide barrier (h complete): while waiting, the producer already streams the CTA's
//      first down-projection weight tiles, which do not depend on h;
//   4. down, cut the same way, row-block-major; the CTA that completes the last unit of a 128-row
//      block of the output writes that block's combine (fixed slot order, no atomics on data).
// Per CTA (one per SM; a cooperative launch, so all CTAs are resident for the barrier):
//   warps 0..15  compute: thread = (weight row r of the tile, quarter q of its 128-byte slice);
//                BF16: mixed-precision FMAs (fma.rn.f32.bf16: exact products, fp32 sums), INT8:
//                dp4a against the token records, reading the weights straight from the TMA-filled
//                tile and the tokens from the slot (INT8 at one token: from shared memory);
//   warp 16      producer: TMA tensor loads of the weight tiles (and INT8 scale boxes), bulk
//                copies of the tokens' slices (x for gate+up, h for down) into the same slot;
//   warp 17      helper: the hand-offs that wait on global memory (gathering a head's later
//                pieces, counting finished down units, the grid barrier's arrival), posted to it by
//                the compute warps through a small ring in shared memory.
// INT8: the int8 weights enter dp4a as they are; the tokens (x, and h between the phases) are held
// as records of 24-bit fixed point per 128-element group (three int8 digit planes and a power-of-two
// scale), so each group's dot product is exact in int32, then scaled in fp32 by the weight group's
// and the record's scales.
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

// Tokens per pass of an expert: a template parameter of the kernel (1, 4 or 8, chosen per launch);
// the slots and shared arrays are sized for the largest.
constexpr int kMaxNEAll = 8;
constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = 32 * kComputeWarps;  // 128 rows x 4 quarters
constexpr int kProducerWarp = kComputeWarps;
constexpr int kHelperWarp = kComputeWarps + 1;
constexpr int kThreads = kComputeThreads + 64;
constexpr int kBar1Threads = kComputeThreads + 32;  // barrier 1: the compute warps and the producer
// Hand-off ring between the compute warps and the helper warp: the compute warps post a finished
// unit piece (or a phase end) and go on; the helper does the part that waits on global memory.
constexpr int kItems = 8;
enum : int {
  kItemGuHead = 0,   // the head piece begins: gather the unit's later pieces (sum in CTA order) meanwhile
  kItemDnHead = 1,
  kItemDnWhole = 2,  // a down unit's Y rows are final: count it toward its row block
  kItemGuEnd = 3,    // gate+up done: arrive at the grid barrier
  kItemEnd = 4,
};
constexpr int kMaxOwed = 128;  // row blocks of the output (H <= 16384)
// INT8 token record of one 128-element group (x for gate+up, h for down): the group's values as 24-bit
// fixed-point integers X = round(v * 2^-e), e chosen so that the group's largest |v| * 2^-e lies in
// [2^22, 2^23), split into three int8 digit planes of 128 bytes (X = d2 * 2^16 + d1 * 2^8 + d0, d0 and d1
// unsigned, d2 signed), then the fp32 2^e and padding to 16 bytes.
constexpr int kRec = 400;
constexpr int kRecScale = 384;

template <bool kInt8>
struct Geo {
  static constexpr int kMaxNE = kInt8 ? 4 : 8;          // tokens per pass at most
  static constexpr int kKt = kInt8 ? 128 : 64;          // reduction elements per 128-byte tile row
  static constexpr int kWBytes = 32768;                 // two 128-row x 128-byte weight boxes
  static constexpr int kScaleBytes = kInt8 ? 4096 : 0;  // INT8: two {4 groups x 128 rows} fp32 boxes
  static constexpr int kSliceGU = kInt8 ? kRec : 128;   // token bytes per slot, gate+up (x)
  static constexpr int kSliceDN = kInt8 ? 2 * kRec : 256;  // and down (h: two reduction slices)
  static constexpr int kSliceMax = kSliceGU > kSliceDN ? kSliceGU : kSliceDN;
  static constexpr int kTokOff = kWBytes + kScaleBytes;
  static constexpr int kSlot = (kTokOff + kMaxNE * kSliceMax + 1023) / 1024 * 1024;
  static constexpr int kStages = kInt8 ? 5 : 6;
  static_assert(kSlot % 1024 == 0, "slots keep the 1024-byte alignment of the 128B swizzle");
};

struct Shared {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t gbar_arrived;  // helper -> producer: this CTA has arrived at the grid barrier
  uint64_t item_full[kItems];   // compute -> helper: an item is posted
  uint64_t item_empty[kItems];  // helper -> compute: the item's entry may be reused
  uint64_t helper_done;         // helper -> compute: every item is handled
  uint64_t pre_ready;           // helper -> compute: the head's later pieces are summed in `pre`
  struct Item {
    int ub, ue;  // split pieces: the unit's tile range
    int kind, p0, n, rb;
  } items[kItems];
  int owed[kMaxOwed];     // complete row blocks, posted by the helper: the compute warps write their combine
  int owed_n;
  int gbar_epoch;         // the barrier's release word as read before arriving
  uint32_t tag_base;      // twice the release word at entry: partial sums carry tag_base + 1 (gate+up), + 2 (down)
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
  int qc[kDecodeMaxP];    // cost of one tile of pass q (tile_cost of its tokens)
  int pc[kDecodeMaxP + 1];  // prefix sums of qc
  float red[2][kComputeWarps][kMaxNEAll];
  int bounds[4];          // this CTA's gate+up and down tile ranges
};

// INT8 at one token (kNE = 1): the token's records stay in shared memory for the whole step (written
// once by the compute warps, H / 128 records of kRec bytes after Shared), so a gate+up slot carries
// only weights and scales and its copies need not wait for the records; the ring has four slots to
// make room. Measured on GB300, the first gate+up slot landed ~9 us after routing when its token
// slice had to be written to global memory and copied back.
//
// Every unit split between CTAs is finished by its head, the CTA that holds its first tiles (at the
// end of that CTA's range); its later pieces (at the start of later CTAs' ranges, or a later CTA's
// whole range) publish their partial sums as tagged 64-bit stores, and the head's helper gathers them into
// `pre` (kNE x 2 x 128 fp32, after Shared) while the head's compute warps work on their part. BF16
// passes of eight tokens keep five slots to make room for it.
//
// A slot holds the pass's kNE token slices at most. INT8 at one token with the records of a row of
// up to kDeepMaxH elements (kDeep) keeps five slots: a fifth slot of weights streams in while the CTA
// waits at the grid barrier.
constexpr int kDeepMaxH = 8448;
template <bool kInt8, int kNE, bool kDeep = false>
struct GeoN : Geo<kInt8> {
  static constexpr bool kRecSmem = kInt8 && kNE == 1;
  static constexpr int kSlot = (Geo<kInt8>::kTokOff + kNE * Geo<kInt8>::kSliceMax + 1023) / 1024 * 1024;
  static constexpr int kStages = kRecSmem ? (kDeep ? 5 : 4) : (!kInt8 && kNE == 8 ? 5 : Geo<kInt8>::kStages);
  static constexpr int kPreBytes = kNE * 2 * 128 * 4;
  static_assert(kSlot % 1024 == 0 && kStages <= 8, "slots keep the 1024-byte alignment; eight mbarriers");
};

constexpr int kSharedBytes = (static_cast<int>(sizeof(Shared)) + 15) / 16 * 16;
template <bool kInt8, int kNE, bool kDeep>
constexpr int smem_bytes(int H) {
  using G = GeoN<kInt8, kNE, kDeep>;
  return G::kStages * G::kSlot + kSharedBytes + G::kPreBytes + (G::kRecSmem ? (H / 128) * kRec : 0);
}
static_assert(smem_bytes<false, 8, false>(0) <= 232448 && smem_bytes<false, 4, false>(0) <= 232448 &&
                  smem_bytes<false, 1, false>(0) <= 232448 && smem_bytes<true, 4, false>(0) <= 232448 &&
                  smem_bytes<true, 1, false>(16384) <= 232448 && smem_bytes<true, 1, true>(kDeepMaxH) <= 232448,
              "dynamic shared memory per CTA");

// Stream-K by cost: a tile of a pass with n tokens costs max(kCostMem, kCostBase + kCostTok * n), its
// HBM time or its compute warps' time, whichever is longer (the compute grows with the tokens: on GB300
// a BF16 tile is bound by HBM up to about two tokens, an INT8 tile up to about one), so CTAs whose
// tiles carry more tokens get fewer tiles.
constexpr int kCostMem = 10;
constexpr int kCostBase = 4;
template <bool kInt8>
__host__ __device__ constexpr int tile_cost(int n) {
  return kCostBase + (kInt8 ? 5 : 3) * n > kCostMem ? kCostBase + (kInt8 ? 5 : 3) * n : kCostMem;
}

// One unit: pass `np` of the a-th active expert (tokens at sorted positions p0 .. p0 + n - 1) and a
// 128-row block of the output rows.
struct Unit {
  int e, p0, n, rb;
};

template <int kNE>
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

// floor(c * C / N) in 32-bit arithmetic, for 0 <= C < 2^31 and 0 <= c <= N < 2^15 (c * C itself
// may not fit).
__device__ __forceinline__ int scaled(int c, int C, int N) {
  const int q = C / N, r = C - q * N;
  return c * q + (c * r) / N;
}

// The CTA that holds cost position pos when C is cut into N ranges [scaled(c), scaled(c + 1)): the
// last c with scaled(c) <= pos (an fp32 estimate, then exact steps).
__device__ __forceinline__ int cta_at(int pos, int C, int N) {
  int c = static_cast<int>(static_cast<float>(pos) * static_cast<float>(N) / static_cast<float>(C));
  c = c < 0 ? 0 : (c > N - 1 ? N - 1 : c);
  while (c + 1 < N && scaled(c + 1, C, N) <= pos) ++c;
  while (c > 0 && scaled(c, C, N) > pos) --c;
  return c;
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

// e with max * 2^-e in [2^22, 2^23) (the 24-bit fixed point of an INT8 token record), kept where 2^e
// and the conversions stay finite in fp32; 0 for an all-zero or non-finite group.
__device__ __forceinline__ int fixed_exponent(float m) {
  int k = 0;
  if (m > 0.0f && m <= 3.0e38f) {
    int e = 0;
    frexpf(m, &e);  // m = f * 2^e, 0.5 <= f < 1
    k = e - 23;
    k = k < -140 ? -140 : k;
  }
  return k;
}

// The three digit bytes of round(v * 2^-e) (|.| < 2^23): d0 = bits 0..7, d1 = bits 8..15 (unsigned),
// d2 = bits 16..23 with the sign (an arithmetic shift).
__device__ __forceinline__ int fixed_value(float v, int e) { return __float2int_rn(ldexpf(v, -e)); }

// dp4a of four unsigned digit bytes (a) with four signed weights (b), or of signed bytes with signed.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Sum over one 16-byte chunk pair of a token record's planes: sum_k X_k * q_k for the 32 elements whose
// weights are in w[0..7] (chunk ca, then chunk cb) and whose digits are at chunk offsets ca and cb of
// the record at `rec` (a shared-memory address). Exact in int32 per plane; returned as fp32.
__device__ __forceinline__ float record_dot(uint32_t rec, int ca, int cb, const uint32_t (&w)[8]) {
  int s[3];
#pragma unroll
  for (int p = 0; p < 3; ++p) {
    const uint4 xa = lds128(rec + p * 128 + ca * 16), xb = lds128(rec + p * 128 + cb * 16);
    const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    int acc = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc = p == 2 ? dp4a_ss(xw[j], w[j], acc) : dp4a_us(xw[j], w[j], acc);
    s[p] = acc;
  }
  return fmaf(static_cast<float>(s[2]), 65536.0f, fmaf(static_cast<float>(s[1]), 256.0f, static_cast<float>(s[0])));
}

template <bool kInt8, int kNE, bool kDeep>
__global__ void __launch_bounds__(kThreads, 1)
    decode_step_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmU,
                       const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmSG,
                       const __grid_constant__ CUtensorMap tmSU, const __grid_constant__ CUtensorMap tmSD,
                       const DecodeArgs a) {
  using G = GeoN<kInt8, kNE, kDeep>;
  extern __shared__ __align__(1024) uint8_t smem[];
  Shared& S = *reinterpret_cast<Shared*>(smem + G::kStages * G::kSlot);
  float* const pre = reinterpret_cast<float*>(smem + G::kStages * G::kSlot + kSharedBytes);  // the head's later pieces
  uint8_t* const rec_smem = smem + G::kStages * G::kSlot + kSharedBytes + G::kPreBytes;  // kRecSmem: the token's records
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
    for (int i = 0; i < kItems; ++i) {
      mbar_init(&S.item_full[i], 1);
      mbar_init(&S.item_empty[i], 1);
    }
    mbar_init(&S.helper_done, 1);
    mbar_init(&S.pre_ready, 1);
    S.owed_n = 0;
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
  prefetch_l2_grid(a.x, static_cast<int64_t>(T) * H * 2);  // the token rows, spread over the grid
  for (int i = tid; i < 256; i += kThreads) {
    S.cnt[i] = 0;
    S.tokmask[i] = 0u;
  }
  pdl_wait_predecessor();
  pdl_allow_successor();
  // the status word starts each call at 0 (a wait gives up only after kWaitLimitNs, long after every
  // CTA of this cooperative launch has passed this point)
  if (cta == 0 && tid == 0) *a.status = 0;
  // the launch's tags: the release word advances once per launch, at the grid barrier, which no CTA
  // passes before every CTA has read it here (the predecessor's advance is visible after the wait)
  if (tid == 0) S.tag_base = 2u * static_cast<uint32_t>(ld_relaxed_gpu(a.gbar + 1));
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
  if (warp == 0) {  // exclusive offsets, active list and the prefix of pass counts, 32 experts at a time
    int run = 0, nact = 0, prun = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int c = e < E ? S.cnt[e] : 0;
      const int pc = (c + kNE - 1) / kNE;
      int incl = c, pin = pc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        const int m = __shfl_up_sync(0xffffffffu, pin, o);
        if (lane >= o) {
          incl += n;
          pin += m;
        }
      }
      const uint32_t act = __ballot_sync(0xffffffffu, c > 0);
      if (e < E) {
        S.off[e] = run + incl - c;
        if (c > 0) {
          const int ai = nact + __popc(act & ((1u << lane) - 1u));
          S.act_e[ai] = e;
          S.pp[ai + 1] = prun + pin;
        }
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      prun += __shfl_sync(0xffffffffu, pin, 31);
      nact += __popc(act);
    }
    if (lane == 0) {
      S.off[E] = run;
      S.A = nact;
      S.pp[0] = 0;
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
  for (int q = tid; q < NU; q += kThreads) S.qc[q] = tile_cost<kInt8>(unit_of<kNE>(S, q, 0).n);
  __syncthreads();
  if (warp == 0) {  // exclusive prefix of the pass costs, eight passes per lane
    int v[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = lane * 8 + j;
      v[j] = q < NU ? S.qc[q] : 0;
      sum += v[j];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int run = incl - sum;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = lane * 8 + j;
      if (q <= NU) S.pc[q] = run;
      run += v[j];
    }
  }
  __syncthreads();
  const int RBg = I / 128, KIg = H / G::kKt;        // gate+up: rows of I, reduction H
  const int RBd = H / 128, KId = I / (2 * G::kKt);  // down: rows of H, reduction I (two slices per slot)
  // Tile indices and cost positions stay below 2^31 (NU <= 256 passes, H <= 16384, I <= 32768, a tile
  // costs at most 28), so the schedule is 32-bit arithmetic; the one product that does not fit,
  // c * C / N, is split (scaled). A 64-bit division is a long dependent chain: a dozen of them on one
  // thread held the producer's first copy back by ~3 us (measured on GB300 at one token).
  const int TPg = RBg * KIg;  // gate+up tiles of one pass
  const int Wg = NU * TPg;
  const int Wd = NU * RBd * KId;
  const int PC = S.pc[NU];
  const int Cg = PC * TPg, Rd = PC * KId, Cd = Rd * RBd;  // total costs; Rd: one row block of down
  // CTAs taking part: each range is at least one tile's cost wide, so every one holds a tile
  constexpr int kMaxCost = tile_cost<kInt8>(kNE);
  const int Ng = Cg / kMaxCost < N ? (Cg / kMaxCost > 0 ? Cg / kMaxCost : 1) : N;
  const int Nd = Cd / kMaxCost < N ? (Cd / kMaxCost > 0 ? Cd / kMaxCost : 1) : N;
  auto pass_at = [&](int X) -> int {  // the last pass q with pc[q] <= X
    int lo = 0, hi = NU - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (S.pc[mid] <= X) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  // cost position of a tile, and the first tile at or past a cost position (gate+up: tiles of pass
  // q at q * TPg .., each costing qc[q]; down: row block rb, then pass q, KId tiles each)
  auto pos_gu = [&](int i) -> int {
    const int q = i / TPg;
    return S.pc[q] * TPg + (i - q * TPg) * S.qc[q];
  };
  auto first_gu = [&](int X) -> int {
    if (X >= Cg) return Wg;
    const int q = pass_at(X / TPg);
    return q * TPg + (X - S.pc[q] * TPg + S.qc[q] - 1) / S.qc[q];
  };
  auto pos_dn = [&](int i) -> int {
    const int u = i / KId, rb = u / NU, q = u - rb * NU;
    return rb * Rd + S.pc[q] * KId + (i - u * KId) * S.qc[q];
  };
  auto first_dn = [&](int X) -> int {
    if (X >= Cd) return Wd;
    const int rb = X / Rd, rem = X - rb * Rd;
    const int q = pass_at(rem / KId);
    return (rb * NU + q) * KId + (rem - S.pc[q] * KId + S.qc[q] - 1) / S.qc[q];
  };
  // The CTA's tile ranges, [first(scaled(cta)), first(scaled(cta + 1))) per phase, one bound per thread
  if (tid < 4) {
    const bool dn = tid >= 2;
    const int Nx = dn ? Nd : Ng, Cx = dn ? Cd : Cg, Wx = dn ? Wd : Wg;
    const int X = scaled(cta + (tid & 1), Cx, Nx);
    S.bounds[tid] = cta < Nx ? (dn ? first_dn(X) : first_gu(X)) : Wx;
  }
  __syncthreads();
  const int g_beg = S.bounds[0], g_end = S.bounds[1];
  const int d_beg = S.bounds[2], d_end = S.bounds[3];
  // gate+up units are pass-major (q * RBg + rb): a CTA's range touches few experts' tokens;
  // down units are row-block-major (rb * NU + q): a row block's combine becomes ready as soon as
  // its last unit is done, spread over the step instead of all at its end.
  auto gu_unit = [&](int u) { return unit_of<kNE>(S, u / RBg, u % RBg); };
  auto dn_unit = [&](int u) { return unit_of<kNE>(S, u % NU, u / NU); };

  // INT8: records (the digit planes above) of the token rows this CTA's gate+up tiles read, one per
  // 128-element scale group, the same layout as h's. CTAs that share a token write the same bytes;
  // each CTA reads only records it has written itself.
  if (kInt8) {
    uint32_t need = 0u;
    if constexpr (G::kRecSmem) {
      need = g_beg < g_end ? 1u : 0u;  // the one token, if this CTA has gate+up tiles (the producer need not wait)
    } else {
      if (tid == 0) {
        if (g_beg < g_end) {
          const int q0 = (g_beg / KIg) / RBg, q1 = ((g_end - 1) / KIg) / RBg;
          const Unit u0 = unit_of<kNE>(S, q0, 0), u1 = unit_of<kNE>(S, q1, 0);
          for (int p = u0.p0; p < u1.p0 + u1.n; ++p) need |= 1u << S.sorted[p];
        }
        S.need = need;
      }
      __syncthreads();
      need = S.need;
    }
    if (warp < kComputeWarps) {
      const int ng = H / 128;
      const int nrec = __popc(need) * ng;
      for (int w = warp; w < nrec; w += kComputeWarps) {  // a warp per (token, group) record
        const int j = w / ng, g = w - j * ng;
        uint32_t m = need;
        for (int z = 0; z < j; ++z) m &= m - 1u;
        const int t = __ffs(m) - 1;
        const uint2 v = *reinterpret_cast<const uint2*>(a.x + static_cast<int64_t>(t) * H + g * 128 + lane * 4);
        const float f0 = __uint_as_float(v.x << 16), f1 = __uint_as_float(v.x & 0xffff0000u);
        const float f2 = __uint_as_float(v.y << 16), f3 = __uint_as_float(v.y & 0xffff0000u);
        const float mx = warp_max_abs(fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3))));
        const int kx = fixed_exponent(mx);
        const int X0 = fixed_value(f0, kx), X1 = fixed_value(f1, kx), X2 = fixed_value(f2, kx), X3 = fixed_value(f3, kx);
        uint8_t* rec = G::kRecSmem ? rec_smem + g * kRec  // one token (T = 1)
                                   : reinterpret_cast<uint8_t*>(a.x16) + (static_cast<int64_t>(t) * ng + g) * kRec;
        // plane p, elements 4 lane .. 4 lane + 3: bytes of (X >> 8 p)
#pragma unroll
        for (int p = 0; p < 3; ++p) {
          const uint32_t word = ((X0 >> (8 * p)) & 0xff) | (((X1 >> (8 * p)) & 0xff) << 8) |
                                (((X2 >> (8 * p)) & 0xff) << 16) | (static_cast<uint32_t>((X3 >> (8 * p)) & 0xff) << 24);
          *reinterpret_cast<uint32_t*>(rec + p * 128 + lane * 4) = word;
        }
        if (lane == 0) *reinterpret_cast<float*>(rec + kRecScale) = ldexpf(1.0f, kx);
      }
      if constexpr (G::kRecSmem) {
        named_bar_sync(3, kComputeThreads);  // the compute warps read the records from shared memory
      } else {
        fence_proxy_async_global();  // the producer's bulk copies of these records come after the barrier
        named_bar_sync(1, kBar1Threads);
      }
    }
  }

  if (warp == kProducerWarp) {
    // ================================ producer ================================
    // Lane 0 issues everything; the warp's other lanes only take part in barrier 1 (INT8).
    {
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
      // The tiles are stepped through with cursors: one division and one unit lookup per range (and a
      // lookup per unit), none per tile. The single issuing thread shares the SM's issue slots with
      // sixteen compute warps, and per-tile arithmetic on its path held back every copy behind it.
      // ---- gate+up tiles (pass-major units q * RBg + rb, KIg reduction slices each)
      // The first ring's weight tiles go out at once; their token slices follow when the token rows
      // are ready (INT8: the compute warps' fp16 copies, signalled by barrier 1).
      struct GuCursor {
        int kk, q, rb;
        Unit un;
      };
      GuCursor cur{};
      // token t's row: bf16 x, or its INT8 records (H / 128 of kRec bytes)
      const uint8_t* xrow[kNE];
      const int64_t xrow_bytes = kInt8 ? static_cast<int64_t>(H / 128) * kRec : static_cast<int64_t>(H) * 2;
      const uint8_t* const xbase = kInt8 ? reinterpret_cast<const uint8_t*>(a.x16) : reinterpret_cast<const uint8_t*>(a.x);
      auto rows_of = [&](const Unit& un) {
#pragma unroll
        for (int t = 0; t < kNE; ++t) xrow[t] = xbase + S.sorted[un.p0 + (t < un.n ? t : 0)] * xrow_bytes;
      };
      auto step = [&](GuCursor& c, int i) {  // to tile i + 1
        if (++c.kk == KIg) {
          c.kk = 0;
          if (++c.rb == RBg) {
            c.rb = 0;
            ++c.q;
          }
          if (i + 1 < g_end) c.un = unit_of<kNE>(S, c.q, c.rb);
        }
      };
      auto weights_gu = [&](int sl, const GuCursor& c) {
        uint8_t* st = slots + sl * G::kSlot;
        mbar_arrive_expect_tx(&S.full[sl], G::kWBytes + G::kScaleBytes + (G::kRecSmem ? 0 : c.un.n * G::kSliceGU));
        tma_load_3d(st, &tmG, &S.full[sl], c.kk * G::kKt, c.un.rb * 128, c.un.e, pol);
        tma_load_3d(st + 16384, &tmU, &S.full[sl], c.kk * G::kKt, c.un.rb * 128, c.un.e, pol);
        if (kInt8) {
          tma_load_3d_plain(st + G::kWBytes, &tmSG, &S.full[sl], c.kk & ~3, c.un.rb * 128, c.un.e);
          tma_load_3d_plain(st + G::kWBytes + 2048, &tmSU, &S.full[sl], c.kk & ~3, c.un.rb * 128, c.un.e);
        }
      };
      auto tokens_gu = [&](int sl, const GuCursor& c) {
        if constexpr (G::kRecSmem) return;  // the records are in shared memory already
        uint8_t* st = slots + sl * G::kSlot;
#pragma unroll
        for (int t = 0; t < kNE; ++t)
          if (t < c.un.n)
            bulk_g2s(st + G::kTokOff + t * G::kSliceGU, xrow[t] + c.kk * G::kSliceGU, G::kSliceGU, &S.full[sl]);
      };
      const int npre = (g_end - g_beg) < G::kStages ? (g_end - g_beg) : G::kStages;
      if (g_beg < g_end) {
        const int u0 = g_beg / KIg;
        cur.kk = g_beg - u0 * KIg;
        cur.q = u0 / RBg;
        cur.rb = u0 - cur.q * RBg;
        cur.un = unit_of<kNE>(S, cur.q, cur.rb);
      }
      const GuCursor first = cur;
      if (lane == 0) {
        rows_of(cur.un);
        for (int j = 0; j < npre; ++j) {  // a fresh ring: no slot to wait for
          weights_gu(static_cast<int>(j), cur);
          if (!kInt8) tokens_gu(static_cast<int>(j), cur);  // BF16 reads x itself: each slot whole, in order
          const int q0 = cur.q, rb0 = cur.rb;
          step(cur, g_beg + j);
          if (!kInt8 && (cur.q != q0 || cur.rb != rb0)) rows_of(cur.un);
        }
      }
      __syncwarp();
      if (kInt8 && !G::kRecSmem) named_bar_sync(1, kBar1Threads);
      if (lane == 0) {
      if (kInt8 && !G::kRecSmem) {  // the records are written: the first ring's token slices
        GuCursor c = first;
        rows_of(c.un);
        for (int j = 0; j < npre; ++j) {
          tokens_gu(static_cast<int>(j), c);
          const int q0 = c.q, rb0 = c.rb;
          step(c, g_beg + j);
          if (c.q != q0 || c.rb != rb0) rows_of(c.un);
        }
        rows_of(cur.un);
      }
      for (int j = 0; j < npre; ++j) advance();
      for (int i = g_beg + npre; i < g_end && ok; ++i) {
        if (!mbar_wait(&S.empty[slot], ph ^ 1u)) {
          ok = false;
          atomicExch(a.status, kStatusWaitEmptyTimeout);
          break;
        }
        weights_gu(slot, cur);
        tokens_gu(slot, cur);
        advance();
        const int q0 = cur.q, rb0 = cur.rb;
        step(cur, i);
        if (cur.q != q0 || cur.rb != rb0) rows_of(cur.un);
      }
      // ---- down tiles (row-block-major units rb * NU + q, KId slots of two reduction slices each):
      // weights as slots free up; the h slices of a slot once the grid barrier is passed
      int pend_slot[8];
      int pend_kk2[8];
      const uint8_t* pend_src[8];
      int pend_n[8];
      int npend = 0;
      bool passed = false;
      auto issue_h = [&](int sl, const uint8_t* src, int n, int kk2) {
        uint8_t* st = slots + sl * G::kSlot;
        // h rows of the unit's tokens are consecutive (sorted positions p0 ..): I * 2 bytes apart in
        // bf16, I / 128 records apart for INT8
        const int64_t row_bytes = kInt8 ? static_cast<int64_t>(I / 128) * kRec : static_cast<int64_t>(I) * 2;
        const int64_t off = kInt8 ? static_cast<int64_t>(2 * kk2) * kRec : static_cast<int64_t>(kk2) * 256;
        for (int t = 0; t < n; ++t)
          bulk_g2s(st + G::kTokOff + t * G::kSliceDN, src + t * row_bytes + off, G::kSliceDN, &S.full[sl]);
      };
      // the grid barrier has been passed: every CTA's h is written (acquire, then order the async
      // proxy's later reads after it)
      auto barrier_ready = [&]() -> bool {
        if (!mbar_try_wait_short(&S.gbar_arrived, 0)) return false;
        return ld_acquire_gpu(a.gbar + 1) != *reinterpret_cast<volatile int*>(&S.gbar_epoch);
      };
      auto release_pending = [&]() {
        fence_proxy_async_global();
        passed = true;
        for (int j = 0; j < npend; ++j) issue_h(pend_slot[j], pend_src[j], pend_n[j], pend_kk2[j]);
        npend = 0;
      };
      // wait for a free slot, issuing the pending h slices as soon as the barrier opens (the slots
      // they complete are the ones the compute warps wait for)
      auto wait_slot = [&]() -> bool {
        if (mbar_try_wait(&S.empty[slot], ph ^ 1u)) return true;
        const uint64_t t0 = global_timer_ns();
        uint64_t tb = t0;
        for (;;) {
          // while h slices wait for the grid barrier, poll both with short tries (the barrier opening is
          // what the compute warps wait for; measured ~2.3 us from the last arrival to the release)
          const bool polling = !passed && npend > 0;
          if (polling ? mbar_try_wait_short(&S.empty[slot], ph ^ 1u) : mbar_try_wait(&S.empty[slot], ph ^ 1u))
            return true;
          if (polling) {
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
      if (d_beg < d_end && ok) {
        const int u0 = d_beg / KId;
        int kk2 = d_beg - u0 * KId;
        int rb = u0 / NU, q = u0 - rb * NU;
        Unit un = unit_of<kNE>(S, q, rb);
        auto h_of = [&]() -> const uint8_t* {
          return kInt8 ? static_cast<const uint8_t*>(a.h) + static_cast<int64_t>(un.p0) * (I / 128) * kRec
                       : static_cast<const uint8_t*>(a.h) + static_cast<int64_t>(un.p0) * I * 2;
        };
        const uint8_t* hsrc = h_of();
        for (int i = d_beg; i < d_end; ++i) {
          if (!wait_slot()) {
            ok = false;
            atomicExch(a.status, kStatusWaitEmptyTimeout);
            break;
          }
          uint8_t* st = slots + slot * G::kSlot;
          mbar_arrive_expect_tx(&S.full[slot], G::kWBytes + (kInt8 ? 2048 : 0) + un.n * G::kSliceDN);
          tma_load_3d(st, &tmD, &S.full[slot], 2 * kk2 * G::kKt, un.rb * 128, un.e, pol);
          tma_load_3d(st + 16384, &tmD, &S.full[slot], (2 * kk2 + 1) * G::kKt, un.rb * 128, un.e, pol);
          if (kInt8) tma_load_3d_plain(st + G::kWBytes, &tmSD, &S.full[slot], (2 * kk2) & ~3, un.rb * 128, un.e);
          if (passed) {
            issue_h(slot, hsrc, un.n, kk2);
          } else {
            pend_slot[npend] = slot;
            pend_src[npend] = hsrc;
            pend_n[npend] = un.n;
            pend_kk2[npend] = kk2;
            ++npend;
          }
          advance();
          if (++kk2 == KId) {
            kk2 = 0;
            if (++q == NU) {
              q = 0;
              ++rb;
            }
            if (i + 1 < d_end) {
              un = unit_of<kNE>(S, q, rb);
              hsrc = h_of();
            }
          }
        }
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
      }  // lane 0
    }
    __syncwarp();
  } else if (warp == kHelperWarp) {
    // ================================ helper ================================
    // The part of a unit's end that waits on global memory, in the order the compute warps post it:
    // a head piece's start makes the helper gather the unit's later pieces, in CTA order, into `pre`
    // (the later pieces publish themselves, as tagged partial sums);
    // a finished down unit is counted toward its row block, and the row block's last unit posts the
    // block's combine to the compute warps; the gate+up phase's end is the arrival at the grid
    // barrier. Each round trip takes microseconds while HBM streams at full rate (measured on GB300,
    // ~2.7 us per hand-off), time the compute warps now spend on their next tiles.
    int it = 0;
    uint32_t iph = 0;
    int owed_n = 0;
    // count a finished down unit toward row block rb; the last one posts the row block's combine
    auto count_dn = [&](int rb) {
      __syncwarp();  // the lanes' Y stores before lane 0's release
      if (lane == 0) {
        __threadfence();
        const int old = atomicAdd(&a.ccount[rb], 1);
        if (old == NU - 1) {
          a.ccount[rb] = 0;
          __threadfence();  // acquire: every unit's Y of the row block
          if (owed_n < kMaxOwed) {
            S.owed[owed_n] = rb;
            __threadfence_block();
            *reinterpret_cast<volatile int*>(&S.owed_n) = ++owed_n;
          }
        }
      }
      __syncwarp();
    };
    for (;;) {
      if (!mbar_wait(&S.item_full[it], iph)) {
        if (lane == 0) atomicExch(a.status, kStatusWaitFullTimeout);
        break;
      }
      const Shared::Item m = S.items[it];
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.item_empty[it]);
      if (++it == kItems) {
        it = 0;
        iph ^= 1u;
      }
      if (m.kind == kItemEnd) break;
      if (m.kind == kItemGuEnd) {
        if (lane == 0) {
          S.gbar_epoch = grid_arrive(a.gbar, N + a.grid_extra);
          mbar_arrive(&S.gbar_arrived);
        }
        __syncwarp();
        continue;
      }
      if (m.kind == kItemDnWhole) {
        count_dn(m.rb);
        continue;
      }
      // a head piece begins: sum the unit's later pieces, CTAs cta + 1 .. c_last in order, into `pre`.
      // Each later piece's partial sums are 64-bit stores of (tag, value): a value is this phase's once
      // its tag is, so the loads themselves are the wait (no flag, no fence on either side). A down head
      // starts gathering before the grid barrier opens, while the slots may still hold gate+up sums:
      // those carry the gate+up tag.
      const bool gu = m.kind == kItemGuHead;
      const uint32_t tag = S.tag_base + (gu ? 1u : 2u);
      const int c_last = cta_at(gu ? pos_gu(m.ue - 1) : pos_dn(m.ue - 1), gu ? Cg : Cd, gu ? Ng : Nd);
      const int nv = m.n * 256;  // values of a piece (token t, gate/up m at (2 t + m) * 128 + row)
      for (int c = cta + 1; c <= c_last; ++c) {
        const unsigned long long* src =
            reinterpret_cast<const unsigned long long*>(a.partials + static_cast<int64_t>(c) * 2 * kPartialSlotFloats);
        for (int base = 0; base < nv; base += 256) {  // eight loads in flight per lane
          float v[8];
          const uint64_t t0 = global_timer_ns();
          for (;;) {  // until every value of the batch carries the tag (bounded)
            bool ready = true;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int idx = base + lane + 32 * j;
              v[j] = 0.0f;
              if (idx < nv && (gu || !(idx & 128))) {  // down: one sum per token
                const unsigned long long w = ld_relaxed_gpu_u64(src + idx);
                ready = ready && static_cast<uint32_t>(w >> 32) == tag;
                v[j] = __uint_as_float(static_cast<uint32_t>(w));
              }
            }
            if (__all_sync(0xffffffffu, ready)) break;
            if (__shfl_sync(0xffffffffu, global_timer_ns() - t0 > kWaitLimitNs ? 1 : 0, 0)) {
              if (lane == 0) atomicExch(a.status, kStatusWaitFullTimeout);
              break;
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int idx = base + lane + 32 * j;
            if (idx < nv && (gu || !(idx & 128))) pre[idx] = c == cta + 1 ? v[j] : pre[idx] + v[j];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pre_ready);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.helper_done);
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

    // A later piece of a unit split between CTAs (the range's first unit, begun in an earlier CTA):
    // this CTA's partial sums (vals[t][m], m < kM, full in every quarter after the shuffles) into its
    // partial slot as (tag, value) pairs, for the unit's head to gather; nothing else to wait for.
    auto publish = [&](auto& vals, auto kMc, uint32_t tag) {
      constexpr int kM = decltype(kMc)::value;
      unsigned long long* mine =
          reinterpret_cast<unsigned long long*>(a.partials + static_cast<int64_t>(cta) * 2 * kPartialSlotFloats);
      if (q == 0) {
        const unsigned long long hi = static_cast<unsigned long long>(tag) << 32;
#pragma unroll
        for (int t = 0; t < kNE; ++t)
#pragma unroll
          for (int m = 0; m < kM; ++m) st_relaxed_gpu_u64(mine + (t * 2 + m) * 128 + r, hi | __float_as_uint(vals[t][m]));
      }
    };
    // A head piece: add the later pieces' sum the helper gathered (their CTA order after the head's)
    uint32_t pre_ph = 0;
    auto add_pre = [&](auto& vals, auto kMc) {
      constexpr int kM = decltype(kMc)::value;
      if (!mbar_wait(&S.pre_ready, pre_ph) && tid == 0) atomicExch(a.status, kStatusWaitFullTimeout);
      pre_ph ^= 1u;
      if (q == 0) {
#pragma unroll
        for (int t = 0; t < kNE; ++t)
#pragma unroll
          for (int m = 0; m < kM; ++m) vals[t][m] += pre[(t * 2 + m) * 128 + r];
      }
    };
    // Post an item to the helper once every compute thread's stores (partial sums, h, Y) are done
    // (the barrier, then one thread's release on the item's mbarrier), and go on. An entry is written
    // again only after the helper has read it.
    int it = 0;
    uint32_t iph = 0;
    auto post = [&](int kind, int ub, int ue, const Unit& un) {
      named_bar_sync(2, kComputeThreads);
      if (tid == 0) {
        if (!mbar_wait(&S.item_empty[it], iph ^ 1u)) atomicExch(a.status, kStatusWaitEmptyTimeout);
        Shared::Item& m = S.items[it];
        m.ub = ub;
        m.ue = ue;
        m.kind = kind;
        m.p0 = un.p0;
        m.n = un.n;
        m.rb = un.rb;
        mbar_arrive(&S.item_full[it]);
      }
      if (++it == kItems) {
        it = 0;
        iph ^= 1u;
      }
    };
    // The combines of the row blocks the helper found complete, out[t, rows] = bf16(sum_j w[t, j] *
    // Y[inv_pos[t, j], rows]) in slot order: each thread takes outputs tid, tid + 512, ..., so the
    // threads need not agree on when they look. A row block's last unit is nearly always a range's
    // last piece, i.e. found at the phase's end, where the compute warps have nothing else to do.
    int owed_done = 0;
    auto drain_owed = [&]() {
      for (;;) {
        const int n = *reinterpret_cast<volatile int*>(&S.owed_n);
        if (owed_done >= n) return;
        __threadfence();  // the helper acquired every unit's Y of the row block before posting it
        const int rb = reinterpret_cast<volatile int*>(S.owed)[owed_done++];
        for (int idx = tid; idx < T * 128; idx += kComputeThreads) {
          const int t = idx >> 7;
          const int row = rb * 128 + (idx & 127);
          float acc2 = 0.0f;
          for (int j = 0; j < k; ++j) {
            const float y = __ldcg(a.Y + static_cast<int64_t>(S.inv[t * k + j]) * H + row);
            acc2 = __fadd_rn(acc2, __fmul_rn(S.w[t * k + j], y));
          }
          a.out[static_cast<int64_t>(t) * H + row] = __bfloat16_as_ushort(__float2bfloat16_rn(acc2));
        }
      }
    };

    // ---------------------------- gate+up ----------------------------
    for (int i = g_beg; i < g_end;) {
      const int u = i / KIg;
      const int ub = u * KIg, ue = ub + KIg;
      const int pe = ue < g_end ? ue : g_end;
      const Unit un = gu_unit(u);
      const bool head = ub >= g_beg && ue > g_end;  // the unit goes on in later CTAs; this one finishes it
      if (head) post(kItemGuHead, ub, ue, un);      // the helper gathers the later pieces meanwhile
      float acc[kNE][2];  // gate, up (INT8: sums of scaled group sums)
#pragma unroll
      for (int t = 0; t < kNE; ++t) acc[t][0] = acc[t][1] = 0.0f;
      for (; i < pe; ++i) {
        const uint32_t st = take();
        const uint32_t rowg = st + r * 128, rowu = rowg + 16384;
        if constexpr (!kInt8) {
          const uint32_t c0 = ((2 * q) ^ x7) << 4, c1 = ((2 * q + 1) ^ x7) << 4;
          const uint4 g0 = lds128(rowg + c0), g1 = lds128(rowg + c1);
          const uint4 u0 = lds128(rowu + c0), u1 = lds128(rowu + c1);
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
          // chunks 2q and 2q + 1 (int8 elements 32q .. 32q + 31) of the group: the weights as they are,
          // against the token record's digit planes (dp4a); quarters 2 and 3 take the two chunks in the
          // other order so that, in every load, the four quarters' digit reads fall in distinct banks
          const int ca = 2 * q + (q >> 1), cb = 2 * q + 1 - (q >> 1);
          const uint32_t c0 = (ca ^ x7) << 4, c1 = (cb ^ x7) << 4;
          const uint4 g0 = lds128(rowg + c0), g1 = lds128(rowg + c1);
          const uint4 u0 = lds128(rowu + c0), u1 = lds128(rowu + c1);
          const uint32_t gq[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          const uint32_t uq[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          const int kk = static_cast<int>(i - ub);
          const float sg = lds_f32(st + G::kWBytes + r * 16 + (kk & 3) * 4);
          const float su = lds_f32(st + G::kWBytes + 2048 + r * 16 + (kk & 3) * 4);
#pragma unroll
          for (int t = 0; t < kNE; ++t) {
            if (t < un.n) {
              const uint32_t rec = G::kRecSmem ? smem_addr(rec_smem) + kk * kRec : st + G::kTokOff + t * G::kSliceGU;
              const float xsc = lds_f32(rec + kRecScale);  // the record's 2^e
              acc[t][0] = fmaf(record_dot(rec, ca, cb, gq), sg * xsc, acc[t][0]);
              acc[t][1] = fmaf(record_dot(rec, ca, cb, uq), su * xsc, acc[t][1]);
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
      if (ub < g_beg) {  // a later piece of a unit begun in an earlier CTA: published for its head
        publish(acc, std::integral_constant<int, 2>{}, S.tag_base + 1u);
        continue;
      }
      if (head) add_pre(acc, std::integral_constant<int, 2>{});
      {
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
          // h rounded to bf16, then its record: this unit's 128 rows are one scale group of the down
          // projection's reduction, so the group's largest |h| sets the record's fixed point
          float hv[kNE];
#pragma unroll
          for (int t = 0; t < kNE; ++t) {
            float m = 0.0f;  // only quarter 0 holds the full sums after add_pre
            if (t < un.n) {
              hv[t] = __bfloat162float(__float2bfloat16_rn(silu_mul(acc[t][0], acc[t][1])));
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
                const int kh = fixed_exponent(m);
                const int X = fixed_value(hv[t], kh);
                uint8_t* rec = static_cast<uint8_t*>(a.h) +
                               (static_cast<int64_t>(un.p0 + t) * (I / 128) + un.rb) * kRec;
                rec[r] = static_cast<uint8_t>(X & 0xff);
                rec[128 + r] = static_cast<uint8_t>((X >> 8) & 0xff);
                rec[256 + r] = static_cast<uint8_t>((X >> 16) & 0xff);
                if (r == 0) *reinterpret_cast<float*>(rec + kRecScale) = ldexpf(1.0f, kh);
              }
            }
          }
          red_buf ^= 1;
        }
      }
    }

    // ---- gate+up done: the helper arrives at the grid barrier after the items before this one (the
    // split units it finishes write h too)
    post(kItemGuEnd, 0, 0, Unit{0, 0, 0, 0});

    // ---------------------------- down ----------------------------
    for (int i = d_beg; i < d_end;) {
      const int u = i / KId;
      const int ub = u * KId, ue = ub + KId;
      const int pe = ue < d_end ? ue : d_end;
      const Unit un = dn_unit(u);
      const bool head = ub >= d_beg && ue > d_end;
      if (head) post(kItemDnHead, ub, ue, un);
      float acc[kNE][1];
#pragma unroll
      for (int t = 0; t < kNE; ++t) acc[t][0] = 0.0f;
      for (; i < pe; ++i) {
        const uint32_t st = take();
        // every quarter reads the same two chunks of both reduction slices of the slot (the two boxes):
        // in every load the four quarters touch four distinct chunk pairs, i.e. distinct banks
        const uint32_t rowa = st + r * 128, rowb = rowa + 16384;
        if constexpr (!kInt8) {
          const int ca = 2 * q, cb = 2 * q + 1;
          const uint4 w0 = lds128(rowa + ((ca ^ x7) << 4)), w1 = lds128(rowa + ((cb ^ x7) << 4));
          const uint4 w2 = lds128(rowb + ((ca ^ x7) << 4)), w3 = lds128(rowb + ((cb ^ x7) << 4));
          const uint32_t wq[16] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w,
                                   w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
          // h elements 16q .. 16q + 15 of each 64-element slice: bytes 32q and 128 + 32q of the slot
          const uint32_t tb = st + G::kTokOff + q * 32;
#pragma unroll
          for (int t = 0; t < kNE; ++t) {
            if (t < un.n) {
              float ya = acc[t][0], yb = 0.0f;
#pragma unroll
              for (int hq = 0; hq < 4; ++hq) {
                const uint4 xv = lds128(tb + t * G::kSliceDN + (hq >> 1) * 128 + (hq & 1) * 16);
                ya = fma2_bf16(wq[4 * hq + 0], xv.x, ya);
                yb = fma2_bf16(wq[4 * hq + 1], xv.y, yb);
                ya = fma2_bf16(wq[4 * hq + 2], xv.z, ya);
                yb = fma2_bf16(wq[4 * hq + 3], xv.w, yb);
              }
              acc[t][0] = ya + yb;
            }
          }
        } else {
          // int8 elements 32q .. 32q + 31 of each of the slot's two scale groups (one per box), against
          // the two h records' digit planes; quarters 2 and 3 take their two chunks in the other order
          const int ca = 2 * q + (q >> 1), cb = 2 * q + 1 - (q >> 1);
          const uint4 w0 = lds128(rowa + ((ca ^ x7) << 4)), w1 = lds128(rowa + ((cb ^ x7) << 4));
          const uint4 w2 = lds128(rowb + ((ca ^ x7) << 4)), w3 = lds128(rowb + ((cb ^ x7) << 4));
          const uint32_t wa[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          const uint32_t wb[8] = {w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
          const int kk2 = static_cast<int>(i - ub);
          const uint32_t sbox = st + G::kWBytes + r * 16;
          const float sa = lds_f32(sbox + ((2 * kk2) & 3) * 4), sb = lds_f32(sbox + ((2 * kk2 + 1) & 3) * 4);
#pragma unroll
          for (int t = 0; t < kNE; ++t) {
            if (t < un.n) {
              const uint32_t reca = st + G::kTokOff + t * G::kSliceDN, recb = reca + kRec;
              acc[t][0] = fmaf(record_dot(reca, ca, cb, wa), sa * lds_f32(reca + kRecScale), acc[t][0]);
              acc[t][0] = fmaf(record_dot(recb, ca, cb, wb), sb * lds_f32(recb + kRecScale), acc[t][0]);
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
      if (ub < d_beg) {  // a later piece of a unit begun in an earlier CTA: published for its head
        publish(acc, std::integral_constant<int, 1>{}, S.tag_base + 2u);
      } else {
        if (head) add_pre(acc, std::integral_constant<int, 1>{});
        // the unit's Y rows are final; the helper counts the unit toward its row block
        const int h_row = un.rb * 128 + r;
        if (q == 0) {
#pragma unroll
          for (int t = 0; t < kNE; ++t)
            if (t < un.n) a.Y[static_cast<int64_t>(un.p0 + t) * H + h_row] = acc[t][0];
        }
        post(kItemDnWhole, ub, ue, un);
      }
      drain_owed();
    }
    post(kItemEnd, 0, 0, Unit{0, 0, 0, 0});
    if (!mbar_wait(&S.helper_done, 0) && tid == 0) atomicExch(a.status, kStatusWaitFullTimeout);
    drain_owed();
  }
  __syncthreads();
}

template <bool kInt8, int kNE, bool kDeep>
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
  e = cudaFuncSetAttribute(decode_step_kernel<kInt8, kNE, kDeep>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
  if (e != cudaSuccess) return e;
  int per_sm = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_step_kernel<kInt8, kNE, kDeep>, kThreads,
                                                    smem_bytes<kInt8, kNE, kDeep>(kDeep ? kDeepMaxH : 16384));
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

template <bool kInt8, int kNE, bool kDeep = false>
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
  cudaError_t e = prepare<kInt8, kNE, kDeep>(&max_ctas);
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
  cfg.dynamicSmemBytes = smem_bytes<kInt8, kNE, kDeep>(p.H);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_ok.load(std::memory_order_relaxed) ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, decode_step_kernel<kInt8, kNE, kDeep>, tg, tu, td, tsg, tsu, tsd, p.args);
  if (e != cudaSuccess && cfg.numAttrs == 2) {
    cudaGetLastError();  // clear the launch error, then launch cooperatively alone
    pdl_ok.store(0, std::memory_order_relaxed);
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_step_kernel<kInt8, kNE, kDeep>, tg, tu, td, tsg, tsu, tsd, p.args);
  }
  return e;
}

}  // namespace dec

bool decode_step_supported(int T, int H, int I, int E, int k, bool int8) {
  if (T < 1 || T > kDecodeMaxT || static_cast<int64_t>(T) * k > kDecodeMaxP || E > 256) return false;
  if (H % 128 || I % 128) return false;
  if (int8 && (H % 512 || I % 512)) return false;  // scale boxes of 4 groups; two groups per down slot
  // 32-bit schedule arithmetic and the helper's list of row blocks; INT8 at T = 1: the records in shared memory
  if (H > 16384 || I > 32768) return false;
  return true;
}

// Tokens per pass: exactly one per expert at T = 1; four while the batch has at most one assignment
// per expert on average (a hotter expert takes several passes); eight above. Fewer tokens per pass
// keep the compute loops short (instruction-cache misses were the top stall of the INT8 kernel at T = 1
// with eight-token loops).
template <bool kInt8>
cudaError_t launch_ne(const DecodePlan& plan, cudaStream_t stream) {
  const DecodeArgs& a = plan.args;
  if (a.T == 1) {
    if constexpr (kInt8) {  // five slots where the token's records leave room for them
      if (a.H <= dec::kDeepMaxH) return dec::launch<true, 1, true>(plan, stream);
    }
    return dec::launch<kInt8, 1>(plan, stream);
  }
  if constexpr (kInt8) {
    return dec::launch<true, 4>(plan, stream);  // INT8: passes of at most 4 (the slots hold 4 tokens' records)
  } else {
    if (static_cast<int64_t>(a.T) * a.k <= a.E) return dec::launch<false, 4>(plan, stream);
    return dec::launch<false, 8>(plan, stream);
  }
}

cudaError_t launch_decode_step(const DecodePlan& plan, cudaStream_t stream) {
  return plan.int8 ? launch_ne<true>(plan, stream) : launch_ne<false>(plan, stream);
}

}  // namespace moe
