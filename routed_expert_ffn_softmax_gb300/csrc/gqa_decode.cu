// Decode-phase grouped-query attention on the 5th-generation tensor cores.
//
// HiNa-MoE (arXiv 2610.05123), §6.1 and Figure 9: in decoding, the G = h_q / h_kv query heads
// that share a key/value head form a small G x d block, and attention for that key/value head is
// two small matrix products: scores = (query block) x K^T, then probabilities x V. Here both run
// on tcgen05.mma with the key dimension as the 128-row M side:
//     S^T [128 keys x 16]  = K_tile [128 keys x d] . Q_block^T       (A = K tile, K-major)
//     O^T [d x 16]        += V_tile^T [d x 128 keys] . P^T            (A = V tile read MN-major)
// so neither the key/value cache nor the query is rearranged in memory: TMA lands K and V tiles
// exactly as the cache stores them ([B, h_kv, L_cap, d], d contiguous) and the V tile is consumed
// transposed through the MMA's operand descriptor, the GPU counterpart of §6.1's on-demand
// layout change of the value tiles. The query block (G rows, padded to 16 with whatever rows follow
// it, whose probabilities are written as zero) stays in shared memory for the whole piece.
//
// Numerics: scores and the online softmax in fp32 (base-2 exponent, scale * log2(e) folded into
// the scores, the hardware's approximate 2^x at about 2^-22 relative error), probabilities rounded
// to bf16 for the second product (its operands must share one 16-bit type with V), fp32
// accumulation, output rounded once to bf16.
//
// Work split: the key tiles of all (sequence, key/value head) segments form one list; each CTA
// (one per SM) takes a contiguous range of it (stream-K), so long and short sequences balance to
// within one tile. A segment cut between CTAs is finished by the CTA that arrives last, which
// merges the pieces' (max, sum, unnormalised output) in CTA order: the result does not depend on
// timing.
//
// Per CTA, 10 warps:
//   warp 0      TMA producer: per piece the query block, per tile K and V (4 boxes of
//               128 keys x 64 dims, 64 KB) into a 3-stage ring;
//   warp 1      owns TMEM (64 columns); lane 0 issues the MMAs: S^T of tile i+1 before O^T of
//               tile i within a piece, so the softmax of a tile always finds the next tile's
//               scores under way (at a piece boundary the last O^T goes first);
//               a tile's S^T and the O^T of the tile two before it sit in adjacent TMEM columns
//               and are read back with one load, two tiles after that O^T's MMA was issued;
//   warps 2-5   softmax (thread = key of the tile for the scores, = dimension for the output):
//               masked scaled scores, tile maxima across the 128 keys, probabilities to shared
//               memory in the MMA's operand layout, and the rescale-and-add of earlier O^T; at
//               the end of a piece they hand its running state over through TMEM and go on;
//   warps 6-9   finisher: per piece, the last two O^T, the softmax denominators over the 128
//               key threads, and the output row, or the partial and the merge of a cut segment,
//               all while the softmax warps work on the next piece.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace gqa {

constexpr int kD = 128;                       // head dimension
constexpr int kKeys = 128;                    // keys per tile
constexpr int kN = 16;                        // MMA N: query heads of a group, padded
constexpr int kStages = 3;
constexpr int kBox = kKeys * 64 * 2;          // one TMA box: 128 rows x 64 dims x 2 B = 16 KB
constexpr int kStageBytes = 4 * kBox;         // K (2 boxes) then V (2 boxes)
constexpr int kQBytes = kN * kD * 2;          // 4 KB: 2 boxes of 16 rows x 128 B
constexpr int kPBytes = kN * kKeys * 2;       // 4 KB
constexpr int kThreads = 320;
constexpr int kSoft = 128;                    // softmax threads (warps 2..5); finisher: warps 6..9
constexpr int kScan = 256;                    // threads of the sequence prefix (warps 2..9)
constexpr int kSlotFloats = kGqaSlotFloats;   // partial of one piece: o[16][128], m[16], l[16]
constexpr int kNumBars = 2 * kStages + 2 * 9 + 1;

// TMEM columns: S^T of buffer k at 32k, O^T of buffer k at 32k + 16, so a tile's scores and the
// O^T of the tile two before it (same buffer) are 32 adjacent columns, read with one load.
// Columns 64 + 32k hold hand-off k from the softmax warps to the finisher warps: the piece's
// running output (16 columns) and each key thread's partial softmax sums (16 columns).
constexpr int kTmemCols = 128;
__host__ __device__ constexpr uint32_t col_s(int k) { return 32u * k; }
__host__ __device__ constexpr uint32_t col_o(int k) { return 32u * k + 16u; }
__host__ __device__ constexpr uint32_t col_h(int k) { return 64u + 32u * k; }

constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffP = kOffQ + 2 * kQBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kOffRed = kOffBar + 256;         // tile maxima [2][4][16] + sums [4][16] floats
constexpr int kOffHand = kOffRed + (2 * 4 * kN + 4 * kN) * 4;  // hand-off scalars [2][3][16] floats
constexpr int kOffMisc = kOffHand + 2 * 3 * kN * 4;
constexpr int kOffPre = kOffMisc + 64;         // tile prefix over sequences, kMaxSeqs + 1 ints
constexpr int kSmem = kOffPre + (kGqaMaxSeqs + 1) * 4;
static_assert(kNumBars * 8 <= 256, "barrier area");
static_assert(kSlotFloats == kN * kD + 2 * kN, "partial slot layout");
static_assert(kSmem <= 232448, "dynamic shared memory per CTA");
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "operand tiles keep the 1024-byte swizzle alignment");
static_assert(kGqaMaxSeqs <= 8 * kScan, "each prefix thread keeps at most 8 lengths in registers");

struct Params {
  const int32_t* seq_lens;  // [B]
  uint16_t* out;            // [B, h_q, d] bf16
  float* partials;          // [kPartialCtas][2][kSlotFloats]
  int32_t* counters;        // [kPartialCtas], zero on entry, left zero
  int32_t* status;
  int B, h_q, h_kv, G, L_cap;
  float scale_log2;         // softmax scale * log2(e)
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Byte offset of element (row, col) of a 16-row operand tile stored K-major with the 128-byte
// swizzle: two 64-column boxes of 16 x 128 B, 16-byte chunks XORed with the row within 8.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col) {
  const int box = col >> 6;
  const int c = col & 63;
  return static_cast<uint32_t>(box * 2048 + (row >> 3) * 1024 + (row & 7) * 128 + ((((c >> 3) ^ row) & 7) << 4) +
                               (c & 7) * 2);
}

// Sequence b's tile count; a length outside [0, L_cap] counts as empty (and is reported).
__device__ __forceinline__ int seq_tiles(int len, int L_cap) {
  return (len <= 0 || len > L_cap) ? 0 : (len + kKeys - 1) / kKeys;
}

// kGP: the group size rounded up to a power of two (1..16); p.G <= kGP is the real group size.
template <int kGP>
__global__ void __launch_bounds__(kThreads, 1)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmQ, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* empty = full + kStages;
  uint64_t* q_full = empty + kStages;  // [2]
  uint64_t* q_empty = q_full + 2;      // [2]
  uint64_t* s_full = q_empty + 2;      // [2]
  uint64_t* s_free = s_full + 2;       // [2]
  uint64_t* p_full = s_free + 2;       // [2]
  uint64_t* o_full = p_full + 2;       // [2]
  uint64_t* o_free = o_full + 2;       // [2]
  uint64_t* h_full = o_free + 2;       // [2] softmax -> finisher hand-off
  uint64_t* h_empty = h_full + 2;      // [2]
  uint64_t* mma_done = h_empty + 2;    // [1]
  float* red_max = reinterpret_cast<float*>(smem + kOffRed);  // [2][4][kN]
  float* red_sum = red_max + 2 * 4 * kN;                       // [4][kN]
  float* hand = reinterpret_cast<float*>(smem + kOffHand);     // [2][3][kN]: m, a1, a2
  int* misc = reinterpret_cast<int*>(smem + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 12);
  int* pre = reinterpret_cast<int*>(smem + kOffPre);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], kSoft);
      mbar_init(&p_full[b], kSoft);
      mbar_init(&o_full[b], 1);
      mbar_init(&o_free[b], kSoft);  // softmax or finisher threads, 128 either way
      mbar_init(&h_full[b], kSoft);
      mbar_init(&h_empty[b], kSoft);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmQ);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);

  // ---- tile prefix over sequences: pre[b] = tiles of sequences < b (warps 2..9, <= 8 each)
  const int sc = tid - 64;
  const int per = (p.B + kScan - 1) / kScan;
  const int i0 = sc * per;
  const int i1 = warp >= 2 ? min(p.B, i0 + per) : 0;
  // warming L2 with the lengths is safe before the wait (L2 is where later writes land too)
  if (warp >= 2 && i0 < i1) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.seq_lens + i0));
  // The lengths (and the cache rows of the newest token) may come from the preceding kernel.
  pdl_wait_predecessor();
  pdl_allow_successor();
  if (warp >= 2) {
    int nt[8];
    int sum = 0;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      nt[k] = 0;
      if (i0 + k < i1) {
        const int len = p.seq_lens[i0 + k];
        bad |= (len < 0 || len > p.L_cap);
        nt[k] = seq_tiles(len, p.L_cap);
        sum += nt[k];
      }
    }
    if (bad) atomicExch(p.status, kStatusBadSeqLen);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) misc[warp - 2] = incl;
    named_bar_sync(3, kScan);
    int base = 0;
    for (int w = 0; w < warp - 2; ++w) base += misc[w];
    int run = base + incl - sum;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (i0 + k < i1) {
        pre[i0 + k] = run;
        run += nt[k];
      }
    if (sc == kScan - 1) pre[p.B] = base + incl;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // The first NC = min(tiles, CTAs) CTAs share the tiles, each at least one (a CTA with an empty
  // range would be counted as a piece of a segment it never touched): CTA c < rm takes q + 1
  // tiles, the others q. All tile arithmetic is 32-bit (the host bounds the tile count).
  const int total = p.h_kv * pre[p.B];
  const int grid = gridDim.x;
  const int NC = total < grid ? total : grid;
  const int cta = blockIdx.x;
  const int q_tiles = NC > 0 ? total / NC : 0;
  const int rm = NC > 0 ? total - q_tiles * NC : 0;
  auto range_start = [&](int c) { return c * q_tiles + min(c, rm); };
  const int beg = cta < NC ? range_start(cta) : 0;
  const int end = cta < NC ? range_start(cta + 1) : 0;

  // The piece of the range that starts at tile x: sequence b, key/value head j, first tile tl of
  // nt tiles in the segment, n tiles in this piece, segment's first tile in the global list.
  struct Piece {
    int b, j, tl, nt, n, seg0;
  };
  auto locate = [&](int x) -> Piece {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {  // last sequence whose first tile is <= x (skips empty sequences)
      const int mid = (lo + hi + 1) >> 1;
      if (p.h_kv * pre[mid] <= x) lo = mid; else hi = mid - 1;
    }
    Piece r;
    r.b = lo;
    r.nt = pre[lo + 1] - pre[lo];
    const int off = x - p.h_kv * pre[lo];  // < h_kv * nt
    r.j = off / r.nt;
    r.tl = off - r.j * r.nt;
    r.seg0 = x - r.tl;
    r.n = min(end - x, r.nt - r.tl);
    return r;
  };

  if (warp == 0) {
    // =========================== TMA producer ===========================
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      int it = 0;
      int pi = 0;
      bool ok = true;
      for (int x = beg; x < end && ok; ++pi) {
        const Piece pc = locate(x);
        const int qb = pi & 1;
        if (!mbar_wait(&q_empty[qb], ((pi >> 1) & 1) ^ 1)) {
          ok = false;
          break;
        }
        uint8_t* qs = smem + kOffQ + qb * kQBytes;
        const int qrow = pc.b * p.h_q + pc.j * p.G;
        mbar_arrive_expect_tx(&q_full[qb], kQBytes);
        tma_load_2d(qs, &tmQ, &q_full[qb], 0, qrow);
        tma_load_2d(qs + 2048, &tmQ, &q_full[qb], 64, qrow);
        const int z = pc.b * p.h_kv + pc.j;
        for (int t = pc.tl; t < pc.tl + pc.n; ++t, ++it) {
          const int st = it % kStages;
          if (!mbar_wait(&empty[st], static_cast<uint32_t>(((it / kStages) & 1) ^ 1))) {
            ok = false;
            break;
          }
          uint8_t* kv = smem + st * kStageBytes;
          mbar_arrive_expect_tx(&full[st], kStageBytes);
          tma_load_3d(kv, &tmK, &full[st], 0, t * kKeys, z, policy);
          tma_load_3d(kv + kBox, &tmK, &full[st], 64, t * kKeys, z, policy);
          tma_load_3d(kv + 2 * kBox, &tmV, &full[st], 0, t * kKeys, z, policy);
          tma_load_3d(kv + 3 * kBox, &tmV, &full[st], 64, t * kKeys, z, policy);
        }
        x += pc.n;
      }
      if (!ok) atomicExch(p.status, kStatusWaitEmptyTimeout);
      // never leave copies in flight: the last stages and query blocks issued
      const int n = it < kStages ? it : kStages;
      for (int i = it - n; i < it; ++i)
        if (!mbar_wait(&full[i % kStages], static_cast<uint32_t>((i / kStages) & 1))) {
          atomicExch(p.status, kStatusDrainTimeout);
          break;
        }
      for (int q = pi - 2 < 0 ? 0 : pi - 2; q < pi; ++q)
        if (!mbar_wait(&q_full[q & 1], (q >> 1) & 1)) {
          atomicExch(p.status, kStatusDrainTimeout);
          break;
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // =========================== MMA issuer ===========================
    if (lane == 0) {
      const uint32_t sbase = smem_addr(smem);
      const uint32_t idesc_s = umma_idesc_bf16_m128(kN);
      const uint32_t idesc_o = umma_idesc_bf16_m128(kN) | kIdescAMajorMN;
      bool ok = true;
      auto fail = [&](int code) {
        ok = false;
        atomicExch(p.status, code);
      };
      // O^T of tile i: V^T (MN-major view of the V boxes) times the probabilities
      auto issue_o = [&](int i) {
        const int sb = i & 1;
        const uint32_t ph = static_cast<uint32_t>((i >> 1) & 1);
        const int st = i % kStages;
        if (ok && !mbar_wait(&p_full[sb], ph)) fail(kStatusWaitFullTimeout);
        if (ok && !mbar_wait(&o_free[sb], ph ^ 1)) fail(kStatusWaitEmptyTimeout);
        if (ok) {
          tc_fence_after_sync();
          const uint32_t v = sbase + st * kStageBytes + 2 * kBox;
          const uint32_t pt = sbase + kOffP + sb * kPBytes;
#pragma unroll
          for (int s = 0; s < kKeys / 16; ++s)
            umma_bf16(tmem_base + col_o(sb), umma_desc_sw128_mn(v + s * 2048, kBox),
                      umma_desc_sw128(pt + (s >> 2) * 2048 + (s & 3) * 32), idesc_o, s > 0);
        }
        umma_commit(&o_full[sb]);
        umma_commit(&empty[st]);
      };
      int it = 0;
      int pi = 0;
      for (int x = beg; x < end; ++pi) {
        const Piece pc = locate(x);
        const int qb = pi & 1;
        if (ok && !mbar_wait(&q_full[qb], (pi >> 1) & 1)) fail(kStatusWaitFullTimeout);
        const uint32_t qs = sbase + kOffQ + qb * kQBytes;
        for (int t = 0; t < pc.n; ++t, ++it) {
          const int st = it % kStages;
          const int sb = it & 1;
          if (ok && !mbar_wait(&full[st], static_cast<uint32_t>((it / kStages) & 1))) fail(kStatusWaitFullTimeout);
          if (ok && !mbar_wait(&s_free[sb], static_cast<uint32_t>(((it >> 1) & 1) ^ 1)))
            fail(kStatusWaitEmptyTimeout);
          if (ok) {
            tc_fence_after_sync();
            const uint32_t k = sbase + st * kStageBytes;
#pragma unroll
            for (int s = 0; s < kD / 16; ++s)
              umma_bf16(tmem_base + col_s(sb), umma_desc_sw128(k + (s >> 2) * kBox + (s & 3) * 32),
                        umma_desc_sw128(qs + (s >> 2) * 2048 + (s & 3) * 32), idesc_s, s > 0);
          }
          umma_commit(&s_full[sb]);
          if (t == pc.n - 1) umma_commit(&q_empty[qb]);
          // the previous tile's O^T (across a piece boundary too: the finisher, not the softmax,
          // waits for a piece's last one)
          if (it > 0) issue_o(it - 1);
        }
        x += pc.n;
      }
      if (it > 0) issue_o(it - 1);
      // every MMA has completed before TMEM is released
      umma_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) atomicExch(p.status, kStatusDrainTimeout);
    }
    __syncwarp();
  } else {
    const bool finisher = warp >= 6;
    const int gt = finisher ? tid - 192 : tid - 64;  // 0..127 within the warpgroup
    const int q4 = warp & 3;                       // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;                  // key of the tile (scores), dimension (output)
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16);
    // `ok` stays uniform across each warp (the waits below vote), because tcgen05.ld/st must be
    // executed by all 32 lanes together
    bool ok = true;
    auto wait_warp = [&](uint64_t* bar, uint32_t parity, int code) {
      const bool w = __all_sync(0xffffffffu, ok && mbar_wait(bar, parity));
      if (!w && ok) {
        ok = false;
        atomicExch(p.status, code);
      }
    };

    if (!finisher) {
      // =========================== softmax (warps 2..5) ===========================
      // probability rows G..15 of both buffers stay zero for the whole kernel
      for (int i = gt; i < 2 * kN * kKeys; i += kSoft) {
        const int buf = i / (kN * kKeys);
        const int row = (i / kKeys) % kN;
        const int col = i % kKeys;
        if (row >= p.G) *reinterpret_cast<uint16_t*>(smem + kOffP + buf * kPBytes + sw128_offset(row, col)) = 0;
      }
      fence_proxy_async_smem();

      int it = 0;
      int pi = 0;
      for (int x = beg; x < end; ++pi) {
        const Piece pc = locate(x);
        const int len = p.seq_lens[pc.b];
        // a1, a2: the rescale factors of the previous tile and of the one before it
        float m_run[kGP], l_thr[kGP], o_acc[kGP], a1[kGP], a2[kGP];
#pragma unroll
        for (int h = 0; h < kGP; ++h) {
          m_run[h] = -INFINITY;
          l_thr[h] = 0.0f;
          o_acc[h] = 0.0f;
          a1[h] = a2[h] = 0.0f;
        }
        for (int t = pc.tl; t < pc.tl + pc.n; ++t, ++it) {
          const int sb = it & 1;
          const int st = it % kStages;
          // the O^T of the tile two before (same buffer) is consumed with this tile's scores: its
          // MMA was issued a whole tile ago, so this wait is normally already satisfied
          const bool prev = t >= pc.tl + 2;
          wait_warp(&s_full[sb], static_cast<uint32_t>((it >> 1) & 1), kStatusWaitFullTimeout);
          if (prev) wait_warp(&o_full[sb], static_cast<uint32_t>(((it - 2) >> 1) & 1), kStatusWaitFullTimeout);
          tc_fence_after_sync();
          float so[32];  // scores of this tile, then O^T of the tile two before
          if (ok) {
            tmem_ld32(lane_base + col_s(sb), so);
          } else {
#pragma unroll
            for (int h = 0; h < 32; ++h) so[h] = 0.0f;
          }
          tc_fence_before_sync();
          mbar_arrive(&s_free[sb]);
          if (prev) {
            mbar_arrive(&o_free[sb]);
#pragma unroll
            for (int h = 0; h < kGP; ++h) o_acc[h] = fmaf(o_acc[h], a2[h], so[16 + h]);
          }

          const bool valid = t * kKeys + r < len;
          float sv[kGP], alpha[kGP];
#pragma unroll
          for (int h = 0; h < kGP; ++h) {
            sv[h] = valid ? so[h] * p.scale_log2 : -INFINITY;
            const float mx = warp_max_f32(sv[h]);
            if (lane == 0) red_max[(sb * 4 + q4) * kN + h] = mx;
          }
          named_bar_sync(1, kSoft);
          uint8_t* pt = smem + kOffP + sb * kPBytes;
#pragma unroll
          for (int h = 0; h < kGP; ++h) {
            const float* rm = red_max + sb * 4 * kN + h;
            const float mt = fmaxf(fmaxf(rm[0], rm[kN]), fmaxf(rm[2 * kN], rm[3 * kN]));
            const float m_new = fmaxf(m_run[h], mt);  // finite: every tile holds a valid key
            alpha[h] = ex2_approx(m_run[h] - m_new);
            const float pr = ex2_approx(sv[h] - m_new);
            l_thr[h] = fmaf(l_thr[h], alpha[h], pr);
            m_run[h] = m_new;
            if (h < p.G) {
              const __nv_bfloat16 pb = __float2bfloat16_rn(pr);
              *reinterpret_cast<__nv_bfloat16*>(pt + sw128_offset(h, r)) = pb;
            }
          }
          if (!valid) {
            // keys past the sequence: the cache rows there are arbitrary (even NaN) and a zero
            // probability times NaN is NaN, so clear this key's row of the V tile
            // (the wait makes the tile's landing visible to this thread before it overwrites)
            if (mbar_wait(&full[st], static_cast<uint32_t>((it / kStages) & 1))) {
              uint4* v0 = reinterpret_cast<uint4*>(smem + st * kStageBytes + 2 * kBox + r * 128);
              uint4* v1 = reinterpret_cast<uint4*>(smem + st * kStageBytes + 3 * kBox + r * 128);
#pragma unroll
              for (int c = 0; c < 8; ++c) v0[c] = v1[c] = make_uint4(0u, 0u, 0u, 0u);
            } else {
              atomicExch(p.status, kStatusWaitFullTimeout);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(&p_full[sb]);
#pragma unroll
          for (int h = 0; h < kGP; ++h) {
            a2[h] = a1[h];
            a1[h] = alpha[h];
          }
        }
        // hand the piece over: running output and partial sums to TMEM, scalars to shared memory
        const int hb = pi & 1;
        wait_warp(&h_empty[hb], ((pi >> 1) & 1) ^ 1, kStatusWaitEmptyTimeout);
        tc_fence_after_sync();
        uint32_t hv[32];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          hv[h] = __float_as_uint(h < kGP ? o_acc[h] : 0.0f);
          hv[16 + h] = __float_as_uint(h < kGP ? l_thr[h] : 0.0f);
        }
        if (ok) {
          tmem_st32(lane_base + col_h(hb), hv);
          tmem_wait_st();
        }
        if (gt == 0) {
#pragma unroll
          for (int h = 0; h < kGP; ++h) {
            hand[(hb * 3 + 0) * kN + h] = m_run[h];
            hand[(hb * 3 + 1) * kN + h] = a1[h];
            hand[(hb * 3 + 2) * kN + h] = a2[h];
          }
        }
        tc_fence_before_sync();
        mbar_arrive(&h_full[hb]);
        x += pc.n;
      }
    } else {
      // =========================== finisher (warps 6..9) ===========================
      int it = 0;
      int pi = 0;
      for (int x = beg; x < end; ++pi) {
        const Piece pc = locate(x);
        it += pc.n;  // tiles through the end of this piece
        const int hb = pi & 1;
        wait_warp(&h_full[hb], (pi >> 1) & 1, kStatusWaitFullTimeout);
        tc_fence_after_sync();
        float hv[32];
        if (ok) {
          tmem_ld32(lane_base + col_h(hb), hv);
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) hv[h] = 0.0f;
        }
        float o_acc[kGP], l_thr[kGP], m_run[kGP], a1[kGP], a2[kGP];
#pragma unroll
        for (int h = 0; h < kGP; ++h) {
          o_acc[h] = hv[h];
          l_thr[h] = hv[16 + h];
          m_run[h] = hand[(hb * 3 + 0) * kN + h];
          a1[h] = hand[(hb * 3 + 1) * kN + h];
          a2[h] = hand[(hb * 3 + 2) * kN + h];
        }
        tc_fence_before_sync();
        mbar_arrive(&h_empty[hb]);

        // the piece's last one or two O^T, in tile order
        auto drain_o = [&](int i, const float (&a)[kGP]) {
          const int sb = i & 1;
          wait_warp(&o_full[sb], static_cast<uint32_t>((i >> 1) & 1), kStatusWaitFullTimeout);
          tc_fence_after_sync();
          float ot[16];
          if (ok) {
            tmem_ld16(lane_base + col_o(sb), ot);
          } else {
#pragma unroll
            for (int h = 0; h < 16; ++h) ot[h] = 0.0f;
          }
          tc_fence_before_sync();
          mbar_arrive(&o_free[sb]);
#pragma unroll
          for (int h = 0; h < kGP; ++h) o_acc[h] = fmaf(o_acc[h], a[h], ot[h]);
        };
        if (pc.n >= 2) drain_o(it - 2, a2);
        drain_o(it - 1, a1);

        // ---- the piece's softmax denominators: sum of the 128 key threads' partial sums
        float l_tot[kGP];
#pragma unroll
        for (int h = 0; h < kGP; ++h) {
          const float sm = warp_sum(l_thr[h]);
          if (lane == 0) red_sum[q4 * kN + h] = sm;
        }
        named_bar_sync(2, kSoft);
#pragma unroll
        for (int h = 0; h < kGP; ++h)
          l_tot[h] = (red_sum[h] + red_sum[kN + h]) + (red_sum[2 * kN + h] + red_sum[3 * kN + h]);

        const bool whole = pc.tl == 0 && pc.n == pc.nt;
        uint16_t* outp = p.out + (static_cast<int64_t>(pc.b) * p.h_q + static_cast<int64_t>(pc.j) * p.G) * kD + r;
        if (whole) {
#pragma unroll
          for (int h = 0; h < kGP; ++h)
            if (h < p.G) {
              const __nv_bfloat16 v = __float2bfloat16_rn(o_acc[h] / l_tot[h]);
              outp[h * kD] = *reinterpret_cast<const uint16_t*>(&v);
            }
          named_bar_sync(2, kSoft);  // red_sum is reused by the next piece
        } else {
          // Segment cut between CTAs: its pieces are merged in CTA order by the CTA that completes
          // the set. If every other piece is already published, this one merges straight from its
          // registers; otherwise it publishes (o, m, l) and the last to arrive merges.
          auto cta_of = [&](int i) {  // the CTA whose range holds tile i
            const int big = rm * (q_tiles + 1);
            return i < big ? i / (q_tiles + 1) : rm + (i - big) / q_tiles;
          };
          const int c_first = cta_of(pc.seg0);
          const int c_last = cta_of(pc.seg0 + pc.nt - 1);
          const int others = c_last - c_first;
          if (gt == 0) misc[8] = ld_acquire_gpu(&p.counters[c_first]) == others;
          named_bar_sync(2, kSoft);
          const bool direct = misc[8] != 0;
          bool merge = direct;
          if (!direct) {
            const int slot = pi == 0 ? 0 : 1;
            float* mine = p.partials + (cta * 2 + slot) * kSlotFloats;
#pragma unroll
            for (int h = 0; h < kGP; ++h) mine[h * kD + r] = o_acc[h];
            if (gt == 0) {
#pragma unroll
              for (int h = 0; h < kGP; ++h) {
                mine[kN * kD + h] = m_run[h];
                mine[kN * kD + kN + h] = l_tot[h];
              }
            }
            named_bar_sync(2, kSoft);
            if (gt == 0) {
              // the fence after the barrier publishes the whole warpgroup's writes (cumulativity)
              __threadfence();
              const int old = atomicAdd(&p.counters[c_first], 1);
              const int last = old == others;
              if (last) p.counters[c_first] = 0;
              misc[8] = last;
            }
            named_bar_sync(2, kSoft);
            merge = misc[8] != 0;
            if (merge) __threadfence();
          } else if (gt == 0) {
            p.counters[c_first] = 0;  // every other piece has arrived: none will touch it again
          }
          if (merge) {
            // pieces whose loads are in flight together (within the 168 registers a thread has)
            constexpr int kChunk = kGP <= 4 ? 4 : (kGP <= 8 ? 2 : 1);
            float M[kGP], O[kGP], L[kGP];
#pragma unroll
            for (int h = 0; h < kGP; ++h) {
              M[h] = -INFINITY;
              O[h] = 0.0f;
              L[h] = 0.0f;
            }
            for (int c0 = c_first; c0 <= c_last; c0 += kChunk) {
              float mc[kChunk][kGP], lc[kChunk][kGP], oc[kChunk][kGP];
#pragma unroll
              for (int u = 0; u < kChunk; ++u) {
                const int c = c0 + u;
                if (c > c_last) continue;
                if (direct && c == cta) {
#pragma unroll
                  for (int h = 0; h < kGP; ++h) {
                    mc[u][h] = m_run[h];
                    lc[u][h] = l_tot[h];
                    oc[u][h] = o_acc[h];
                  }
                } else {
                  const int cslot = range_start(c) >= pc.seg0 ? 0 : 1;
                  const float* src = p.partials + (c * 2 + cslot) * kSlotFloats;
#pragma unroll
                  for (int h = 0; h < kGP; ++h) {
                    mc[u][h] = __ldcg(src + kN * kD + h);
                    lc[u][h] = __ldcg(src + kN * kD + kN + h);
                    oc[u][h] = __ldcg(src + h * kD + r);
                  }
                }
              }
#pragma unroll
              for (int u = 0; u < kChunk; ++u) {
                if (c0 + u > c_last) continue;
#pragma unroll
                for (int h = 0; h < kGP; ++h) {
                  const float m_new = fmaxf(M[h], mc[u][h]);
                  const float a_old = exp2f(M[h] - m_new);
                  const float a_c = exp2f(mc[u][h] - m_new);
                  O[h] = O[h] * a_old + oc[u][h] * a_c;
                  L[h] = L[h] * a_old + lc[u][h] * a_c;
                  M[h] = m_new;
                }
              }
            }
#pragma unroll
            for (int h = 0; h < kGP; ++h)
              if (h < p.G) {
                const __nv_bfloat16 v = __float2bfloat16_rn(O[h] / L[h]);
                outp[h * kD] = *reinterpret_cast<const uint16_t*>(&v);
              }
          }
          named_bar_sync(2, kSoft);  // misc[8] and red_sum are reused by the next piece
        }
        x += pc.n;
      }

      // ---- sequences with no keys (or a length outside [0, L_cap]) attend to nothing: output 0
      for (int b = cta; b < p.B; b += grid) {
        if (pre[b + 1] != pre[b]) continue;
        uint16_t* o = p.out + static_cast<int64_t>(b) * p.h_q * kD;
        for (int i = gt; i < p.h_q * kD; i += kSoft) o[i] = 0;
      }
    }
  }

  // ---- teardown: every role has finished; warp 1 releases TMEM
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

bool encode_kv(CUtensorMap* map, const uint16_t* base, int B, int h_kv, int L_cap) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(L_cap),
                              static_cast<cuuint64_t>(B) * h_kv};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(L_cap) * kD * 2};
  const cuuint32_t box[3] = {64, kKeys, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  TensorMapEncodeFn enc = tensor_map_encoder();
  return enc && enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_q(CUtensorMap* map, const uint16_t* q, int rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {64, kN};
  const cuuint32_t estr[2] = {1, 1};
  TensorMapEncodeFn enc = tensor_map_encoder();
  return enc && enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kGP>
cudaError_t launch_g(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q, const Params& p, int grid,
                     cudaStream_t stream) {
  constexpr int kMaxDev = 64;  // the shared-memory opt-in is per device: done once on each
  static std::atomic<bool> done[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDev || !done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(gqa_decode_kernel<kGP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDev) done[dev].store(true, std::memory_order_release);
  }
  return launch_pdl(gqa_decode_kernel<kGP>, dim3(grid), dim3(kThreads), kSmem, stream, k, v, q, p);
}

}  // namespace gqa

cudaError_t launch_gqa_decode(const GqaPlan& plan, cudaStream_t stream) {
  using namespace gqa;
  CUtensorMap tk, tv, tq;
  if (!encode_kv(&tk, plan.k_cache, plan.B, plan.h_kv, plan.L_cap) ||
      !encode_kv(&tv, plan.v_cache, plan.B, plan.h_kv, plan.L_cap) ||
      !encode_q(&tq, plan.q, plan.B * plan.h_q))
    return cudaErrorInvalidValue;
  Params p{};
  p.seq_lens = plan.seq_lens;
  p.out = plan.out;
  p.partials = plan.partials;
  p.counters = plan.counters;
  p.status = plan.status;
  p.B = plan.B;
  p.h_q = plan.h_q;
  p.h_kv = plan.h_kv;
  p.G = plan.h_q / plan.h_kv;
  p.L_cap = plan.L_cap;
  p.scale_log2 = plan.scale_log2;
  const int grid = plan.num_ctas;
  if (p.G <= 1) return launch_g<1>(tk, tv, tq, p, grid, stream);
  if (p.G <= 2) return launch_g<2>(tk, tv, tq, p, grid, stream);
  if (p.G <= 4) return launch_g<4>(tk, tv, tq, p, grid, stream);
  if (p.G <= 8) return launch_g<8>(tk, tv, tq, p, grid, stream);
  return launch_g<16>(tk, tv, tq, p, grid, stream);
}

}  // namespace moe
