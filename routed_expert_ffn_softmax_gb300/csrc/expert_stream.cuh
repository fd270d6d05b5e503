// Weight-streaming grouped expert kernels (gate+up with fused SiLU*up, and down).
//
// What they compute (HiNa-MoE, arXiv 2610.05123, §4.1 FFN equation):
//   gate+up: h[p, i] = bf16( SiLU(sum_c xg[p,c] Wg[e,i,c]) * sum_c xg[p,c] Wu[e,i,c] )
//   down:    Y[p, r] = sum_i h[p,i] Wd[e,r,i]
// for every row p of an active expert e's token block, fp32 accumulation (§4.2.1).
//
// How (GB300 design; the pages' AMX micro-kernel is prior art, not the blueprint):
//  * The weights are the large operand and are read exactly once per pass of tokens,
//    in their general row-major layout (§2.2; "transform I, not W", §4.1). They sit on
//    the 16-row side of the MMA ("swap AB"), the few tokens on the 8-wide side, so even
//    one token per expert runs on the tensor cores (§4.2.1: the matrix engine is used
//    for every row count, no vector-unit fallback).
//  * One persistent CTA per SM. A producer warp streams one stage of weight rows
//    (16 KB) with TMA (cp.async.bulk.tensor, evict-first L2 policy: the weights have no
//    reuse, the streaming analogue of tileloadt1 in §4.2.2) together with the stage's
//    token tiles, through a ring of mbarrier-guarded stages; consumer warps run
//    mma.sync m16n8k16 out of shared memory, one 16-row weight tile each.
//      BF16: 128 rows x 128 B (64 elements) per stage, 8 consumer warps, <= 64 tokens/pass.
//      INT8: 256 rows x 64 B (64 elements) per stage, 16 consumer warps, <= 32 tokens/pass;
//            twice the warps per weight byte, because every int8 weight is converted to
//            fp16 in registers before it reaches the tensor core. Each consumer lane reads
//            its two rows' group scales itself, so the producer issues nothing but TMA.
//  * Gate and up rows of the same intermediate index are paired inside one MMA tile
//    (tile rows 0-7 gate, 8-15 up), so the SiLU(g)*u epilogue is register-local
//    (the second layout transformation of §4.1 happens in this epilogue: h is
//    written token-major, the layout the down kernel's token tiles load). The down
//    kernel writes Y token-major (the third transformation).
//  * Work = (active expert, pass of tokens, block of output rows) x reduction stages.
//    The flattened stage range is split evenly over the CTAs (stream-K), so every SM
//    streams the same number of weight bytes whatever the routing. A unit cut by a CTA
//    boundary is finished by whichever of its CTAs arrives last (atomic counter, no
//    waiting), which sums the fp32 partials in a fixed order: results are deterministic.
//  * Shared-memory loads are bank-conflict free: BF16 tiles use the 128-byte TMA swizzle
//    with the MMA's row/column order permuted (sigma); INT8 weight rows are 64 bytes
//    apart, so the two rows a quarter-warp reads fall in different bank halves.
#pragma once

#include "moe_device.cuh"

namespace moe {
namespace stream {

constexpr int kTable = 256;          // max experts (routing limit)
constexpr int kMaxCtas = 256;        // partial-slot capacity of the workspace
constexpr int kIssueGroup = 4;       // reduction stages issued back to back per row block
constexpr int kABytes = 16384;       // weight bytes per stage
constexpr int kPartialFloats = 8192; // one CTA's partial slot (fp32)

template <bool kInt8>
struct Geometry {
  static constexpr int kConsumerWarps = kInt8 ? 16 : 8;
  static constexpr int kConsumerThreads = kConsumerWarps * 32;
  static constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
  static constexpr int kRowsA = kInt8 ? 256 : 128;        // weight rows per stage
  static constexpr int kRowBytes = kInt8 ? 64 : 128;      // bytes of each weight row per stage
  static constexpr int kK = 64;                           // reduction elements per stage
  static constexpr int kNMax = kInt8 ? 32 : 64;           // tokens per pass
  static constexpr int kNT = kNMax / 8;                   // n8 token tiles per pass
  static constexpr int kBTileBytes = 1024;                // one n8 tile: 8 rows x 64 x 2 B
  static constexpr int kBBytes = kNT * kBTileBytes;
  static constexpr int kStage = kABytes + kBBytes;
  static constexpr int kStages = kInt8 ? 10 : 8;
  static constexpr int kBarBytes = 2 * kStages * 8;
  static constexpr int kTableBytes = (4 * kTable + 32) * 4;
  static constexpr int kSmem = kStages * kStage + kBarBytes + kTableBytes;
  static_assert(kRowsA * kRowBytes == kABytes, "a stage holds 16 KB of weights");
  static_assert(kStage % 1024 == 0, "stage must keep 1024-byte alignment for the 128B swizzle");
  static_assert(kIssueGroup <= kStages, "an issue group must fit in the ring");
  static_assert(kNT * 4 * kConsumerThreads == kPartialFloats, "partial slot size");
};

struct Args {
  const int32_t* offsets;     // [E+1]
  const int32_t* active;      // [E]
  const int32_t* num_active;  // [1]
  const float* s0;            // int8 scales: gate (gate+up) or down
  const float* s1;            // int8 scales: up (gate+up only)
  void* out;                  // h bf16 [P, I] (gate+up) or Y f32 [P, H] (down)
  int64_t out_ld;
  float* partials;            // [kMaxCtas][2][kPartialFloats]
  int32_t* counters;          // [kMaxCtas], zero on entry, left zero on exit
  int32_t* status;            // workspace status word
  int rows;                   // output rows per expert: I (gate+up) or H (down)
  int K;                      // reduction length: H (gate+up) or I (down)
  int E;
  int P;                      // rows of the token block
  // INT8 only: the token tiles are fp16 copies of the bf16 rows, each row multiplied by a power
  // of two that keeps it inside fp16's range; row_scale[p] undoes that factor (exactly).
  const float* row_scale;
};

// MMA row/column g (0..7) -> row within an 8-row swizzle atom. Lanes g and g^1 share a
// quarter-warp; sigma puts them in rows whose swizzle keys differ in bit 2, so their
// 64-byte halves land on disjoint banks (BF16 tiles).
__device__ __forceinline__ int sigma(int g) { return ((g & 1) << 2) | (g >> 1); }

// Byte offset of 16-byte chunk `c` of row `r` in a tile of 128-byte rows (128B swizzle).
__device__ __forceinline__ int swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

struct Unit {
  int e, tok0, ntok, rb;
};

// One stage of MMAs for a warp: its m16 weight tile (rows rowLo / rowHi) against NT n8 token
// tiles. NT is a compile-time constant so no instruction is issued for unused token tiles.
template <bool kInt8, int NT>
__device__ __forceinline__ void stage_mma(float (&acc)[Geometry<kInt8>::kNT][4], const uint8_t* st, int rowLo,
                                          int rowHi, int brow, int t, float slo, float shi) {
  using G = Geometry<kInt8>;
  const uint8_t* sb = st + kABytes;
  if constexpr (!kInt8) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint4 alo = *reinterpret_cast<const uint4*>(st + swz(rowLo, 4 * b + t));
      const uint4 ahi = *reinterpret_cast<const uint4*>(st + swz(rowHi, 4 * b + t));
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const uint4 bv = *reinterpret_cast<const uint4*>(sb + j * G::kBTileBytes + swz(brow, 4 * b + t));
        mma_16816_bf16(acc[j], alo.x, ahi.x, alo.y, ahi.y, bv.x, bv.y);
        mma_16816_bf16(acc[j], alo.z, ahi.z, alo.w, ahi.w, bv.z, bv.w);
      }
    }
  } else {
    // 16 int8 weights per row: reduction index 16t + [0, 16) of this stage's 64; converted
    // exactly to fp16 and multiplied with the fp16 token tile (see Args::row_scale)
    const uint4 alo = *reinterpret_cast<const uint4*>(st + rowLo * 64 + t * 16);
    const uint4 ahi = *reinterpret_cast<const uint4*>(st + rowHi * 64 + t * 16);
    const uint32_t aw_lo[4] = {alo.x, alo.y, alo.z, alo.w};
    const uint32_t aw_hi[4] = {ahi.x, ahi.y, ahi.z, ahi.w};
    uint32_t a_lo_l[4], a_lo_h[4], a_hi_l[4], a_hi_h[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      int8x4_to_f16x2x2(aw_lo[s], a_lo_l[s], a_lo_h[s]);
      int8x4_to_f16x2x2(aw_hi[s], a_hi_l[s], a_hi_h[s]);
    }
    float accg[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int q = 0; q < 4; ++q) accg[j][q] = 0.0f;
      // the same 16 reduction indices of the lane's token row: 32 bytes = chunks 2t, 2t+1
      const uint8_t* tb = sb + j * G::kBTileBytes;
      const uint4 b0 = *reinterpret_cast<const uint4*>(tb + swz(brow, 2 * t));
      const uint4 b1 = *reinterpret_cast<const uint4*>(tb + swz(brow, 2 * t + 1));
      mma_16816_f16(accg[j], a_lo_l[0], a_hi_l[0], a_lo_h[0], a_hi_h[0], b0.x, b0.y);
      mma_16816_f16(accg[j], a_lo_l[1], a_hi_l[1], a_lo_h[1], a_hi_h[1], b0.z, b0.w);
      mma_16816_f16(accg[j], a_lo_l[2], a_hi_l[2], a_lo_h[2], a_hi_h[2], b1.x, b1.y);
      mma_16816_f16(accg[j], a_lo_l[3], a_hi_l[3], a_lo_h[3], a_hi_h[3], b1.z, b1.w);
    }
    // this stage is half of one 128-wide scale group: its partial sum takes the group scale
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      acc[j][0] = fmaf(slo, accg[j][0], acc[j][0]);
      acc[j][1] = fmaf(slo, accg[j][1], acc[j][1]);
      acc[j][2] = fmaf(shi, accg[j][2], acc[j][2]);
      acc[j][3] = fmaf(shi, accg[j][3], acc[j][3]);
    }
  }
}

template <bool kInt8>
__device__ __forceinline__ void stage_mma_dispatch(int nt8, float (&acc)[Geometry<kInt8>::kNT][4],
                                                   const uint8_t* st, int rowLo, int rowHi, int brow, int t,
                                                   float slo, float shi) {
  if constexpr (kInt8) {
    switch (nt8) {
      case 1: stage_mma<kInt8, 1>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
      case 2: stage_mma<kInt8, 2>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
      case 3: stage_mma<kInt8, 3>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
      default: stage_mma<kInt8, 4>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
    }
  } else {
    switch (nt8) {
      case 1: stage_mma<kInt8, 1>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
      case 2: stage_mma<kInt8, 2>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
      case 3: stage_mma<kInt8, 3>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
      case 4: stage_mma<kInt8, 4>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
      case 5: stage_mma<kInt8, 5>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
      case 6: stage_mma<kInt8, 6>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
      case 7: stage_mma<kInt8, 7>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
      default: stage_mma<kInt8, 8>(acc, st, rowLo, rowHi, brow, t, slo, shi); break;
    }
  }
}

template <bool kInt8, bool kGateUp>
__global__ void __launch_bounds__(Geometry<kInt8>::kThreads, 1)
    expert_stream_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                         const __grid_constant__ CUtensorMap tmB, const Args args) {
  using G = Geometry<kInt8>;
  constexpr int kNMax = G::kNMax;
  constexpr int kNT = G::kNT;
  constexpr int kCW = G::kConsumerWarps;
  constexpr int kCT = G::kConsumerThreads;
  constexpr int kPairRows = G::kRowsA / 2;                       // gate (or up) rows per stage
  constexpr int kRowsPerUnit = kGateUp ? kPairRows : G::kRowsA;  // output rows per unit

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::kStages * G::kStage);
  uint64_t* empty = full + G::kStages;
  int* t_e = reinterpret_cast<int*>(empty + G::kStages);
  int* t_tok0 = t_e + kTable;
  int* t_ntok = t_tok0 + kTable;
  int* t_pp = t_ntok + kTable;        // pass prefix, kTable + 1 entries
  int* s_misc = t_pp + kTable + 4;    // 8 warp sums + flags

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(&full[s], 1);  // the producer's expect_tx arrival
      mbar_init(&empty[s], kCW);
    }
    fence_mbar_init();
  }
  if (warp == kCW && lane == 0) {
    tma_prefetch_desc(&tmA0);
    if (kGateUp) tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB);
  }
  // ---- per-CTA schedule tables: active experts, their token blocks, pass prefix
  // (threads 0..255, i.e. warps 0..7, build them). They are read before waiting for the
  // preceding kernel: every kernel of this library waits for its predecessor before it lets
  // its successor start, so all work two launches back has completed, and the routing tables
  // are always at least that far back (moe_ffn_forward's gather, or moe_expert_ffn's leading
  // memset, sits in between). The token block and h are read only after the wait below.
  int A = *args.num_active;
  A = A < 0 ? 0 : (A > args.E ? args.E : A);
  int passes = 0;
  if (tid < kTable && tid < A) {
    const int e = args.active[tid];
    int tok0 = 0, ntok = 0;
    if (e >= 0 && e < args.E) {
      tok0 = args.offsets[e];
      ntok = args.offsets[e + 1] - tok0;
    }
    // an entry that does not describe rows of the token block is skipped
    if (tok0 < 0 || ntok < 0 || static_cast<int64_t>(tok0) + ntok > args.P) ntok = 0;
    t_e[tid] = e;
    t_tok0[tid] = tok0;
    t_ntok[tid] = ntok;
    passes = (ntok + kNMax - 1) / kNMax;
  }
  int incl = passes;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (tid < kTable && lane == 31) s_misc[warp] = incl;
  __syncthreads();
  if (tid < kTable) {
    int add = 0;
    for (int w = 0; w < warp; ++w) add += s_misc[w];
    t_pp[tid + 1] = incl + add;
  }
  if (tid == 0) t_pp[0] = 0;
  __syncthreads();

  const int RB = (args.rows + kRowsPerUnit - 1) / kRowsPerUnit;
  const int KI = (args.K + G::kK - 1) / G::kK;
  const int64_t W = static_cast<int64_t>(t_pp[A]) * RB * KI;  // total stages
  // Only min(grid, W) CTAs take part, so each owns at least one stage and every CTA
  // between a unit's first and last owner holds a piece of it.
  const int64_t NC = W < static_cast<int64_t>(gridDim.x) ? W : static_cast<int64_t>(gridDim.x);
  const int64_t cta = blockIdx.x;
  const int64_t it_beg = cta < NC ? cta * W / NC : 0;
  const int64_t it_end = cta < NC ? (cta + 1) * W / NC : 0;

  auto decode = [&](int64_t u) -> Unit {
    const int q = static_cast<int>(u / RB);
    Unit r;
    r.rb = static_cast<int>(u % RB);
    int lo = 0, hi = A - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (t_pp[mid] <= q) lo = mid; else hi = mid - 1;
    }
    const int np = q - t_pp[lo];
    r.e = t_e[lo];
    r.tok0 = t_tok0[lo] + np * kNMax;
    const int left = t_ntok[lo] - np * kNMax;
    r.ntok = left < kNMax ? left : kNMax;
    return r;
  };

  if (warp == kCW) {
    // =========================== producer warp ===========================
    const uint64_t policy = l2_policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    int64_t u = it_beg / KI;
    int kk0 = static_cast<int>(it_beg - u * KI);
    Unit un = it_beg < it_end ? decode(u) : Unit{};
    auto issue_a = [&](int stg, const Unit& w, int kk) {
      uint8_t* st = smem + stg * G::kStage;
      const int k0 = kk * G::kK;
      if (kGateUp) {
        tma_load_3d(st, &tmA0, &full[stg], k0, w.rb * kPairRows, w.e, policy);
        tma_load_3d(st + kPairRows * G::kRowBytes, &tmA1, &full[stg], k0, w.rb * kPairRows, w.e, policy);
      } else {
        tma_load_3d(st, &tmA0, &full[stg], k0, w.rb * G::kRowsA, w.e, policy);
      }
    };
    auto issue_b = [&](int stg, const Unit& w, int kk) {
      uint8_t* sb = smem + stg * G::kStage + kABytes;
      const int nt8 = (w.ntok + 7) >> 3;
      for (int j = 0; j < nt8; ++j) tma_load_2d(sb + j * G::kBTileBytes, &tmB, &full[stg], kk * G::kK, w.tok0 + 8 * j);
    };
    // The weights do not depend on the preceding kernel: the weight tiles of the first ring's
    // worth of stages are requested before waiting for it, their token tiles after.
    const int64_t npre = (it_end - it_beg) < G::kStages ? (it_end - it_beg) : G::kStages;
    {
      int64_t pu = u;
      int pk = kk0;
      Unit pun = un;
      for (int64_t q = 0; q < npre; ++q) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[q], kABytes + ((pun.ntok + 7) >> 3) * G::kBTileBytes);
          issue_a(static_cast<int>(q), pun, pk);
        }
        if (++pk == KI && q + 1 < npre) {
          pk = 0;
          pun = decode(++pu);
        }
      }
    }
    pdl_wait_predecessor();
    pdl_allow_successor();
    for (int64_t q = 0; q < npre; ++q) {
      if (lane == 0) issue_b(static_cast<int>(q), un, kk0);
      ++issued;
      if (++stage == G::kStages) {
        stage = 0;
        phase ^= 1;
      }
      if (++kk0 == KI) {
        kk0 = 0;
        ++u;
        if (it_beg + q + 1 < it_end) un = decode(u);
      }
    }
    for (int64_t it = it_beg + npre; it < it_end && ok;) {
      const int nt8 = (un.ntok + 7) >> 3;
      // Issue up to kIssueGroup consecutive reduction stages of the same rows back to back,
      // so each weight row is requested as one longer contiguous run.
      int64_t n = KI - kk0;
      if (n > it_end - it) n = it_end - it;
      if (n > kIssueGroup) n = kIssueGroup;
      bool drained = true;
      if (lane == 0) {
        int s = stage;
        uint32_t ph = phase;
        for (int64_t q = 0; q < n && drained; ++q) {
          drained = mbar_wait(&empty[s], ph ^ 1);
          if (++s == G::kStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      drained = __shfl_sync(0xffffffffu, drained, 0);
      if (!drained) {
        ok = false;
        break;
      }
      for (int64_t q = 0; q < n; ++q) {
        const int kk = kk0 + static_cast<int>(q);
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], kABytes + nt8 * G::kBTileBytes);
          issue_a(stage, un, kk);
          issue_b(stage, un, kk);
        }
        ++issued;
        if (++stage == G::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      it += n;
      kk0 += static_cast<int>(n);
      if (kk0 == KI && it < it_end) {
        kk0 = 0;
        ++u;
        un = decode(u);
      }
    }
    // Never leave with copies in flight: wait for the last phase issued on each stage.
    if (lane == 0) {
      const int64_t n = issued < G::kStages ? issued : G::kStages;
      int s = stage;
      uint32_t ph = phase;
      for (int64_t i = 0; i < n; ++i) {
        if (--s < 0) {
          s = G::kStages - 1;
          ph ^= 1;
        }
        if (!mbar_wait(&full[s], ph)) {
          atomicExch(args.status, kStatusDrainTimeout);
          break;
        }
      }
      if (!ok) atomicExch(args.status, kStatusWaitEmptyTimeout);
    }
    return;
  }

  // ============================ consumer warps ============================
  // the stages' token tiles, the row scales and the counters come from earlier kernels
  pdl_wait_predecessor();
  pdl_allow_successor();
  const int cw = warp;           // 0 .. kCW-1
  const int ctid = tid;          // 0 .. kCT-1
  const int g = lane >> 2;
  const int t = lane & 3;
  const int sg = kInt8 ? g : sigma(g);
  // weight rows of this warp's MMA tile (rows g / g+8 of the m16 tile)
  const int rowLo = kGateUp ? cw * 8 + sg : cw * 16 + sg;
  const int rowHi = kGateUp ? kPairRows + cw * 8 + sg : cw * 16 + 8 + sg;
  // token row of this lane's B fragment inside each n8 tile (MMA column g)
  const int brow = kInt8 ? g : sg;

  float acc[kNT][4];
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  const int64_t first_unit = it_beg / KI;
  int64_t u = first_unit;
  int kk = static_cast<int>(it_beg - u * KI);
  Unit un{};
  // INT8: this lane's two weight rows' group scales for the current unit (read straight from
  // global memory; each 32-byte sector serves eight groups, so most reads hit L1)
  const int KG = args.K / 128;
  const float* scale_lo = nullptr;
  const float* scale_hi = nullptr;
  auto scale_rows = [&]() {
    if constexpr (kInt8) {
      int glo, ghi;
      const float* blo;
      const float* bhi;
      if (kGateUp) {
        glo = ghi = un.rb * kPairRows + cw * 8 + sg;
        blo = args.s0;
        bhi = args.s1;
      } else {
        glo = un.rb * G::kRowsA + cw * 16 + sg;
        ghi = glo + 8;
        blo = bhi = args.s0;
      }
      glo = glo < args.rows ? glo : args.rows - 1;  // rows past the end are zero-filled by TMA
      ghi = ghi < args.rows ? ghi : args.rows - 1;
      scale_lo = blo + (static_cast<int64_t>(un.e) * args.rows + glo) * KG;
      scale_hi = bhi + (static_cast<int64_t>(un.e) * args.rows + ghi) * KG;
    }
  };
  if (it_beg < it_end) {
    un = decode(u);
    scale_rows();
  }
#pragma unroll
  for (int j = 0; j < kNT; ++j)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[j][q] = 0.0f;

#pragma unroll 1
  for (int64_t it = it_beg; it < it_end; ++it) {
    if (kk == 0 && it != it_beg) {  // first stage of the next unit
      ++u;
      un = decode(u);
      scale_rows();
#pragma unroll
      for (int j = 0; j < kNT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q] = 0.0f;
    }
    const int nt8 = (un.ntok + 7) >> 3;
    float slo = 1.0f, shi = 1.0f;
    if constexpr (kInt8) {  // one 128-wide scale group spans two stages
      slo = __ldg(scale_lo + (kk >> 1));
      shi = __ldg(scale_hi + (kk >> 1));
    }
    if (ok && !mbar_wait(&full[stage], phase)) {
      ok = false;
      atomicExch(args.status, kStatusWaitFullTimeout);
    }
    if (ok) stage_mma_dispatch<kInt8>(nt8, acc, smem + stage * G::kStage, rowLo, rowHi, brow, t, slo, shi);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == G::kStages) {
      stage = 0;
      phase ^= 1;
    }
    const bool piece_end = (kk == KI - 1) || (it == it_end - 1);
    if (++kk == KI) kk = 0;
    if (!piece_end) continue;

    // ---------------- end of this CTA's piece of unit u ----------------
    const int64_t ub = u * KI;
    const int64_t ue = ub + KI;
    bool finish = true;
    if (ub < it_beg || ue > it_end) {
      // unit split across CTAs: publish the fp32 partial, last arriver reduces
      auto cta_of = [&](int64_t i) -> int64_t { return ((i + 1) * NC - 1) / W; };
      const int64_t c_first = cta_of(ub);
      const int64_t c_last = cta_of(ue - 1);
      const int slot = (u == first_unit) ? 0 : 1;
      float* mine = args.partials + (cta * 2 + slot) * static_cast<int64_t>(kPartialFloats) + ctid;
#pragma unroll
      for (int j = 0; j < kNT; ++j)
        if (j < nt8)
#pragma unroll
          for (int q = 0; q < 4; ++q) mine[(j * 4 + q) * kCT] = acc[j][q];
      __threadfence();
      named_bar_sync(1, kCT);
      if (ctid == 0) {
        const int old = atomicAdd(&args.counters[c_first], 1);
        const int last = (old == static_cast<int>(c_last - c_first));
        if (last) args.counters[c_first] = 0;  // leave the counter clean for the next launch
        s_misc[8] = last;
      }
      named_bar_sync(1, kCT);
      finish = s_misc[8] != 0;
      if (finish) {
        __threadfence();
#pragma unroll
        for (int j = 0; j < kNT; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[j][q] = 0.0f;
        for (int64_t c = c_first; c <= c_last; ++c) {
          const int64_t c_first_unit = (c * W / NC) / KI;
          const int cslot = (u == c_first_unit) ? 0 : 1;
          const float* src = args.partials + (c * 2 + cslot) * static_cast<int64_t>(kPartialFloats) + ctid;
#pragma unroll
          for (int j = 0; j < kNT; ++j)
            if (j < nt8)
#pragma unroll
              for (int q = 0; q < 4; ++q) acc[j][q] += __ldcg(src + (j * 4 + q) * kCT);
        }
      }
      named_bar_sync(1, kCT);  // s_misc[8] is reused by the next piece
    }
    if (!finish) continue;

    // ---------------- epilogue ----------------
    if constexpr (kGateUp) {
      const int i = un.rb * kPairRows + cw * 8 + sg;  // intermediate index of rows g (gate) / g+8 (up)
      if (i < args.rows) {
        __nv_bfloat16* h = static_cast<__nv_bfloat16*>(args.out);
#pragma unroll
        for (int j = 0; j < kNT; ++j) {
          if (j < nt8) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int col = 2 * t + c;
              const int n = 8 * j + (kInt8 ? col : sigma(col));
              if (n < un.ntok) {
                const float rs = kInt8 ? args.row_scale[un.tok0 + n] : 1.0f;
                const float gv = acc[j][c] * rs;
                const float uv = acc[j][2 + c] * rs;
                const float silu = gv / (1.0f + expf(-gv));
                h[static_cast<int64_t>(un.tok0 + n) * args.out_ld + i] = __float2bfloat16_rn(silu * uv);
              }
            }
          }
        }
      }
    } else {
      const int r_lo = un.rb * G::kRowsA + cw * 16 + sg;
      const int r_hi = r_lo + 8;
      float* y = static_cast<float*>(args.out);
#pragma unroll
      for (int j = 0; j < kNT; ++j) {
        if (j < nt8) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int col = 2 * t + c;
            const int n = 8 * j + (kInt8 ? col : sigma(col));
            if (n < un.ntok) {
              float* yr = y + static_cast<int64_t>(un.tok0 + n) * args.out_ld;
              const float rs = kInt8 ? args.row_scale[un.tok0 + n] : 1.0f;
              if (r_lo < args.rows) yr[r_lo] = acc[j][c] * rs;
              if (r_hi < args.rows) yr[r_hi] = acc[j][2 + c] * rs;
            }
          }
        }
      }
    }
  }
}

}  // namespace stream
}  // namespace moe
