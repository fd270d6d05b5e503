// INT8 expert kernels on CTA pairs: tcgen05.mma with cta_group::2 (M = 256 over two SMs).
//
// Same computation and outputs as the INT8 case of expert_tc.cuh (HiNa-MoE, arXiv 2610.05123, §4.1
// FFN equation with symmetric group-128 INT8 weights; fp32 accumulation §4.2.1): every stage is
// one 128-element scale group, converter warps turn each int8 weight row into exact fp16 values in
// TMEM, the MMAs write the group sums into TMEM, and promotion warps multiply them by the group
// scale and accumulate in fp32 registers. What changes is who issues the MMAs. An fp16 MMA with
// M = 128 covers only 2 KB of int8 weights, and one issuing thread pays tens of cycles per MMA and
// per barrier wait, so one SM cannot issue fast enough to keep up with its share of HBM. A pair
// MMA covers the 256 rows held by two SMs at the same issue cost, which halves the instructions and
// waits per weight byte.
//
// Work: a cluster of two CTAs (rank 0 = even, rank 1 = odd) takes a stream-K range of
// (expert pass, 256-row block) x stages; CTA `rank` holds rows 128 * rank .. 128 * rank + 127 of
// the block and token rows kN / 2 * rank .. of the pass (the pair MMA reads B half from each
// CTA's shared memory and writes each CTA's 128 rows of D into its own TMEM). Every stage has the
// same shape: the MMAs always take N = kN token columns and every CTA always loads its kN / 2 token
// rows, whatever the pass holds. Columns past the pass's tokens meet the rows that follow them (the
// next expert's tokens, or TMA's zero fill past the block) and are never read. Measured on GB300,
// stages whose shape followed the pass's token count were slower: 13% at 16 tokens per expert. A stage holds two
// 16 KB weight tiles per CTA: gate and up of one scale group (gate+up), or two consecutive scale
// groups of the down rows (down), so both kernels move the same bytes per hand-off.
// Per CTA (15 warps):
//   warp 0      TMA producer for this CTA's weight rows and token rows;
//   warps 1, 14 MMA issuers, even CTA only (gate / up, or the first / second group of a down stage),
//               committing to the barriers of both CTAs; warp 1 also allocates the pair's TMEM;
//   warps 2-5   scale promotion and epilogue for this CTA's rows;
//   warps 6-13  converters for this CTA's rows.
// Hand-offs (one issuing thread pays for every wait and commit, so the issuers have one wait and
// two commits per stage): converters of both CTAs arrive on the even CTA's operand-ready barrier,
// the even CTA's converters first waiting until both CTAs' promotion warps have freed the stage's
// accumulator buffer; the issuers' commits arrive on the same barrier in both CTAs (multicast),
// and the stage-free commit also tells the promotion warps that the stage's group sums are done.
#pragma once

#include "expert_tc.cuh"
#include "moe_device.cuh"

namespace moe {
namespace pair {

using tc::Args;
using tc::Unit;
constexpr int kTable = tc::kTable;
constexpr int kPartialFloats = tc::kPartialFloats;
constexpr int kEpiThreads = 128;   // warps 2..5
constexpr int kPromoWarp0 = 2;
constexpr int kConvWarp0 = 6;      // warps 6..13
constexpr int kConvWarps = 8;
constexpr int kIssuer1Warp = 14;
constexpr int kThreads = 32 * (kIssuer1Warp + 1);
constexpr int kScaleLook = 4;      // group scales are fetched this many stages ahead

// kN: tokens per pass (each CTA holds kN / 2 of them), 16 or 32; experts with more tokens than a
// pass take several passes. Four accumulator buffers: a stage's MMAs wait for the promotion of the
// stage four back, which loosens the per-stage chain (measured on GB300 against two and three:
// +3% at T = 256, +1% at T = 1). With 16-token passes the buffers take 128 TMEM columns and three
// operand buffers fit, with 32-token passes 256 columns and two.
// The unit list: pass np of the a-th active expert (passes t_pp[a] .. t_pp[a + 1] - 1 of the
// flattened list q) and 256-row block rb form unit q * RB + rb. A role finds its first unit with
// one division and a binary search, then steps through the list without either: a lookup per
// unit cost the single issuing thread several percent when it sat on its path.
struct Units {
  const int* e;
  const int* tok0;
  const int* ntok;
  const int* pp;  // prefix sums of the passes per active expert, A + 1 entries
  int A, RB, kN;
  struct Cursor {
    int a, np, rb;
  };
  __device__ __forceinline__ Cursor seek(int64_t u) const {
    const int q = static_cast<int>(u / RB);
    Cursor c;
    c.rb = static_cast<int>(u - static_cast<int64_t>(q) * RB);
    int lo = 0, hi = A - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pp[mid] <= q) lo = mid; else hi = mid - 1;
    }
    c.a = lo;
    c.np = q - pp[lo];
    return c;
  }
  __device__ __forceinline__ void next(Cursor& c) const {
    if (++c.rb < RB) return;
    c.rb = 0;
    ++c.np;
    while (c.a + 1 < A && c.np >= pp[c.a + 1] - pp[c.a]) {  // also skips experts without passes
      c.np = 0;
      ++c.a;
    }
  }
  __device__ __forceinline__ Unit unit(const Cursor& c) const {
    Unit r;
    r.rb = c.rb;
    r.e = e[c.a];
    r.tok0 = tok0[c.a] + c.np * kN;
    const int left = ntok[c.a] - c.np * kN;
    r.ntok = left < kN ? left : kN;
    return r;
  }
};

template <bool kGateUp, int kN>
struct Geo {
  static constexpr bool kGU = kGateUp;
  static constexpr int kNMax = kN;
  static constexpr int kDBufs = 4;                          // accumulator buffers
  static constexpr int kKStage = kGateUp ? 128 : 256;       // reduction elements per stage
  static constexpr int kWBytes = 32768;                     // this CTA's two weight tiles per stage
  static constexpr int kBRows = kNMax / 2;                  // token rows per CTA
  static constexpr int kBHalf = kBRows * 128;               // one 64-element slice of the token tile
  static constexpr int kBHalves = kKStage / 64;
  static constexpr int kBBytes = kBHalves * kBHalf;
  static constexpr int kStage = kWBytes + kBBytes;
  static constexpr int kStages = 5;
  static constexpr int kAccCols = 2 * kNMax;                // the two issuers' accumulators
  static constexpr int kABase = kDBufs * kAccCols;          // operand buffers after the accumulators
  static constexpr int kACols = 128;                        // two tiles x 128 elements (fp16 pairs)
  static constexpr int kAFit = (512 - kABase) / kACols;
  static constexpr int kABufs = kAFit < kStages ? kAFit : kStages;
  static constexpr int kBarBytes = (2 * kStages + kDBufs + 2 + 2 * kABufs) * 8;
  static constexpr int kTableBytes = (4 * kTable + 32) * 4;
  static constexpr int kScaleOff = kStages * kStage + kBarBytes + kTableBytes;
  static constexpr int kScaleBytes = (kScaleLook + 1) * 2 * kEpiThreads * 4;
  static constexpr int kSmem = kScaleOff + kScaleBytes;
  static_assert(kStage % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
  static_assert(kABufs >= 2 && kABase + kABufs * kACols <= 512, "TMEM operand buffers");
  // The stage-free barrier (shared-memory stage consumed: converters done and the stage's MMAs
  // complete) also tells the promotion warps that the stage's group sums are done; they wait on it
  // by phase parity. The converters may run kDBufs stages ahead of the promotion, so the next
  // phase of that barrier (the MMAs kStages stages later) must not be able to complete first:
  // with kDBufs > kStages the parity would alias and the promotion would wait for a phase it
  // already missed.
  static_assert(kDBufs <= kStages, "promotion may lag at most the shared-memory stages");
  static_assert(128 * kAccCols <= kPartialFloats, "partial slot size");
  static_assert(kSmem <= 232448, "dynamic shared memory per CTA");
};

// Converters: this thread's weight row of every stage -> exact fp16 in the next TMEM operand
// buffer (warps 6-9 the first tile, 10-13 the second, whole 128-byte rows); then tell the even
// CTA's issuers.
template <typename G>
__device__ __forceinline__ void convert(const uint8_t* smem, uint64_t* full, uint64_t* empty, uint64_t* a_full,
                                        uint64_t* a_empty, uint64_t* d_empty, uint32_t tmem_base, uint32_t rank,
                                        const Args& args, int64_t it_beg, int64_t it_end) {
  pdl_wait_predecessor();
  pdl_allow_successor();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quarter = warp & 3;               // TMEM lane quarter this warp may access
  const int r = quarter * 32 + lane;          // weight row within this CTA's 128 = TMEM lane
  const int part = (warp - kConvWarp0) >> 2;  // first / second tile of the stage
  const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
  bool ok = true;
  int stage = 0, ab = 0, db = 0;
  uint32_t phase = 0, aph = 0, dph = 0;
#pragma unroll 1
  for (int64_t it = it_beg; it < it_end; ++it) {
    if (ok && !mbar_wait(&a_empty[ab], aph ^ 1)) atomicExch(args.status, kStatusWaitEmptyTimeout), ok = false;
    if (ok && !mbar_wait(&full[stage], phase)) atomicExch(args.status, kStatusWaitFullTimeout), ok = false;
    ok = __all_sync(0xffffffffu, ok);  // keep the warp-wide TMEM stores uniform
    tc_fence_after_sync();
    if (ok) {
      const uint8_t* rowp = smem + stage * G::kStage + part * 16384 + r * 128;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c0 = 4 * h;  // first 16-byte chunk of this half (128B swizzle below)
        uint32_t o[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = *reinterpret_cast<const uint4*>(rowp + (((c0 + i) ^ (r & 7)) << 4));
          int8x4_to_f16x2x2(v.x, o[8 * i + 0], o[8 * i + 1]);
          int8x4_to_f16x2x2(v.y, o[8 * i + 2], o[8 * i + 3]);
          int8x4_to_f16x2x2(v.z, o[8 * i + 4], o[8 * i + 5]);
          int8x4_to_f16x2x2(v.w, o[8 * i + 6], o[8 * i + 7]);
        }
        const int col = G::kABase + ab * G::kACols + part * 64 + 32 * h;
        tmem_st32(lane_base + col, o);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);  // this stage's weight bytes are consumed
    tmem_wait_st();
    tc_fence_before_sync();
    // even CTA: the stage's accumulator buffer (last used kDBufs stages ago) must be free in both
    // CTAs before the issuers may start on it
    if (rank == 0 && lane == 0 && ok && !mbar_wait(&d_empty[db], dph ^ 1))
      atomicExch(args.status, kStatusWaitEmptyTimeout), ok = false;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (lane == 0) mbar_arrive_cta(&a_full[ab], 0);
    if (++stage == G::kStages) {
      stage = 0;
      phase ^= 1;
    }
    if (++ab == G::kABufs) {
      ab = 0;
      aph ^= 1;
    }
    if (++db == G::kDBufs) {
      db = 0;
      dph ^= 1;
    }
  }
}

// Issuers (lane 0 of warps 1 and 14 of the even CTA): pair MMAs over both CTAs' rows.
template <typename G>
__device__ __forceinline__ void issue(const uint8_t* smem, uint64_t* empty, uint64_t* a_full, uint64_t* a_empty,
                                      uint64_t* done_bar, uint32_t tmem_base, const Args& args, int64_t it_beg,
                                      int64_t it_end) {
  pdl_wait_predecessor();
  pdl_allow_successor();
  if ((threadIdx.x & 31) != 0) return;
  const int which = (threadIdx.x >> 5) == 1 ? 0 : 1;
  const uint32_t smem_base = smem_addr(smem);
  bool ok = true;
  int stage = 0, ab = 0, db = 0;
  uint32_t aph = 0;
  // issuer `which` multiplies tile `which` (gate / up, or the first / second scale group) by the
  // token tile: 8 steps of 16 elements; gate and up share the stage's 128 token columns, the two
  // down groups take columns 0..127 and 128..255
  constexpr int kSteps = 8;
  const int s0 = G::kGU ? 0 : 8 * which;
  const uint32_t a_off = G::kABase + 64 * which;
  const uint32_t idesc = umma_idesc_f16_m256(G::kNMax);
#pragma unroll 1
  for (int64_t it = it_beg; it < it_end; ++it) {
    // the converters of both CTAs arrive on a_full after they saw their stage land (so this also
    // covers both halves of the token tile), the even CTA's after the accumulator buffer was freed
    if (ok && !mbar_wait(&a_full[ab], aph)) atomicExch(args.status, kStatusWaitFullTimeout), ok = false;
    if (ok) {
      tc_fence_after_sync();
      const uint32_t a = tmem_base + a_off + ab * G::kACols;
      const uint32_t d = tmem_base + db * G::kAccCols + G::kNMax * which;
      // descriptor of the stage's token tile; each step adds its byte offset / 16
      const uint64_t bdesc = umma_desc_sw128(smem_base + stage * G::kStage + G::kWBytes);
#pragma unroll
      for (int q = 0; q < kSteps; ++q) {
        const int s = s0 + q;  // 16-element step of the token tile
        umma_f16_pair_tmem_a(d, a + 8 * q, bdesc + (((s >> 2) * G::kBHalf + 32 * (s & 3)) >> 4), idesc, q != 0);
      }
    }
    umma_commit_pair(&empty[stage]);  // both CTAs' stages are free once these MMAs have read them,
                                      // and the group sums are complete
    umma_commit_pair(&a_empty[ab]);   // and both operand buffers
    if (++stage == G::kStages) stage = 0;
    if (++ab == G::kABufs) {
      ab = 0;
      aph ^= 1;
    }
    if (++db == G::kDBufs) db = 0;
  }
  // every issued MMA has finished before the pair's TMEM is released
  umma_commit_pair(&done_bar[which]);
  if (!mbar_wait(&done_bar[which], 0)) atomicExch(args.status, kStatusDrainTimeout);
}

// Promotion and epilogue (warps 2-5, thread = row r of this CTA's 128, TMEM lane r): per stage,
// read the group sums, multiply by the row's group scale(s), accumulate in fp32 registers; at the
// end of each unit write h = SiLU(g) * u or Y, or publish the partial of a unit another pair
// finishes (the last arriver reduces, in pair order).
template <typename G>
__device__ __forceinline__ void promote(uint8_t* smem, uint64_t* empty, uint64_t* d_empty, uint32_t tmem_base,
                                        const Args& args, int64_t it_beg, int64_t it_end, int KI, int64_t W,
                                        int64_t NC, int64_t pair_id, uint32_t rank, int* s_misc,
                                        const Units& units) {
  constexpr int N = G::kNMax;
  pdl_wait_predecessor();
  pdl_allow_successor();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int etid = threadIdx.x - 32 * kPromoWarp0;  // 0..127
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;
  const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
  const int KG = args.K / 128;
  const int row_off = 128 * static_cast<int>(rank) + r;  // row within the 256-row block

  float* ring = reinterpret_cast<float*>(smem + G::kScaleOff) + etid;
  constexpr int kRing = kScaleLook + 1;
  Units::Cursor lc = units.seek(it_beg / KI);  // unit and stage of the next scale to fetch
  int lk = static_cast<int>(it_beg % KI);
  int64_t off = -1;  // the row's first scale in [E, rows, K/128] (the same in every scale array)
  int put = 0, get = 0;
  auto fetch_next = [&](int64_t stage_index) {
    if (stage_index < it_end) {
      if (off < 0 || lk == 0) {
        const Unit w = units.unit(lc);
        int row = w.rb * 256 + row_off;
        row = row < args.rows ? row : args.rows - 1;  // rows past the end are zero-filled by TMA
        off = (static_cast<int64_t>(w.e) * args.rows + row) * KG;
      }
      if constexpr (G::kGU) {  // gate and up scales of group lk (stages past KG: the residual parts')
        const bool rr = lk >= KG;
        const int g = rr ? lk - KG : lk;
        cp_async_4(ring + (put * 2) * kEpiThreads, (rr ? args.s0r : args.s0) + off + g);
        cp_async_4(ring + (put * 2 + 1) * kEpiThreads, (rr ? args.s1r : args.s1) + off + g);
      } else {  // down scales of groups 2 lk and 2 lk + 1 (none past the row's end)
        cp_async_4(ring + (put * 2) * kEpiThreads, args.s0 + off + 2 * lk);
        if (2 * lk + 1 < KG) cp_async_4(ring + (put * 2 + 1) * kEpiThreads, args.s0 + off + 2 * lk + 1);
        else ring[(put * 2 + 1) * kEpiThreads] = 0.0f;
      }
      if (++lk == KI) {
        lk = 0;
        units.next(lc);
      }
    }
    cp_async_commit();  // one group per stage, empty past the end
    if (++put == kRing) put = 0;
  };
  for (int j = 0; j < kScaleLook; ++j) fetch_next(it_beg + j);

  float acc0[N], acc1[N];  // gate (or down) and up sums of this row for the unit's tokens
  auto zero = [&]() {
#pragma unroll
    for (int n = 0; n < N; ++n) acc0[n] = acc1[n] = 0.0f;
  };
  zero();
  bool ok = true;
  int db = 0, stage = 0;
  uint32_t sph = 0;
  const int64_t first_unit = it_beg / KI;
  int64_t u = first_unit;
  int kk = static_cast<int>(it_beg - u * KI);
  Units::Cursor uc = units.seek(first_unit);
  Unit un{};
  if (it_beg < it_end) un = units.unit(uc);

  auto emit = [&]() {
    const int row = un.rb * 256 + row_off;
    if (row >= args.rows) return;
#pragma unroll
    for (int n = 0; n < N; ++n) {
      if (n < un.ntok) {
        const int64_t p = un.tok0 + n;
        const float rs = __ldg(args.row_scale + p);
        if constexpr (G::kGU) {
          const float g = acc0[n] * rs;
          const float v = acc1[n] * rs;
          const float silu = g / (1.0f + expf(-g));
          static_cast<__nv_bfloat16*>(args.out)[p * args.out_ld + row] = __float2bfloat16_rn(silu * v);
        } else {
          static_cast<float*>(args.out)[p * args.out_ld + row] = acc0[n] * rs;
        }
      }
    }
  };

#pragma unroll 1
  for (int64_t it = it_beg; it < it_end; ++it) {
    if (kk == 0 && it != it_beg) {
      ++u;
      units.next(uc);
      un = units.unit(uc);
      zero();
    }
    fetch_next(it + kScaleLook);
    cp_async_wait<kScaleLook>();
    const float s0 = ring[(get * 2) * kEpiThreads];
    const float s1 = ring[(get * 2 + 1) * kEpiThreads];
    if (++get == kRing) get = 0;
    // the issuers' stage-free commit for this stage: its MMAs, and so its group sums, are done
    if (ok && !mbar_wait(&empty[stage], sph)) atomicExch(args.status, kStatusWaitFullTimeout), ok = false;
    ok = __all_sync(0xffffffffu, ok);  // keep the warp-wide TMEM loads uniform
    tc_fence_after_sync();
    const int npad = ((un.ntok + 15) >> 4) * 16;
    const uint32_t tb = lane_base + db * G::kAccCols;
#pragma unroll
    for (int c = 0; c < N / 16; ++c) {
      if (ok && c * 16 < npad) {
        float g[16], v[16];
        tmem_ld16(tb + 16 * c, g);
        tmem_ld16(tb + N + 16 * c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if constexpr (G::kGU) {
            acc0[16 * c + j] = fmaf(s0, g[j], acc0[16 * c + j]);
            acc1[16 * c + j] = fmaf(s1, v[j], acc1[16 * c + j]);
          } else {  // down: the stage's two scale groups
            acc0[16 * c + j] = fmaf(s1, v[j], fmaf(s0, g[j], acc0[16 * c + j]));
          }
        }
      }
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive_cta(&d_empty[db], 0);
    if (++db == G::kDBufs) db = 0;
    if (++stage == G::kStages) {
      stage = 0;
      sph ^= 1;
    }
    const bool piece_end = (kk == KI - 1) || (it == it_end - 1);
    if (++kk == KI) kk = 0;
    if (!piece_end) continue;

    // ---------------- end of this pair's piece of unit u ----------------
    const int64_t ub = u * KI;
    const int64_t ue = ub + KI;
    if (ub >= it_beg && ue <= it_end) {
      emit();
      continue;
    }
    auto pair_of = [&](int64_t i) -> int64_t { return ((i + 1) * NC - 1) / W; };
    const int64_t c_first = pair_of(ub);
    const int64_t c_last = pair_of(ue - 1);
    const int slot = (u == first_unit) ? 0 : 1;
    const int64_t cta = 2 * pair_id + rank;
    float* mine = args.partials + (cta * 2 + slot) * static_cast<int64_t>(kPartialFloats) + etid;
#pragma unroll
    for (int n = 0; n < N; ++n) {
      if (n < npad) {
        mine[n * kEpiThreads] = acc0[n];
        if (G::kGU) mine[(N + n) * kEpiThreads] = acc1[n];
      }
    }
    // every thread's partial stores, then one thread's release (fence, atomic) makes them all visible
    named_bar_sync(1, kEpiThreads);
    if (etid == 0) {
      __threadfence();
      int32_t* counter = &args.counters[2 * c_first + rank];
      const int old = atomicAdd(counter, 1);
      const int last = (old == static_cast<int>(c_last - c_first));
      if (last) *counter = 0;  // leave the counter clean for the next launch
      s_misc[8] = last;
    }
    named_bar_sync(1, kEpiThreads);
    if (s_misc[8] != 0) {
      __threadfence();
      zero();
      for (int64_t c = c_first; c <= c_last; ++c) {  // fixed order: the result is deterministic
        const int64_t c_first_unit = (c * W / NC) / KI;
        const int cslot = (u == c_first_unit) ? 0 : 1;
        const float* src =
            args.partials + ((2 * c + rank) * 2 + cslot) * static_cast<int64_t>(kPartialFloats) + etid;
#pragma unroll
        for (int n = 0; n < N; ++n) {
          if (n < npad) {
            acc0[n] += __ldcg(src + n * kEpiThreads);
            if (G::kGU) acc1[n] += __ldcg(src + (N + n) * kEpiThreads);
          }
        }
      }
      emit();
    }
    named_bar_sync(1, kEpiThreads);  // s_misc[8] is reused by the next piece
  }
}

template <bool kGateUp, int kN>
__global__ void __launch_bounds__(kThreads, 1)
    expert_pair_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                       const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA0r,
                       const __grid_constant__ CUtensorMap tmA1r, const Args args) {
  using G = Geo<kGateUp, kN>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::kStages * G::kStage);
  uint64_t* empty = full + G::kStages;
  uint64_t* d_empty = empty + G::kStages; // [kDBufs] even CTA: group sums read by both CTAs
  uint64_t* mma_done = d_empty + G::kDBufs;  // [2] one per issuer
  uint64_t* a_full = mma_done + 2;        // [kABufs] even CTA: both CTAs' operands written
  uint64_t* a_empty = a_full + G::kABufs; // [kABufs] operand buffer read (issuer commits)
  int* t_e = reinterpret_cast<int*>(a_empty + G::kABufs);
  int* t_tok0 = t_e + kTable;
  int* t_ntok = t_tok0 + kTable;
  int* t_pp = t_ntok + kTable;  // kTable + 1 entries
  int* s_misc = t_pp + kTable + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_misc + 16);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_cta_rank();

  if (tid == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(&full[s], 1);              // producer expect_tx
      mbar_init(&empty[s], kConvWarps + 2);  // this CTA's converters + the two issuers' commits
    }
    for (int b = 0; b < G::kDBufs; ++b) mbar_init(&d_empty[b], 2 * 4);  // promotion warps of both CTAs
    for (int b = 0; b < 2; ++b) mbar_init(&mma_done[b], 1);
    for (int b = 0; b < G::kABufs; ++b) {
      mbar_init(&a_full[b], 2 * kConvWarps);  // converter warps of both CTAs
      mbar_init(&a_empty[b], 2);              // the two issuers' commits
    }
    fence_mbar_init();
  }
  const bool residual = kGateUp && args.kq > 0;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    if (kGateUp) tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB);
    if (residual) {
      tma_prefetch_desc(&tmA0r);
      tma_prefetch_desc(&tmA1r);
    }
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, 512);

  // schedule tables, read before waiting for the preceding kernel (see expert_tc.cuh)
  const int A = tc::load_schedule<kThreads, G::kNMax>(args, t_e, t_tok0, t_ntok, t_pp);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) {  // prefix sum of the 256 pass counts: 8 per lane, then a warp scan
    int v[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = t_pp[1 + lane * 8 + i];
      sum += v[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      run += v[i];
      t_pp[1 + lane * 8 + i] = run;
    }
    if (lane == 0) t_pp[0] = 0;
  }
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before any cross-CTA arrival
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const int RB = (args.rows + 255) / 256;
  // reduction stages of a unit: one weight part, or (residual split) W^Q then W^R
  const int KQ = (args.K + G::kKStage - 1) / G::kKStage;
  const int KI = residual ? 2 * KQ : KQ;
  const int64_t W = static_cast<int64_t>(t_pp[A]) * RB * KI;
  const int64_t pairs = gridDim.x / 2;
  const int64_t NC = W < pairs ? W : pairs;
  const int64_t pair_id = blockIdx.x / 2;
  const int64_t it_beg = pair_id < NC ? pair_id * W / NC : 0;
  const int64_t it_end = pair_id < NC ? (pair_id + 1) * W / NC : 0;

  const Units units{t_e, t_tok0, t_ntok, t_pp, A, RB, G::kNMax};

  if (warp == 0) {
    // =========================== TMA producer (this CTA's rows and token half) ==============
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      auto issue_a = [&](int stg, const Unit& w, int kk) {
        uint8_t* st = smem + stg * G::kStage;
        const int row0 = w.rb * 256 + 128 * static_cast<int>(rank);
        if (kGateUp) {
          const bool r = kk >= KQ;  // residual part
          const int x = (r ? kk - KQ : kk) * 128;
          tma_load_3d(st, r ? &tmA0r : &tmA0, &full[stg], x, row0, w.e, policy);
          tma_load_3d(st + 16384, r ? &tmA1r : &tmA1, &full[stg], x, row0, w.e, policy);
        } else {  // groups 2 kk and 2 kk + 1 (zero-filled past the row's end)
          tma_load_3d(st, &tmA0, &full[stg], kk * 256, row0, w.e, policy);
          tma_load_3d(st + 16384, &tmA0, &full[stg], kk * 256 + 128, row0, w.e, policy);
        }
      };
      auto issue_b = [&](int stg, const Unit& w, int kk) {
        uint8_t* sb = smem + stg * G::kStage + G::kWBytes;
        const int t0 = w.tok0 + G::kBRows * static_cast<int>(rank);  // this CTA's kN / 2 token rows
        const int kx = (kk < KQ ? kk : kk - KQ) * G::kKStage;  // both parts meet the same tokens
#pragma unroll
        for (int h = 0; h < G::kBHalves; ++h)
#pragma unroll
          for (int j = 0; j < G::kBRows; j += 8)
            tma_load_2d(sb + h * G::kBHalf + j * 128, &tmB, &full[stg], kx + 64 * h, t0 + j);
      };
      int kk0 = static_cast<int>(it_beg % KI);
      Units::Cursor uc = units.seek(it_beg / KI);
      Unit un = it_beg < it_end ? units.unit(uc) : Unit{};
      // The first stage's weights go out before the wait (they do not depend on the preceding
      // kernel), then its token tile, then the next stages whole. Issuing all prefetched stages'
      // weights before the first token tile let the first stage land late: the SM's share of
      // bandwidth went to all of them at once (measured on GB300: 4% slower at T = 1, 1% at
      // T = 8; the BF16 kernels measured 1% slower with this order and keep the other).
      const int64_t npre = (it_end - it_beg) < G::kStages ? (it_end - it_beg) : G::kStages;
      if (npre > 0) {
        mbar_arrive_expect_tx(&full[0], G::kWBytes + G::kBBytes);
        issue_a(0, un, kk0);
      }
      pdl_wait_predecessor();
      pdl_allow_successor();
      for (int64_t q = 0; q < npre; ++q) {
        if (q > 0) {
          mbar_arrive_expect_tx(&full[q], G::kWBytes + G::kBBytes);
          issue_a(static_cast<int>(q), un, kk0);
        }
        issue_b(static_cast<int>(q), un, kk0);
        ++issued;
        if (++stage == G::kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++kk0 == KI) {
          kk0 = 0;
          units.next(uc);
          if (it_beg + q + 1 < it_end) un = units.unit(uc);
        }
      }
      for (int64_t it = it_beg + npre; it < it_end; ++it) {
        if (!mbar_wait(&empty[stage], phase ^ 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], G::kWBytes + G::kBBytes);
        issue_a(stage, un, kk0);
        issue_b(stage, un, kk0);
        ++issued;
        if (++stage == G::kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++kk0 == KI && it + 1 < it_end) {
          kk0 = 0;
          units.next(uc);
          un = units.unit(uc);
        }
      }
      // never leave copies in flight
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
    } else {
      pdl_wait_predecessor();
      pdl_allow_successor();
    }
  } else if (warp == 1 || warp == kIssuer1Warp) {
    // =========================== MMA issuers (even CTA) ===========================
    if (rank == 0) {
      issue<G>(smem, empty, a_full, a_empty, mma_done, tmem_base, args, it_beg, it_end);
    } else {
      pdl_wait_predecessor();
      pdl_allow_successor();
    }
  } else if (warp < kConvWarp0) {
    promote<G>(smem, empty, d_empty, tmem_base, args, it_beg, it_end, KI, W, NC, pair_id, rank, s_misc, units);
  } else {
    convert<G>(smem, full, empty, a_full, a_empty, d_empty, tmem_base, rank, args, it_beg, it_end);
  }

  // ---- teardown: every role of both CTAs has finished (the even CTA's issuers have seen their
  // last MMAs complete) before the pair's TMEM is released and either CTA exits
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tmem_base, 512);
}

}  // namespace pair
}  // namespace moe
