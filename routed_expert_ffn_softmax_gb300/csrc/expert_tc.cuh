// BF16 expert kernels on the 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM).
//
// HiNa-MoE (arXiv 2610.05123), §4.1 FFN equation with bf16 inputs and fp32 accumulation (§4.2.1):
// gate+up with SiLU(g) * u -> h (bf16), then down -> Y (fp32), over an expert-sorted token block.
// The weights stream from HBM once per pass of an expert's tokens (64, 128, 192 or 256 tokens per
// pass; above 64 the passes of one expert share each weight block, see Geo and the schedule); one
// thread issues asynchronous MMAs that read the TMA-filled shared-memory tiles directly.
//
// Per CTA (persistent; decode sizes: one CTA per SM, prefill sizes: CTA pairs; units of
// (expert round, 128- or 256-row block) x 64-element reduction stages):
//   warp 0      TMA producer: per stage the weight tile(s) (gate and up: 2 x 128 rows x 128 B;
//               down: 128 rows x 128 B) and the stage's token tile (the launch's largest pass
//               share, rounded up; a pair's CTAs each load half of it);
//   warp 1      owns the TMEM allocation; its lane 0 (the even CTA's, on pairs) issues tcgen05.mma
//               (M = 128, or 256 over a pair; N = the token tile; K = 16 per instruction) and
//               commits each stage back to the producer(s) and each finished unit to the epilogue;
//   warps 2..   epilogue (4 warps, 8 on pairs): TMEM -> registers (thread = weight row), SiLU(g)*u
//               -> h (gate+up) or Y (down), or the fp32 partial of a unit that another column
//               finishes.
// Accumulators are double buffered in TMEM where two fit (gate+up and two-tile down hold one at 192-
// and 256-token passes), so the epilogue of one unit overlaps the MMAs of the next. Gate and up of the same 128 rows go to
// adjacent column ranges of one buffer, so every epilogue thread holds g and u of the same
// intermediate index.
// Args, Unit and the schedule table size are shared with the INT8 pair kernels (expert_pair.cuh).
#pragma once

#include "moe_device.cuh"

namespace moe {
namespace tc {

constexpr int kRows = 128;          // weight rows of one CTA's accumulators (TMEM lanes)
constexpr int kTable = 256;
constexpr int kPartialFloats = 16384;  // one INT8 pair-kernel CTA slot: 128 rows x 128 accumulator columns
constexpr int kMaxRanks = 8;           // passes sharing one weight block (BF16, 128- and 256-token passes)

// kN: tokens per pass (64, 128, 192 or 256; the launch picks it from the batch's tokens per expert). An
// expert with more tokens than a pass streams its weights once per pass, so larger passes read the
// weights fewer times when experts see many tokens (prefill-sized batches); smaller passes leave room
// for more stages at decode sizes.
//
// kPair: the pass runs on a CTA pair (a cluster of two) with tcgen05.mma cta_group::2, M = 256: each
// CTA holds 128 weight rows of a 256-row block and half of the pass's token rows, and the even CTA
// issues MMAs that read both CTAs' tiles and write each CTA's 128 rows into its own TMEM. Per CTA a
// stage then carries half the token bytes for the same tensor work: at prefill sizes these kernels
// are bound by the L2 -> shared-memory stream of their stages, not by DRAM (measured on GB300).
// kKind: kDown (one 128-row weight tile per stage: the plain form, which the launches no longer use),
// kGateUp (gate and up tiles of the same rows),
// kDown2 (two 128-row tiles of down per stage, on pairs: a unit is 256 rows per CTA, so a stage
// carries as many weight bytes per token byte as gate+up; down on single tiles ran its tensor pipe
// at 59% at prefill sizes, bounded by the token tile's L2 stream).
// kDownK2: down on a single CTA with two consecutive 64-element reduction slices per stage (32 KB of
// weights and two token tiles), one accumulator: on GB300, TMA copies from HBM in 16 KB stages topped
// out near 6.5 TB/s, and down at one token per expert ran at 70% of the copy rate against gate+up's 83%.
constexpr int kDown = 0, kGateUp = 1, kDown2 = 2, kDownK2 = 3;

template <int kKind, int kN = 64, bool kPair = false>
struct Geo {
  static constexpr bool kGU = kKind == kGateUp;
  static constexpr bool kTwoA = kKind == kGateUp || kKind == kDown2;  // two weight tiles, two accumulators
  static constexpr bool kTwoK = kKind == kDownK2;           // two reduction slices per stage, one accumulator
  // Epilogue warps: on pairs two per TMEM lane quarter, taking alternate groups of accumulator
  // columns, so a unit's accumulators drain in half the time (gate+up holds one accumulator buffer
  // at 256-token passes, and its MMAs wait for the drain); at 64-token passes one per quarter
  // (measured on GB300, eight cost decode batches 2-3%).
  static constexpr int kEpiWarps = kPair ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kCtas = kPair ? 2 : 1;               // CTAs per pass
  static constexpr int kUnitRows = 128 * kCtas * (kKind == kDown2 ? 2 : 1);  // weight rows per unit
  static constexpr int kSecondRows = 128 * kCtas;           // kDown2: row offset of a stage's second tile
  static constexpr int kNMax = kN;                          // tokens per pass
  static constexpr int kKStage = kTwoK ? 128 : 64;          // reduction elements per stage
  static constexpr int kWBytes = (kTwoA || kTwoK) ? 32768 : 16384;  // this CTA's weight bytes per stage
  static constexpr int kBRows = kN / kCtas;                 // this CTA's token rows per stage, at most
  static constexpr int kBSlice = kBRows * 128;              // token tile: kBRows rows x 64 elements x 2 B
  static constexpr int kBBytes = (kTwoK ? 2 : 1) * kBSlice;
  // The launch's token tile is a multiple of 16 rows per CTA. Measured on GB300, TMA moves 2 KB
  // boxes from L2 at a quarter of the rate of 16 KB ones, and fewer boxes per stage beat fewer
  // bytes: a pair loads its whole token slot (kBRows rows, rows past its share never read) as one
  // box every stage (5-7% faster at prefill sizes than the exact rows in two or three boxes); a
  // single CTA loads exactly its rows as at most three boxes of 64, 32 or 16 rows (TokenMaps;
  // against 16-row boxes +3% at 64 tokens per expert, the same elsewhere).
  static constexpr int kTileRound = 16 * kCtas;

  static constexpr int kStage = kWBytes + kBBytes;
  static constexpr int kTableBytes = (4 * kTable + 32) * 4;
  // as many stages as fit (down at 64-token passes: 9; measured on GB300 7: -0.4%, 9: +0.3%)
  static constexpr int kStages = (232448 - kTableBytes - 256) / kStage;
  static constexpr int kAccCols = kTwoA ? 2 * kNMax : kNMax;  // one accumulator buffer
  static constexpr int kAccBufs = 2 * kAccCols <= 512 ? 2 : 1;  // double buffered where TMEM allows
  static constexpr int kTmemCols = kAccBufs * kAccCols;
  static constexpr int kTmemAlloc = kTmemCols <= 128 ? 128 : (kTmemCols <= 256 ? 256 : 512);  // a power of two
  static constexpr int kBarBytes = (2 * kStages + 5) * 8;
  static constexpr int kSmem = kStages * kStage + kBarBytes + kTableBytes;
  static constexpr int64_t kPartialSlot = 128LL * kAccCols;     // fp32 per stream-K partial slot
  static_assert(kStage % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
  static_assert(kNMax % 32 == 0, "the gate+up epilogue reads 32 accumulator columns at a time");
  static_assert(kPair ? kBRows <= 256 : kBRows <= 64 + 32 + 16 + 8,
                "a pair's token slot is one box; a single CTA's rows at most three");
  static_assert(kTmemCols <= 512, "TMEM holds 512 columns");
  static_assert(kSmem <= 232448, "dynamic shared memory per CTA");
};

// Tensor maps of the token block, 64 elements wide: for a single CTA boxes of 128 >> m rows
// (m = 1..3: 64, 32, 16); for a pair m[0] has the height of its token slot.
struct TokenMaps {
  CUtensorMap m[4];
};

struct Args {
  const int32_t* offsets;     // [E+1]
  const int32_t* active;      // [E]
  const int32_t* num_active;  // [1]
  void* out;                  // h bf16 [P, I] (gate+up) or Y f32 [P, H] (down)
  int64_t out_ld;
  float* partials;            // [kMaxCtas][2][partial_stride]
  int64_t partial_stride;     // fp32 per partial slot (BF16: at least Geo<kKind, kN, kPair>::kPartialSlot)
  int32_t* counters;          // zero on entry, left zero on exit
  int32_t* status;
  int rows;                   // I (gate+up) or H (down)
  int K;                      // H (gate+up) or I (down)
  int E;
  int P;
  // INT8 (pair kernels) only: group scales [E][rows][K/128] of gate (or down) and up, and the
  // per-token power of two that the fp16 token copy was divided by.
  const float* s0;
  const float* s1;
  const float* row_scale;
  // INT8 gate+up with residual-split weights (W^Q + W^R): the scales of the residual parts, and the
  // reduction stages of one part (0 = no residual). Stages kq .. 2 kq - 1 read the residual parts
  // against the same token columns as stages 0 .. kq - 1.
  const float* s0r;
  const float* s1r;
  int kq;
  // Limit of the pipeline waits in ns (0 = kWaitLimitNs). A failure-detection test shortens it so
  // that the waits run out; only single-CTA kernels take it (a pair's copies complete on the even
  // CTA's barriers, so a pair could not drain its own copies after a short wait gave up).
  uint64_t wait_ns;
};

struct Unit {
  int e, tok0, ntok, rb;
};

// The schedule table of the active experts: expert, first token row and token count per active
// expert, and its pass count in pp[a + 1] (the caller forms the prefix sums). The active count,
// the active list and the offsets are loaded together, the offsets staged in pp (E + 1 <=
// kTable + 1 entries), so the table costs one round trip to memory instead of three dependent
// ones. Every thread of the block calls it (it synchronises the block).
template <int kThreads, int kPassTokens>
__device__ __forceinline__ int load_schedule(const Args& args, int* t_e, int* t_tok0, int* t_ntok, int* pp) {
  constexpr int kPer = (kTable + kThreads - 1) / kThreads;
  const int tid = threadIdx.x;
  int A = *args.num_active;
  int ev[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int a = tid + i * kThreads;
    ev[i] = a < args.E ? args.active[a] : -1;
  }
  for (int j = tid; j <= args.E; j += kThreads) pp[j] = args.offsets[j];
  A = A < 0 ? 0 : (A > args.E ? args.E : A);
  __syncthreads();
  int passes[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int a = tid + i * kThreads;
    passes[i] = 0;
    if (a < A) {
      const int e = ev[i];
      int tok0 = 0, ntok = 0;
      if (e >= 0 && e < args.E) {
        tok0 = pp[e];
        ntok = pp[e + 1] - tok0;
      }
      if (tok0 < 0 || ntok < 0 || static_cast<int64_t>(tok0) + ntok > args.P) ntok = 0;
      t_e[a] = e;
      t_tok0[a] = tok0;
      t_ntok[a] = ntok;
      passes[i] = (ntok + kPassTokens - 1) / kPassTokens;
    }
  }
  __syncthreads();  // every thread has read the staged offsets
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int a = tid + i * kThreads;
    if (a < kTable) pp[a + 1] = passes[i];
  }
  return A;
}

// SiLU(g) * u = g * u / (1 + e^-g), with e^-g = 2^(-g log2 e) and the reciprocal from the hardware's
// approximate instructions (PTX ex2.approx.ftz, rcp.approx.ftz: relative errors near 2^-22 and 2^-23,
// far below the bf16 rounding of h that follows). g -> -inf gives -0, g -> +inf gives g * u. The
// exact division and exponential cost the single epilogue warp per TMEM lane quarter a quarter of
// the gate+up kernel's time at prefill sizes (measured on GB300), while its MMAs wait for the
// accumulator.
__device__ __forceinline__ float silu_mul(float g, float u) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(g * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return g * r * u;
}

// 32 consecutive fp32 TMEM columns at each of two addresses of this thread's lane, one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&a)[32], float (&b)[32]) {
  uint32_t r[32], q[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta));
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]), "=r"(q[8]),
        "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]), "=r"(q[14]), "=r"(q[15]), "=r"(q[16]),
        "=r"(q[17]), "=r"(q[18]), "=r"(q[19]), "=r"(q[20]), "=r"(q[21]), "=r"(q[22]), "=r"(q[23]), "=r"(q[24]),
        "=r"(q[25]), "=r"(q[26]), "=r"(q[27]), "=r"(q[28]), "=r"(q[29]), "=r"(q[30]), "=r"(q[31])
      : "r"(tb));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(q[i]);
  }
}

// try_wait that suspends the thread for at most about hint_ns before returning false.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete; false after limit_ns. The normal limit takes
// mbar_wait's loop; a shorter one (a failure-detection test) bounds each try and checks the clock
// after every try, since a plain try_wait may suspend for microseconds by itself.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (limit_ns >= kWaitLimitNs) return mbar_wait(bar, parity);
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_hint(bar, parity, 64)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// A rank's share of a round of mr tokens split over g ranks: a multiple of 16.
__device__ __forceinline__ int rank_share(int mr, int g) { return ((mr + g - 1) / g + 15) / 16 * 16; }

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B, fp32 D, M = 256 (a CTA pair),
// N = n (a multiple of 16, each CTA holding n / 2 rows of B).
__device__ __forceinline__ uint32_t umma_idesc_bf16_m256(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (16u << 24);
}

// Pair MMA issued by the even CTA: D (+)= A * B^T, A and B from the same shared-memory offsets in
// both CTAs (each CTA's 128 rows of A, and its half of B's rows), each CTA's D rows in its TMEM.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// Shared::cluster address of the mbarrier at this offset in the pair's even CTA.
__device__ __forceinline__ uint32_t leader_barrier(uint64_t* bar) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(bar)), "r"(0));
  return remote;
}

// Tiled loads into this CTA's shared memory whose completion is counted on the even CTA's
// mbarrier (`bar`, a shared::cluster address): both CTAs' tiles of a stage complete one barrier.
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                                 int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

template <int kKind, int kN, bool kPair>
__global__ void __launch_bounds__(Geo<kKind, kN, kPair>::kThreads, 1)
    expert_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ TokenMaps tmB, const Args args) {
  using G = Geo<kKind, kN, kPair>;
  constexpr int kThreads = G::kThreads;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::kStages * G::kStage);
  uint64_t* empty = full + G::kStages;
  uint64_t* acc_full = empty + G::kStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2]
  uint64_t* mma_done = acc_empty + 2;       // [1]
  int* t_e = reinterpret_cast<int*>(mma_done + 1);
  int* t_tok0 = t_e + kTable;
  int* t_ntok = t_tok0 + kTable;
  int* t_pp = t_ntok + kTable;  // kTable + 1 entries
  int* s_misc = t_pp + kTable + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_misc + 16);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(&full[s], 1);   // producer expect_tx
      mbar_init(&empty[s], 1);  // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);              // MMA commit
      mbar_init(&acc_empty[b], G::kEpiWarps * G::kCtas);  // one arrival per epilogue warp (of both CTAs)
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    if (G::kGU) tma_prefetch_desc(&tmA1);
    for (int m = 0; m < 4; ++m) tma_prefetch_desc(&tmB.m[m]);
  }
  if (warp == 1) {
    if constexpr (kPair) tmem_alloc_pair(tmem_slot, G::kTmemAlloc);
    else tmem_alloc(tmem_slot, G::kTmemAlloc);
  }

  // ---- schedule tables. They are read before waiting for the preceding kernel: every kernel of
  // this library waits for its predecessor before it lets its successor start, so all work two
  // launches back has completed, and the routing tables are always at least that far back (a
  // standalone call begins with a memset, after which its first kernel starts only once all
  // earlier work has completed).
  const int A = load_schedule<kThreads, G::kNMax>(args, t_e, t_tok0, t_ntok, t_pp);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) {
    // Ranks per weight block: at 128- and 256-token passes (prefill-sized batches), an expert with
    // more tokens than one pass has them split evenly over g CTAs (ranks) that run the same reduction
    // stages of the same weight blocks side by side, so the weights come from HBM once and from L2
    // for the other ranks, instead of once per pass.
    int mx = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int a = lane * 8 + i;
      if (a < A) mx = t_ntok[a] > mx ? t_ntok[a] : mx;
    }
    mx = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<uint32_t>(mx)));
    int g = 1;
    if (G::kNMax >= 128) {
      g = (mx + G::kNMax - 1) / G::kNMax;
      g = g < 1 ? 1 : (g > kMaxRanks ? kMaxRanks : g);
      const int units = static_cast<int>(gridDim.x) / G::kCtas;
      g = g < units ? g : units;
    }
    const int span = g * G::kNMax;  // tokens of an expert per round
    // rounds per active expert and their prefix sum: 8 per lane, then a warp scan
    int v[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int a = lane * 8 + i;
      v[i] = a < A ? (t_ntok[a] + span - 1) / span : 0;
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
    // One token-tile shape for the whole launch: the largest rank's share, rounded up to the token
    // box. Every stage loads that many token rows and every MMA takes that many columns; columns past
    // a rank's own tokens meet the following rows (or TMA's zero fill) and are never read. Measured
    // on GB300, a shape per pass made stages of different passes cost different times, which the
    // equal-stage stream-K split turned into CTAs finishing apart (4-5% at 16 tokens per expert).
    int m = 16;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int a = lane * 8 + i;
      if (a < A) {
        const int n = rank_share(t_ntok[a] < span ? t_ntok[a] : span, g);
        m = n > m ? n : m;
      }
    }
    m = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<uint32_t>(m)));
    if (lane == 0) {
      s_misc[12] = (m + G::kTileRound - 1) / G::kTileRound * G::kTileRound;
      s_misc[13] = g;
    }
  }
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // both CTAs' barriers are initialised before any cross-CTA use
  const uint32_t tmem_base = *tmem_slot;
  const int n_tile = s_misc[12];  // MMA columns (token rows of the pass's tile), 16..kNMax
  const int b_rows = n_tile / G::kCtas;  // token rows this CTA loads per stage
  const int ranks = s_misc[13];   // CTAs per weight block
  const int span = ranks * G::kNMax;

  // Work split over columns of `ranks` passes (blockIdx = (column * ranks + rank) * kCtas + half, half
  // the CTA's place in its pair): the passes of a column take the same stages of the same units, each
  // with its rank's share of the tokens. A unit is one kUnitRows-row block of one expert round (KI
  // reduction stages).
  //  * 64-token passes (decode-sized batches): stream-K over all units, each column a contiguous
  //    range of stages; a unit split between columns is finished by the last one to arrive.
  //  * 128- and 256-token passes with at least two units per column: whole units in waves
  //    (wave w gives column c unit w * NC + c), so the columns work on neighbouring blocks of one
  //    or two experts at a time and those experts' token rows stay in L2 while the weights stream
  //    past; the last NC to 2 NC units are split stream-K as above. Contiguous ranges over every
  //    expert kept all token rows live at once and re-read them from DRAM (4x the down weights at
  //    512 tokens per expert, measured on GB300).
  const int RB = (args.rows + G::kUnitRows - 1) / G::kUnitRows;
  const int KI = (args.K + G::kKStage - 1) / G::kKStage;
  const int64_t U = static_cast<int64_t>(t_pp[A]) * RB;
  const int64_t pass_id = blockIdx.x / G::kCtas;
  const int half = kPair ? static_cast<int>(cluster_cta_rank()) : 0;
  const int64_t ncols = static_cast<int64_t>(gridDim.x / G::kCtas) / ranks;
  const int64_t col = pass_id / ranks;
  const int rank = static_cast<int>(pass_id % ranks);
  const int64_t cta = blockIdx.x;
  const bool leader = half == 0;  // issues the MMAs of a pair (every CTA when not paired)
  // pipeline waits (the drains of copies and MMAs keep kWaitLimitNs)
  const uint64_t wait_limit = (!kPair && args.wait_ns != 0) ? args.wait_ns : kWaitLimitNs;
  const bool waves = G::kNMax >= 128 && U >= 2 * ncols;
  const int64_t NC = waves ? ncols : (U * KI < ncols ? U * KI : ncols);
  const int64_t nW = (waves && col < NC) ? U / NC - 1 : 0;          // whole-unit waves of this column
  const int64_t D = waves ? (U / NC - 1) * NC : 0;                  // units done in waves
  const int64_t Wt = (U - D) * KI;                                  // stages split stream-K
  const int64_t sb = col < NC ? col * Wt / NC : 0;                  // this column's stream-K range
  const int64_t se = col < NC ? (col + 1) * Wt / NC : 0;
  const int64_t n_sk = sb < se ? (se - 1) / KI - sb / KI + 1 : 0;
  const int64_t n_pieces = nW + n_sk;
  const int64_t n_stages = nW * KI + (se - sb);

  // Piece p of this column: unit u and its stages [kb, ke).
  struct Piece {
    int64_t u;
    int kb, ke;
  };
  auto piece_of = [&](int64_t p) -> Piece {
    Piece r;
    if (p < nW) {
      r.u = p * NC + col;
      r.kb = 0;
      r.ke = KI;
    } else {
      const int64_t uf = sb / KI;
      const int64_t ut = uf + (p - nW);
      r.u = D + ut;
      r.kb = p == nW ? static_cast<int>(sb - uf * KI) : 0;
      const int64_t left = se - ut * KI;
      r.ke = left < KI ? static_cast<int>(left) : KI;
    }
    return r;
  };

  auto decode = [&](int64_t u) -> Unit {
    const int q = static_cast<int>(u / RB);
    Unit r;
    r.rb = static_cast<int>(u % RB);
    int lo = 0, hi = A - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (t_pp[mid] <= q) lo = mid; else hi = mid - 1;
    }
    const int round = q - t_pp[lo];
    r.e = t_e[lo];
    const int left = t_ntok[lo] - round * span;
    const int mr = left < span ? left : span;  // the round's tokens
    const int share = rank_share(mr, ranks);
    const int off = rank * share;
    r.tok0 = t_tok0[lo] + round * span + off;
    const int n = mr - off;
    r.ntok = n < 0 ? 0 : (n < share ? n : share);
    return r;
  };

  if (warp == 0) {
    // =========================== TMA producer ===========================
    // ranks sharing a weight block read it from L2 after the first: keep it there meanwhile
    const uint64_t policy = ranks > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    const int bbytes = kPair ? G::kBBytes : (G::kTwoK ? 2 : 1) * b_rows * 128;
    // both CTAs' bytes of a stage complete the even CTA's barrier (kCtas x this CTA's share)
    const uint32_t stage_tx = G::kCtas * (G::kWBytes + bbytes);
    auto issue_a = [&](int stg, const Unit& w, int kk) {
      uint8_t* st = smem + stg * G::kStage;
      const int row = w.rb * G::kUnitRows + half * 128;
      // the second tile: up of the same rows, or (kDown2) the down rows kSecondRows further on
      const CUtensorMap* a1 = G::kGU ? &tmA1 : &tmA0;
      const int row1 = G::kGU ? row : row + G::kSecondRows;
      if constexpr (kPair) {
        const uint32_t bar = leader_barrier(&full[stg]);
        tma_load_3d_pair(st, &tmA0, bar, kk * G::kKStage, row, w.e, policy);
        if (G::kTwoA) tma_load_3d_pair(st + 16384, a1, bar, kk * G::kKStage, row1, w.e, policy);
      } else {
        tma_load_3d(st, &tmA0, &full[stg], kk * G::kKStage, row, w.e, policy);
        if (G::kTwoA) tma_load_3d(st + 16384, a1, &full[stg], kk * G::kKStage, row1, w.e, policy);
        if (G::kTwoK) tma_load_3d(st + 16384, &tmA0, &full[stg], kk * G::kKStage + 64, row, w.e, policy);
      }
    };
    auto issue_b = [&](int stg, const Unit& w, int kk) {
      uint8_t* sb_ = smem + stg * G::kStage + G::kWBytes;
      const int r0 = w.tok0 + half * b_rows;
      if constexpr (kPair) {
        tma_load_2d_pair(sb_, &tmB.m[0], leader_barrier(&full[stg]), kk * G::kKStage, r0);
      } else {
#pragma unroll
        for (int sl = 0; sl < (G::kTwoK ? 2 : 1); ++sl) {  // each 64-element reduction slice of the stage
          int j = 0;
#pragma unroll
          for (int m = 1; m < 4; ++m) {  // b_rows (a multiple of 16, at most 64) as a sum of box heights
            if (b_rows - j >= (128 >> m)) {
              tma_load_2d(sb_ + sl * G::kBSlice + j * 128, &tmB.m[m], &full[stg], kk * G::kKStage + 64 * sl, r0 + j);
              j += 128 >> m;
            }
          }
        }
      }
    };
    // cursor over this column's stages: piece, its stage range and unit
    struct Cursor {
      int64_t p;
      Piece pc;
      int kk;
      Unit un;
    };
    auto start = [&](Cursor& c) {
      c.p = 0;
      if (n_pieces > 0) {
        c.pc = piece_of(0);
        c.kk = c.pc.kb;
        c.un = decode(c.pc.u);
      }
    };
    auto advance = [&](Cursor& c) {
      if (++c.kk == c.pc.ke && ++c.p < n_pieces) {
        c.pc = piece_of(c.p);
        c.kk = c.pc.kb;
        c.un = decode(c.pc.u);
      }
    };
    // weights first (they do not depend on the preceding kernel), token tiles after the wait
    const int64_t npre = n_stages < G::kStages ? n_stages : G::kStages;
    Cursor cur;
    start(cur);
    {
      Cursor pre = cur;
      for (int64_t q = 0; q < npre; ++q) {
        if (lane == 0) {
          if (leader) mbar_arrive_expect_tx(&full[q], stage_tx);
          issue_a(static_cast<int>(q), pre.un, pre.kk);
        }
        if (q + 1 < npre) advance(pre);
      }
    }
    pdl_wait_predecessor();
    pdl_allow_successor();
    for (int64_t q = 0; q < npre; ++q) {
      if (lane == 0) issue_b(static_cast<int>(q), cur.un, cur.kk);
      ++issued;
      if (++stage == G::kStages) {
        stage = 0;
        phase ^= 1;
      }
      if (issued < n_stages) advance(cur);
    }
    for (int64_t i = npre; i < n_stages; ++i) {
      bool drained = true;
      if (lane == 0) drained = mbar_wait_for(&empty[stage], phase ^ 1, wait_limit);
      drained = __shfl_sync(0xffffffffu, drained, 0);
      if (!drained) {
        ok = false;
        break;
      }
      if (lane == 0) {
        if (leader) mbar_arrive_expect_tx(&full[stage], stage_tx);
        issue_a(stage, cur.un, cur.kk);
        issue_b(stage, cur.un, cur.kk);
      }
      ++issued;
      if (++stage == G::kStages) {
        stage = 0;
        phase ^= 1;
      }
      if (i + 1 < n_stages) advance(cur);
    }
    // never leave copies in flight: the even CTA's barriers count both CTAs' copies (the odd CTA's
    // are covered by the cluster barrier before exit, which the even CTA reaches after this)
    if (lane == 0 && leader) {
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
    }
    if (lane == 0 && !ok) atomicExch(args.status, kStatusWaitEmptyTimeout);
  } else if (warp == 1) {
    // =========================== MMA issuer ===========================
    pdl_wait_predecessor();
    pdl_allow_successor();
    if (lane == 0 && leader) {
      bool ok = true;
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t smem_base = smem_addr(smem);
      const uint32_t idesc = kPair ? umma_idesc_bf16_m256(n_tile) : umma_idesc_bf16_m128(n_tile);
      auto mma = [&](uint32_t d, uint64_t a, uint64_t b_, bool acc) {
        if constexpr (kPair) umma_bf16_pair(d, a, b_, idesc, acc);
        else umma_bf16(d, a, b_, idesc, acc);
      };
      auto commit = [&](uint64_t* bar) {  // arrives in both CTAs of a pair
        if constexpr (kPair) umma_commit_pair(bar);
        else umma_commit(bar);
      };
      // A wait that gives up stops the issuer for good: a stage it has not seen full is never handed
      // back, so the producer cannot re-arm a stage whose copies are still in flight (its own wait for
      // that stage then runs out, and it drains the copies it issued).
      for (int64_t piece = 0; piece < n_pieces && ok; ++piece) {
        const Piece pc = piece_of(piece);
        const int b = G::kAccBufs == 2 ? static_cast<int>(piece & 1) : 0;
        for (int kk = pc.kb; kk < pc.ke; ++kk) {
          const bool first = kk == pc.kb;
          if (first) {
            if (!mbar_wait_for(&acc_empty[b], static_cast<uint32_t>(((piece / G::kAccBufs) & 1) ^ 1), wait_limit)) {
              ok = false;
              atomicExch(args.status, kStatusWaitEmptyTimeout);
              break;
            }
            tc_fence_after_sync();
          }
          if (!mbar_wait_for(&full[stage], phase, wait_limit)) {
            ok = false;
            atomicExch(args.status, kStatusWaitFullTimeout);
            break;
          }
          tc_fence_after_sync();
          const uint32_t st = smem_base + stage * G::kStage;
          const uint32_t d = tmem_base + b * G::kAccCols;
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint64_t db = umma_desc_sw128(st + G::kWBytes + 32 * s);
            const bool acc = !(first && s == 0);
            mma(d, umma_desc_sw128(st + 32 * s), db, acc);
            if (G::kTwoA) mma(d + G::kNMax, umma_desc_sw128(st + 16384 + 32 * s), db, acc);
          }
          if constexpr (G::kTwoK) {  // the stage's second reduction slice, into the same accumulator
#pragma unroll
            for (int s = 0; s < 4; ++s)
              mma(d, umma_desc_sw128(st + 16384 + 32 * s), umma_desc_sw128(st + G::kWBytes + G::kBSlice + 32 * s), true);
          }
          commit(&empty[stage]);  // frees the stage (of both CTAs) once these MMAs have read it
          if (++stage == G::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) commit(&acc_full[b]);
      }
      // every issued MMA has finished before TMEM is released
      commit(mma_done);
      if (!mbar_wait(mma_done, 0)) atomicExch(args.status, kStatusDrainTimeout);
    }
    __syncwarp();
  } else {
    // =========================== epilogue (warps 2..9) ===========================
    pdl_wait_predecessor();
    pdl_allow_successor();
    const int ew = warp - 2;                   // epilogue warp 0..7
    const int quarter = warp & 3;              // TMEM lane quarter this warp may access
    const int ch = ew >> 2;                    // which of the warps of its quarter
    constexpr int kPerQuarter = G::kEpiWarps / 4;
    const int r = quarter * 32 + lane;         // weight row within the CTA's 128 rows
    constexpr int kEpiThreads = G::kEpiWarps * 32;
    bool ok = true;
    // the accumulator buffer is free again: tell the CTA that issues the MMAs
    auto release_acc = [&](uint64_t* bar) {
      if (kPair && !leader) mbar_arrive_cta(bar, 0);
      else mbar_arrive(bar);
    };
    for (int64_t piece = 0; piece < n_pieces; ++piece) {
      const Piece pc = piece_of(piece);
      const Unit un = decode(pc.u);
      const int b = G::kAccBufs == 2 ? static_cast<int>(piece & 1) : 0;
      if (ok && !mbar_wait_for(&acc_full[b], static_cast<uint32_t>((piece / G::kAccBufs) & 1), wait_limit)) {
        ok = false;
        atomicExch(args.status, kStatusWaitFullTimeout);
      }
      tc_fence_after_sync();
      const int npad = ((un.ntok + 15) >> 4) * 16;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * G::kAccCols;
      const bool whole = pc.kb == 0 && pc.ke == KI;

      auto emit = [&](int n0, const float (&g)[16], const float (&v)[16]) {
        // g: gate (or down) accumulators of tokens n0..n0+15, v: up (or the second down tile's)
        if constexpr (G::kGU) {
          // Lanes 2k and 2k + 1 hold rows i and i + 1 (rows is a multiple of 8): for every two tokens
          // one shuffle lets the even lane store both rows of the first token and the odd lane both
          // rows of the second, as 4-byte words (a warp's 32 rows of a token are 64 bytes, so 2-byte
          // stores left half of each store slot empty; 3-5% per prefill step on GB300).
          const int i = un.rb * G::kUnitRows + half * 128 + r;
          const bool odd = (lane & 1) != 0;
          uint32_t* hp = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(args.out) +
                                                     (static_cast<int64_t>(un.tok0 + n0 + (odd ? 1 : 0)) * args.out_ld +
                                                      (i & ~1)));
          const int nmax = un.ntok - n0;
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const uint32_t a0 = __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul(g[j], v[j])));
            const uint32_t a1 = __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul(g[j + 1], v[j + 1])));
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? a0 : a1, 1);
            const uint32_t word = odd ? (recv | (a1 << 16)) : (a0 | (recv << 16));
            if (i < args.rows && (odd ? j + 1 : j) < nmax) *hp = word;
            hp += args.out_ld;  // two tokens: out_ld words of two bf16
          }
        } else {
          float* y = static_cast<float*>(args.out);
          const int row = un.rb * G::kUnitRows + half * 128 + r;
          if (row < args.rows) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = n0 + j;
              if (n < un.ntok) y[static_cast<int64_t>(un.tok0 + n) * args.out_ld + row] = g[j];
            }
          }
          if constexpr (kKind == kDown2) {
            const int row2 = row + G::kSecondRows;
            if (row2 < args.rows) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = n0 + j;
                if (n < un.ntok) y[static_cast<int64_t>(un.tok0 + n) * args.out_ld + row2] = v[j];
              }
            }
          }
        }
      };

      // accumulators of tokens n0..n0+15: g = gate (or down), v = up
      auto load_acc = [&](int n0, float (&g)[16], float (&v)[16]) {
        if (!ok) {
#pragma unroll
          for (int j = 0; j < 16; ++j) g[j] = v[j] = 0.0f;
          return;
        }
        tmem_ld16(tb + n0, g);
        if (G::kTwoA) tmem_ld16(tb + G::kNMax + n0, v);
      };

      if (whole) {
        // 32 tokens per TMEM round trip, the two warps of a quarter alternating (columns past npad,
        // up to kNMax, are read and not stored)
        for (int n0 = 32 * ch; n0 < npad; n0 += 32 * kPerQuarter) {
          float g[32], v[32];
          if (!ok) {
#pragma unroll
            for (int j = 0; j < 32; ++j) g[j] = v[j] = 0.0f;
          } else if constexpr (G::kTwoA) {
            tmem_ld32x2(tb + n0, tb + G::kNMax + n0, g, v);
          } else {
            tmem_ld32(tb + n0, g);
          }
          emit(n0, reinterpret_cast<const float(&)[16]>(g[0]), reinterpret_cast<const float(&)[16]>(v[0]));
          emit(n0 + 16, reinterpret_cast<const float(&)[16]>(g[16]), reinterpret_cast<const float(&)[16]>(v[16]));
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) release_acc(&acc_empty[b]);
      } else {
        // unit split across columns: publish this piece's fp32 accumulators, last arriver reduces.
        // Stage indices here count the stream-K part only (units D.. of the launch).
        const int64_t ut = pc.u - D;
        auto col_of = [&](int64_t i) -> int64_t { return ((i + 1) * NC - 1) / Wt; };
        const int64_t c_first = col_of(ut * KI);  // columns whose ranges hold this unit's stages
        const int64_t c_last = col_of(ut * KI + KI - 1);
        const int slot = piece == nW ? 0 : 1;    // a column's first stream-K piece, or its last
        float* mine = args.partials + (cta * 2 + slot) * args.partial_stride + r;
        for (int n0 = 16 * ch; n0 < npad; n0 += 16 * kPerQuarter) {
          float g[16], v[16];
          load_acc(n0, g, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            mine[(n0 + j) * kRows] = g[j];
            if (G::kTwoA) mine[(G::kNMax + n0 + j) * kRows] = v[j];
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) release_acc(&acc_empty[b]);  // TMEM buffer free again
        // every thread's partial stores, then one thread's release (fence, atomic) makes them all visible
        named_bar_sync(1, kEpiThreads);
        if (ew == 0 && lane == 0) {
          __threadfence();
          int32_t* counter = &args.counters[(c_first * ranks + rank) * G::kCtas + half];
          const int old = atomicAdd(counter, 1);
          const int last = (old == static_cast<int>(c_last - c_first));
          if (last) *counter = 0;
          s_misc[8] = last;
        }
        named_bar_sync(1, kEpiThreads);
        if (s_misc[8] != 0) {
          __threadfence();
          for (int n0 = 16 * ch; n0 < npad; n0 += 16 * kPerQuarter) {
            float g[16], v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) g[j] = v[j] = 0.0f;
            for (int64_t c = c_first; c <= c_last; ++c) {
              const int64_t c_first_unit = (c * Wt / NC) / KI;
              const int cslot = (ut == c_first_unit) ? 0 : 1;
              const int64_t src_cta = (c * ranks + rank) * G::kCtas + half;
              const float* src = args.partials + (src_cta * 2 + cslot) * args.partial_stride + r;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                g[j] += __ldcg(src + (n0 + j) * kRows);
                if (G::kTwoA) v[j] += __ldcg(src + (G::kNMax + n0 + j) * kRows);
              }
            }
            emit(n0, g, v);
          }
        }
        named_bar_sync(1, kEpiThreads);  // s_misc[8] is reused by the next piece
      }
    }
  }

  // ---- teardown: every role has finished (of both CTAs of a pair: the even CTA's issuer has seen its
  // last MMAs complete and no copy or arrival targets either CTA any more); warp 1 releases TMEM
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after_sync();
  if (warp == 1) {
    if constexpr (kPair) tmem_dealloc_pair(tmem_base, G::kTmemAlloc);
    else tmem_dealloc(tmem_base, G::kTmemAlloc);
  }
}

}  // namespace tc
}  // namespace moe
