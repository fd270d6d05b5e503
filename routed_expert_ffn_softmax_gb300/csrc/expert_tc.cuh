// BF16 expert kernels on the 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM).
//
// HiNa-MoE (arXiv 2610.05123), §4.1 FFN equation with bf16 inputs and fp32 accumulation (§4.2.1):
// gate+up with SiLU(g) * u -> h (bf16), then down -> Y (fp32), over an expert-sorted token block.
// The weights stream from HBM once per pass of up to 64 tokens of an expert; one thread issues
// asynchronous MMAs that read the TMA-filled shared-memory tiles directly.
//
// Per CTA (one per SM, persistent, stream-K over (expert pass, 128-row block) x 64-element
// reduction stages; 6 warps):
//   warp 0      TMA producer: per stage the weight tile(s) (gate and up: 2 x 128 rows x 128 B;
//               down: 128 rows x 128 B) and the stage's token tile (the launch's largest pass
//               rounded up to 16 rows, at most 64, 16 at a time);
//   warp 1      owns the TMEM allocation; its lane 0 issues tcgen05.mma (M = 128, N = that tile's
//               rows, K = 16 per instruction) and commits each stage back to the producer and
//               each finished unit to the epilogue;
//   warps 2-5   epilogue: TMEM -> registers (thread = weight row), SiLU(g)*u -> h (gate+up) or
//               Y (down), or the fp32 partial of a unit that another CTA finishes.
// Accumulators are double buffered in TMEM per unit, so the epilogue of one unit overlaps the MMAs
// of the next. Gate and up of the same 128 rows go to adjacent column ranges of one buffer, so
// every epilogue thread holds g and u of the same intermediate index.
// Args, Unit and the schedule table size are shared with the INT8 pair kernels (expert_pair.cuh).
#pragma once

#include "moe_device.cuh"

namespace moe {
namespace tc {

constexpr int kEpiThreads = 128;    // warps 2..5
constexpr int kTable = 256;
constexpr int kPartialFloats = 16384;  // one INT8 pair-kernel CTA slot: 128 rows x 128 accumulator columns
constexpr int kMaxRanks = 4;           // CTAs sharing one weight block (BF16, 128- and 256-token passes)

// kN: tokens per pass (64, 128 or 256; the launch picks it from the batch's tokens per expert). An
// expert with more tokens than a pass streams its weights once per pass, so larger passes read the
// weights fewer times when experts see many tokens (prefill-sized batches); smaller passes leave room
// for more stages at decode sizes.
template <bool kGateUp, int kN = 64>
struct Geo {
  static constexpr int kThreads = 192;
  static constexpr int kNMax = kN;                          // tokens per pass
  static constexpr int kKStage = 64;                        // reduction elements per stage
  static constexpr int kWBytes = kGateUp ? 32768 : 16384;   // weight bytes per stage
  static constexpr int kBBytes = kNMax * 128;               // token tile: kN rows x 64 elements x 2 B
  static constexpr int kBoxRows = kN >= 128 ? 32 : 16;      // token rows per TMA box
  static constexpr int kStage = kWBytes + kBBytes;
  static constexpr int kTableBytes = (4 * kTable + 32) * 4;
  // as many stages as fit (down at 64-token passes: 9; measured on GB300 7: -0.4%, 9: +0.3%)
  static constexpr int kStages = (232448 - kTableBytes - 256) / kStage;
  static constexpr int kAccCols = kGateUp ? 2 * kNMax : kNMax;  // one accumulator buffer
  static constexpr int kAccBufs = 2 * kAccCols <= 512 ? 2 : 1;  // double buffered where TMEM allows
  static constexpr int kTmemCols = kAccBufs * kAccCols;
  static constexpr int kBarBytes = (2 * kStages + 5) * 8;
  static constexpr int kSmem = kStages * kStage + kBarBytes + kTableBytes;
  static constexpr int64_t kPartialSlot = 128LL * kAccCols;     // fp32 per stream-K partial slot
  static_assert(kStage % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
  static_assert(kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512, "TMEM allocations are powers of two");
  static_assert(kSmem <= 232448, "dynamic shared memory per CTA");
};

struct Args {
  const int32_t* offsets;     // [E+1]
  const int32_t* active;      // [E]
  const int32_t* num_active;  // [1]
  void* out;                  // h bf16 [P, I] (gate+up) or Y f32 [P, H] (down)
  int64_t out_ld;
  float* partials;            // [kMaxCtas][2][partial_stride]
  int64_t partial_stride;     // fp32 per partial slot (BF16: at least Geo<kGateUp, kN>::kPartialSlot)
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

// A rank's share of a round of mr tokens split over g ranks: a multiple of 16.
__device__ __forceinline__ int rank_share(int mr, int g) { return ((mr + g - 1) / g + 15) / 16 * 16; }

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

template <bool kGateUp, int kN>
__global__ void __launch_bounds__(Geo<kGateUp, kN>::kThreads, 1)
    expert_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB, const Args args) {
  using G = Geo<kGateUp, kN>;
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
      mbar_init(&acc_full[b], 1);   // MMA commit
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    if (kGateUp) tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, G::kTmemCols);

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
      g = g < static_cast<int>(gridDim.x) ? g : static_cast<int>(gridDim.x);
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
      s_misc[12] = (m + G::kBoxRows - 1) / G::kBoxRows * G::kBoxRows;
      s_misc[13] = g;
    }
  }
  __syncthreads();
  const uint32_t tmem_base = *tmem_slot;
  const int n_tile = s_misc[12];  // token rows per stage and MMA columns, 16..kNMax
  const int ranks = s_misc[13];   // CTAs per weight block
  const int span = ranks * G::kNMax;

  // Work split over columns of `ranks` CTAs (blockIdx = column * ranks + rank): the CTAs of a column
  // take the same stages of the same units, each with its rank's share of the tokens. A unit is one
  // 128-row block of one expert round (KI reduction stages).
  //  * 64-token passes (decode-sized batches): stream-K over all units, each column a contiguous
  //    range of stages; a unit split between columns is finished by the last one to arrive.
  //  * 128- and 256-token passes with at least two units per column: whole units in waves
  //    (wave w gives column c unit w * NC + c), so the columns work on neighbouring blocks of one
  //    or two experts at a time and those experts' token rows stay in L2 while the weights stream
  //    past; the last NC to 2 NC units are split stream-K as above. Contiguous ranges over every
  //    expert kept all token rows live at once and re-read them from DRAM (4x the down weights at
  //    512 tokens per expert, measured on GB300).
  const int RB = (args.rows + 127) / 128;
  const int KI = (args.K + G::kKStage - 1) / G::kKStage;
  const int64_t U = static_cast<int64_t>(t_pp[A]) * RB;
  const int64_t ncols = static_cast<int64_t>(gridDim.x) / ranks;
  const int64_t col = blockIdx.x / ranks;
  const int rank = static_cast<int>(blockIdx.x % ranks);
  const int64_t cta = blockIdx.x;
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
    const int bbytes = n_tile * 128;
    auto issue_a = [&](int stg, const Unit& w, int kk) {
      uint8_t* st = smem + stg * G::kStage;
      if (kGateUp) {
        tma_load_3d(st, &tmA0, &full[stg], kk * G::kKStage, w.rb * 128, w.e, policy);
        tma_load_3d(st + 16384, &tmA1, &full[stg], kk * G::kKStage, w.rb * 128, w.e, policy);
      } else {
        tma_load_3d(st, &tmA0, &full[stg], kk * G::kKStage, w.rb * 128, w.e, policy);
      }
    };
    auto issue_b = [&](int stg, const Unit& w, int kk) {
      uint8_t* sb_ = smem + stg * G::kStage + G::kWBytes;
      for (int j = 0; j < n_tile; j += G::kBoxRows)
        tma_load_2d(sb_ + j * 128, &tmB, &full[stg], kk * G::kKStage, w.tok0 + j);
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
          mbar_arrive_expect_tx(&full[q], G::kWBytes + bbytes);
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
      if (lane == 0) drained = mbar_wait(&empty[stage], phase ^ 1);
      drained = __shfl_sync(0xffffffffu, drained, 0);
      if (!drained) {
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[stage], G::kWBytes + bbytes);
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
    if (lane == 0) {  // never leave copies in flight
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
  } else if (warp == 1) {
    // =========================== MMA issuer ===========================
    pdl_wait_predecessor();
    pdl_allow_successor();
    if (lane == 0) {
      bool ok = true;
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t smem_base = smem_addr(smem);
      const uint32_t idesc = umma_idesc_bf16_m128(n_tile);
      for (int64_t piece = 0; piece < n_pieces; ++piece) {
        const Piece pc = piece_of(piece);
        const int b = G::kAccBufs == 2 ? static_cast<int>(piece & 1) : 0;
        for (int kk = pc.kb; kk < pc.ke; ++kk) {
          const bool first = kk == pc.kb;
          if (first && ok) {
            if (!mbar_wait(&acc_empty[b], static_cast<uint32_t>(((piece / G::kAccBufs) & 1) ^ 1))) {
              ok = false;
              atomicExch(args.status, kStatusWaitEmptyTimeout);
            }
            tc_fence_after_sync();
          }
          if (ok && !mbar_wait(&full[stage], phase)) {
            ok = false;
            atomicExch(args.status, kStatusWaitFullTimeout);
          }
          if (ok) {
            tc_fence_after_sync();
            const uint32_t st = smem_base + stage * G::kStage;
            const uint32_t d = tmem_base + b * G::kAccCols;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const uint64_t db = umma_desc_sw128(st + G::kWBytes + 32 * s);
              const bool acc = !(first && s == 0);
              umma_bf16(d, umma_desc_sw128(st + 32 * s), db, idesc, acc);
              if (kGateUp) umma_bf16(d + G::kNMax, umma_desc_sw128(st + 16384 + 32 * s), db, idesc, acc);
            }
          }
          umma_commit(&empty[stage]);  // frees the stage once these MMAs have read it
          if (++stage == G::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        umma_commit(&acc_full[b]);
      }
      // every issued MMA has finished before TMEM is released
      umma_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) atomicExch(args.status, kStatusDrainTimeout);
    }
    __syncwarp();
  } else {
    // =========================== epilogue (warps 2..5) ===========================
    pdl_wait_predecessor();
    pdl_allow_successor();
    const int etid = tid - 64;                 // 0..127
    const int quarter = warp & 3;              // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;         // weight row within the 128-row block
    bool ok = true;
    for (int64_t piece = 0; piece < n_pieces; ++piece) {
      const Piece pc = piece_of(piece);
      const Unit un = decode(pc.u);
      const int b = G::kAccBufs == 2 ? static_cast<int>(piece & 1) : 0;
      if (ok && !mbar_wait(&acc_full[b], static_cast<uint32_t>((piece / G::kAccBufs) & 1))) {
        ok = false;
        atomicExch(args.status, kStatusWaitFullTimeout);
      }
      tc_fence_after_sync();
      const int npad = ((un.ntok + 15) >> 4) * 16;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * G::kAccCols;
      const bool whole = pc.kb == 0 && pc.ke == KI;

      auto emit = [&](int n0, const float (&g)[16], const float (&v)[16]) {
        // g: gate (or down) accumulators of tokens n0..n0+15, v: up accumulators
        if constexpr (kGateUp) {
          const int i = un.rb * 128 + r;
          if (i < args.rows) {
            __nv_bfloat16* h = static_cast<__nv_bfloat16*>(args.out);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = n0 + j;
              if (n < un.ntok) {
                const float silu = g[j] / (1.0f + expf(-g[j]));
                h[static_cast<int64_t>(un.tok0 + n) * args.out_ld + i] = __float2bfloat16_rn(silu * v[j]);
              }
            }
          }
        } else {
          const int row = un.rb * 128 + r;
          if (row < args.rows) {
            float* y = static_cast<float*>(args.out);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = n0 + j;
              if (n < un.ntok) y[static_cast<int64_t>(un.tok0 + n) * args.out_ld + row] = g[j];
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
        if (kGateUp) tmem_ld16(tb + G::kNMax + n0, v);
      };

      if (whole) {
        for (int n0 = 0; n0 < npad; n0 += 16) {
          float g[16], v[16];
          load_acc(n0, g, v);
          emit(n0, g, v);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[b]);
      } else {
        // unit split across columns: publish this piece's fp32 accumulators, last arriver reduces.
        // Stage indices here count the stream-K part only (units D.. of the launch).
        const int64_t ut = pc.u - D;
        auto col_of = [&](int64_t i) -> int64_t { return ((i + 1) * NC - 1) / Wt; };
        const int64_t c_first = col_of(ut * KI);  // columns whose ranges hold this unit's stages
        const int64_t c_last = col_of(ut * KI + KI - 1);
        const int slot = piece == nW ? 0 : 1;    // a column's first stream-K piece, or its last
        float* mine = args.partials + (cta * 2 + slot) * args.partial_stride + etid;
        for (int n0 = 0; n0 < npad; n0 += 16) {
          float g[16], v[16];
          load_acc(n0, g, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            mine[(n0 + j) * kEpiThreads] = g[j];
            if (kGateUp) mine[(G::kNMax + n0 + j) * kEpiThreads] = v[j];
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[b]);  // TMEM buffer free again
        __threadfence();
        named_bar_sync(1, kEpiThreads);
        if (etid == 0) {
          int32_t* counter = &args.counters[c_first * ranks + rank];
          const int old = atomicAdd(counter, 1);
          const int last = (old == static_cast<int>(c_last - c_first));
          if (last) *counter = 0;
          s_misc[8] = last;
        }
        named_bar_sync(1, kEpiThreads);
        if (s_misc[8] != 0) {
          __threadfence();
          for (int n0 = 0; n0 < npad; n0 += 16) {
            float g[16], v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) g[j] = v[j] = 0.0f;
            for (int64_t c = c_first; c <= c_last; ++c) {
              const int64_t c_first_unit = (c * Wt / NC) / KI;
              const int cslot = (ut == c_first_unit) ? 0 : 1;
              const float* src = args.partials + ((c * ranks + rank) * 2 + cslot) * args.partial_stride + etid;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                g[j] += __ldcg(src + (n0 + j) * kEpiThreads);
                if (kGateUp) v[j] += __ldcg(src + (G::kNMax + n0 + j) * kEpiThreads);
              }
            }
            emit(n0, g, v);
          }
        }
        named_bar_sync(1, kEpiThreads);  // s_misc[8] is reused by the next piece
      }
    }
  }

  // ---- teardown: every role has finished; warp 1 releases TMEM
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, G::kTmemCols);
}

}  // namespace tc
}  // namespace moe
