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
constexpr int kIssueGroup = 1;  // stages issued per producer wake-up: each as soon as its slot drains
constexpr int kPartialFloats = 16384;  // one CTA slot: 128 rows x 128 accumulator columns

template <bool kGateUp>
struct Geo {
  static constexpr int kThreads = 192;
  static constexpr int kNMax = 64;                          // tokens per pass
  static constexpr int kKStage = 64;                        // reduction elements per stage
  static constexpr int kWBytes = kGateUp ? 32768 : 16384;   // weight bytes per stage
  static constexpr int kBBytes = kNMax * 128;               // token tile: 64 rows x 64 elements x 2 B
  static constexpr int kStage = kWBytes + kBBytes;
  static constexpr int kStages = kGateUp ? 5 : 9;                // down: as many as fit (7: -0.4%, 9: +0.3%)
  static constexpr int kAccCols = kGateUp ? 2 * kNMax : kNMax;  // one accumulator buffer
  static constexpr int kTmemCols = 2 * kAccCols;                 // double buffered
  static constexpr int kBarBytes = (2 * kStages + 5) * 8;
  static constexpr int kTableBytes = (4 * kTable + 32) * 4;
  static constexpr int kSmem = kStages * kStage + kBarBytes + kTableBytes;
  static_assert(kStage % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
  static_assert(kTmemCols == 128 || kTmemCols == 256, "TMEM allocations are powers of two");
  static_assert(128 * kAccCols <= kPartialFloats, "partial slot size");
  static_assert(kIssueGroup <= kStages, "an issue group must fit in the ring");
  static_assert(kSmem <= 232448, "dynamic shared memory per CTA");
};

struct Args {
  const int32_t* offsets;     // [E+1]
  const int32_t* active;      // [E]
  const int32_t* num_active;  // [1]
  void* out;                  // h bf16 [P, I] (gate+up) or Y f32 [P, H] (down)
  int64_t out_ld;
  float* partials;            // [kMaxCtas][2][kPartialFloats]
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

template <bool kGateUp>
__global__ void __launch_bounds__(Geo<kGateUp>::kThreads, 1)
    expert_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB, const Args args) {
  using G = Geo<kGateUp>;
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
    // One token-tile shape for the whole launch: the largest pass's token count, rounded up to 16.
    // Every stage loads that many token rows and every MMA takes that many columns; columns past a
    // pass's own tokens meet the following rows (or TMA's zero fill) and are never read. Measured
    // on GB300, a shape per pass made stages of different passes cost different times, which the
    // equal-stage stream-K split turned into CTAs finishing apart (4-5% at 16 tokens per expert).
    int m = 16;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int a = lane * 8 + i;
      if (a < A) {
        const int n = t_ntok[a] < G::kNMax ? t_ntok[a] : G::kNMax;
        m = n > m ? n : m;
      }
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane == 0) s_misc[12] = ((m + 15) >> 4) * 16;
  }
  __syncthreads();
  const uint32_t tmem_base = *tmem_slot;
  const int n_tile = s_misc[12];  // token rows per stage and MMA columns, 16..kNMax

  const int RB = (args.rows + 127) / 128;
  const int KI = (args.K + G::kKStage - 1) / G::kKStage;
  const int64_t W = static_cast<int64_t>(t_pp[A]) * RB * KI;
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
    r.tok0 = t_tok0[lo] + np * G::kNMax;
    const int left = t_ntok[lo] - np * G::kNMax;
    r.ntok = left < G::kNMax ? left : G::kNMax;
    return r;
  };

  if (warp == 0) {
    // =========================== TMA producer ===========================
    const uint64_t policy = l2_policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    int64_t u = it_beg / KI;
    int kk0 = static_cast<int>(it_beg - u * KI);
    Unit un = it_beg < it_end ? decode(u) : Unit{};
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
      uint8_t* sb = smem + stg * G::kStage + G::kWBytes;
      for (int j = 0; j < n_tile; j += 16) tma_load_2d(sb + j * 128, &tmB, &full[stg], kk * G::kKStage, w.tok0 + j);
    };
    // weights first (they do not depend on the preceding kernel), token tiles after the wait
    const int64_t npre = (it_end - it_beg) < G::kStages ? (it_end - it_beg) : G::kStages;
    {
      int64_t pu = u;
      int pk = kk0;
      Unit pun = un;
      for (int64_t q = 0; q < npre; ++q) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[q], G::kWBytes + bbytes);
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
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], G::kWBytes + bbytes);
          issue_a(stage, un, kk0 + static_cast<int>(q));
          issue_b(stage, un, kk0 + static_cast<int>(q));
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
      int64_t piece = 0;
      int kk = static_cast<int>(it_beg % KI);
      const uint32_t smem_base = smem_addr(smem);
      const uint32_t idesc = umma_idesc_bf16_m128(n_tile);
      for (int64_t it = it_beg; it < it_end; ++it) {
        const bool first = (it == it_beg) || (kk == 0);
        const bool last = (kk == KI - 1) || (it == it_end - 1);
        const int b = static_cast<int>(piece & 1);
        if (first && ok) {
          if (!mbar_wait(&acc_empty[b], static_cast<uint32_t>(((piece >> 1) & 1) ^ 1))) {
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
        if (last) {
          umma_commit(&acc_full[b]);
          ++piece;
        }
        if (++stage == G::kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++kk == KI) kk = 0;
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
    int64_t piece = 0;
    const int64_t first_unit = it_beg / KI;
    int64_t u = first_unit;
    for (int64_t it = it_beg; it < it_end;) {
      // one piece: stages [it, pe) of unit u
      const int64_t ub = u * KI;
      const int64_t ue = ub + KI;
      const int64_t pe = ue < it_end ? ue : it_end;
      const Unit un = decode(u);
      const int b = static_cast<int>(piece & 1);
      if (ok && !mbar_wait(&acc_full[b], static_cast<uint32_t>((piece >> 1) & 1))) {
        ok = false;
        atomicExch(args.status, kStatusWaitFullTimeout);
      }
      tc_fence_after_sync();
      const int npad = ((un.ntok + 15) >> 4) * 16;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * G::kAccCols;
      const bool whole = (ub >= it_beg) && (ue <= it_end);

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
        // unit split across CTAs: publish this piece's fp32 accumulators, last arriver reduces
        auto cta_of = [&](int64_t i) -> int64_t { return ((i + 1) * NC - 1) / W; };
        const int64_t c_first = cta_of(ub);
        const int64_t c_last = cta_of(ue - 1);
        const int slot = (u == first_unit) ? 0 : 1;
        float* mine = args.partials + (cta * 2 + slot) * static_cast<int64_t>(kPartialFloats) + etid;
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
          const int old = atomicAdd(&args.counters[c_first], 1);
          const int last = (old == static_cast<int>(c_last - c_first));
          if (last) args.counters[c_first] = 0;
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
              const int64_t c_first_unit = (c * W / NC) / KI;
              const int cslot = (u == c_first_unit) ? 0 : 1;
              const float* src = args.partials + (c * 2 + cslot) * static_cast<int64_t>(kPartialFloats) + etid;
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
      ++piece;
      it = pe;
      ++u;
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
