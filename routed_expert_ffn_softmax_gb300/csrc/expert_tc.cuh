// Expert kernels on the 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM).
//
// Same computation, work split and outputs as the mma.sync kernels in expert_stream.cuh
// (HiNa-MoE, arXiv 2610.05123, §4.1 FFN equation; bf16 inputs, fp32 accumulation §4.2.1), but
// the per-stage MMA work of the consumer warps disappears: one thread issues asynchronous MMAs,
// so the stream is no longer limited by how fast warps can push loads and MMAs through a stage.
//
// Per CTA (one per SM, persistent, stream-K over (expert pass, 128-row block) x reduction
// stages; a stage is 128 bytes of every weight row: 64 bf16 or 128 int8 elements):
//   warp 0      TMA producer: per stage the weight tile(s) (gate and up: 2 x 128 rows x 128 B;
//               down: 128 rows x 128 B) and the stage's token tile (up to 64 rows, 16 at a time);
//   warp 1      owns the TMEM allocation; its lane 0 issues tcgen05.mma (M = 128, N = tokens of
//               the pass rounded up to 16, K = 16 per instruction) and commits each stage back to
//               the producer and each finished unit to the epilogue;
//   warps 2-5   epilogue: TMEM -> registers (thread = weight row), SiLU(g)*u -> h (gate+up) or
//               Y (down), or the fp32 partial of a unit that another CTA finishes;
//   warps 6-13  INT8 only, converters: each thread turns one weight row of the stage (128 int8 =
//               one scale group; for down each of two warps takes half a row) into exact fp16
//               values in a TMEM operand buffer, from which the MMAs read A;
//   warp 14     INT8 only, second MMA issuer (the first takes the gate rows, or the first half of
//               a down stage; the second the up rows, or the second half).
// BF16: accumulators are double buffered in TMEM per unit, so the epilogue of one unit overlaps
// the MMAs of the next. Gate and up of the same 128 rows go to adjacent column ranges of one
// buffer, so every epilogue thread holds g and u of the same intermediate index.
// INT8 (symmetric group-128 weights, §4.1 quantised variant): every stage is one scale group, so
// its MMAs write a fresh group sum into a TMEM buffer (two of them, alternating); warps 2-5
// multiply each group sum by its row's group scale and accumulate in fp32 registers, and write h
// or Y when the unit ends. The tokens are fp16 copies of the bf16 rows scaled by a per-token power
// of two (row_scale), undone in that last step; int8 -> fp16 is exact, so every product is exact
// and only the fp32 sums round.
#pragma once

#include "moe_device.cuh"

namespace moe {
namespace tc {

constexpr int kEpiThreads = 128;    // warps 2..5
constexpr int kTable = 256;
constexpr int kIssueGroup = 1;  // stages issued per producer wake-up: each as soon as its slot drains
constexpr int kPartialFloats = 16384;  // one CTA slot: 128 rows x 128 accumulator columns
constexpr int kConvWarp0 = 6;          // first INT8 converter warp
constexpr int kConvWarps = 8;
constexpr int kIssuer1Warp = kConvWarp0 + kConvWarps;  // INT8: second MMA issuer

template <bool kInt8, bool kGateUp>
struct Geo {
  static constexpr bool kGU = kGateUp;
  // INT8: two MMA issuers (gate / up, or the two halves of a down stage into two accumulators),
  // because an fp16 MMA covers half the weight bytes of a bf16 one and one issuing thread
  // cannot keep up; 32 tokens per pass keep the token tile small so five stages fit.
  static constexpr int kIssuers = kInt8 ? 2 : 1;
  static constexpr int kThreads = kInt8 ? 32 * (kIssuer1Warp + 1) : 192;
  static constexpr int kNMax = kInt8 ? 32 : 64;             // tokens per pass
  static constexpr int kKStage = kInt8 ? 128 : 64;          // reduction elements per stage
  static constexpr int kWBytes = kGateUp ? 32768 : 16384;   // weight bytes per stage
  static constexpr int kBHalf = kNMax * 128;                // token rows x 64 elements x 2 B
  static constexpr int kBBytes = kInt8 ? 2 * kBHalf : kBHalf;
  static constexpr int kStage = kWBytes + kBBytes;
  static constexpr int kStages = kInt8 ? (kGateUp ? 5 : 8) : (kGateUp ? 5 : 8);
  // one accumulator buffer: gate | up, or (INT8 down) the two issuers' partial sums; INT8 buffers
  // hold one stage's group sums
  static constexpr int kAccCols = (kGateUp || kInt8) ? 2 * kNMax : kNMax;
  static constexpr int kABase = 2 * kAccCols;                    // INT8 operand buffers start here
  static constexpr int kACols = kGateUp ? 128 : 64;              // one INT8 operand buffer
  static constexpr int kAFit = (512 - kABase) / kACols;
  static constexpr int kABufs = kInt8 ? (kAFit < kStages ? kAFit : kStages) : 0;
  static constexpr int kTmemCols = kInt8 ? 512 : 2 * kAccCols;
  static constexpr int kBarBytes = (2 * kStages + 6 + 2 * kABufs) * 8;
  static constexpr int kTableBytes = (4 * kTable + 32) * 4;
  static constexpr int kScaleLook = 4;  // INT8: group scales are fetched this many stages ahead
  static constexpr int kScaleOff = kStages * kStage + kBarBytes + kTableBytes;
  static constexpr int kScaleBytes = kInt8 ? (kScaleLook + 1) * 2 * kEpiThreads * 4 : 0;
  static constexpr int kSmem = kScaleOff + kScaleBytes;
  static_assert(kStage % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
  static_assert(kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512, "TMEM allocations are powers of two");
  static_assert(!kInt8 || (kABufs >= 2 && kABase + kABufs * kACols <= kTmemCols), "INT8 operand buffers");
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
  // INT8 only: group scales [E][rows][K/128] of gate (or down) and up, and the per-token power of
  // two that the fp16 token copy was divided by.
  const float* s0;
  const float* s1;
  const float* row_scale;
};

struct Unit {
  int e, tok0, ntok, rb;
};

// INT8 converter warps: for every stage of this CTA's range, turn this thread's weight row
// (gate+up: warps 6-9 the gate row, 10-13 the up row, all 128 bytes; down: warps 6-9 the first
// 64 bytes, 10-13 the last 64) into exact fp16 values in the next TMEM operand buffer.
template <typename G>
__device__ __forceinline__ void convert_stages(const uint8_t* smem, uint64_t* full, uint64_t* empty, uint64_t* a_full,
                                               uint64_t* a_empty, uint32_t tmem_base, const Args& args,
                                               int64_t it_beg, int64_t it_end) {
  pdl_wait_predecessor();
  pdl_allow_successor();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quarter = warp & 3;                   // TMEM lane quarter this warp may access
  const int r = quarter * 32 + lane;              // weight row within the block = TMEM lane
  const int part = (warp - kConvWarp0) >> 2;      // gate+up: gate / up; down: first / last half
  const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
  bool ok = true;
  int stage = 0;
  uint32_t phase = 0;
  int ab = 0;
  uint32_t aph = 0;
#pragma unroll 1
  for (int64_t it = it_beg; it < it_end; ++it) {
    if (ok && !mbar_wait(&a_empty[ab], aph ^ 1)) atomicExch(args.status, kStatusWaitEmptyTimeout), ok = false;
    if (ok && !mbar_wait(&full[stage], phase)) atomicExch(args.status, kStatusWaitFullTimeout), ok = false;
    ok = __all_sync(0xffffffffu, ok);  // keep the warp-wide TMEM stores uniform
    tc_fence_after_sync();
    if (ok) {
      const uint8_t* rowp = smem + stage * G::kStage + (G::kGU ? part * 16384 : 0) + r * 128;
#pragma unroll
      for (int h = 0; h < (G::kGU ? 2 : 1); ++h) {
        const int c0 = G::kGU ? 4 * h : 4 * part;  // first 16-byte chunk (128B swizzle below)
        uint32_t o[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = *reinterpret_cast<const uint4*>(rowp + (((c0 + i) ^ (r & 7)) << 4));
          int8x4_to_f16x2x2(v.x, o[8 * i + 0], o[8 * i + 1]);
          int8x4_to_f16x2x2(v.y, o[8 * i + 2], o[8 * i + 3]);
          int8x4_to_f16x2x2(v.z, o[8 * i + 4], o[8 * i + 5]);
          int8x4_to_f16x2x2(v.w, o[8 * i + 6], o[8 * i + 7]);
        }
        const int col = G::kABase + ab * G::kACols + (G::kGU ? part * 64 + 32 * h : 32 * part);
        tmem_st32(lane_base + col, o);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);  // this stage's weight bytes are consumed
    tmem_wait_st();
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&a_full[ab]);
    if (++stage == G::kStages) {
      stage = 0;
      phase ^= 1;
    }
    if (++ab == G::kABufs) {
      ab = 0;
      aph ^= 1;
    }
  }
}

// INT8 warps 2-5 (thread = weight row r of the block, TMEM lane r): for every stage, read the
// group sums the MMAs left in TMEM, multiply by the row's group scale(s) and accumulate in fp32
// registers; at the end of each unit write h = SiLU(g) * u (gate+up) or Y (down), or publish the
// partial of a unit that another CTA finishes (the last arriver reduces, in CTA order).
template <typename G, typename Decode>
__device__ __forceinline__ void promote_stages(uint8_t* smem, uint64_t* d_full, uint64_t* d_empty,
                                               uint32_t tmem_base, const Args& args, int64_t it_beg,
                                               int64_t it_end, int KI, int64_t W, int64_t NC, int* s_misc,
                                               const Decode& decode) {
  constexpr int N = G::kNMax;
  pdl_wait_predecessor();
  pdl_allow_successor();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int etid = threadIdx.x - 64;  // 0..127
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;
  const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
  const int KG = args.K / 128;
  const int64_t cta = blockIdx.x;

  // group scales travel by cp.async into a per-thread ring, kScaleLook stages ahead of use
  float* ring = reinterpret_cast<float*>(smem + G::kScaleOff) + etid;
  constexpr int kRing = G::kScaleLook + 1;
  int64_t lu = it_beg / KI;  // unit and stage of the next scale to fetch
  int lk = static_cast<int>(it_beg - lu * KI);
  const float* l0 = nullptr;
  const float* l1 = nullptr;
  int put = 0, get = 0;
  auto fetch_next = [&](int64_t stage_index) {
    if (stage_index < it_end) {
      if (l0 == nullptr || lk == 0) {
        const Unit w = decode(lu);
        int row = w.rb * 128 + r;
        row = row < args.rows ? row : args.rows - 1;  // rows past the end are zero-filled by TMA
        const int64_t off = (static_cast<int64_t>(w.e) * args.rows + row) * KG;
        l0 = args.s0 + off;
        l1 = args.s1 + off;
      }
      cp_async_4(ring + (put * 2) * kEpiThreads, l0 + lk);
      if (G::kGU) cp_async_4(ring + (put * 2 + 1) * kEpiThreads, l1 + lk);
      if (++lk == KI) {
        lk = 0;
        ++lu;
      }
    }
    cp_async_commit();  // one group per stage, empty past the end
    if (++put == kRing) put = 0;
  };
  for (int j = 0; j < G::kScaleLook; ++j) fetch_next(it_beg + j);

  float acc0[N], acc1[N];  // gate (or down) and up sums of this row for the unit's tokens
  auto zero = [&]() {
#pragma unroll
    for (int n = 0; n < N; ++n) acc0[n] = acc1[n] = 0.0f;
  };
  zero();
  bool ok = true;
  int db = 0;
  uint32_t dph = 0;
  const int64_t first_unit = it_beg / KI;
  int64_t u = first_unit;
  int kk = static_cast<int>(it_beg - u * KI);
  Unit un{};
  if (it_beg < it_end) un = decode(u);

  auto emit = [&]() {
    const int row = un.rb * 128 + r;
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
      un = decode(u);
      zero();
    }
    fetch_next(it + G::kScaleLook);
    cp_async_wait<G::kScaleLook>();
    const float s0 = ring[(get * 2) * kEpiThreads];
    const float s1 = G::kGU ? ring[(get * 2 + 1) * kEpiThreads] : 0.0f;
    if (++get == kRing) get = 0;
    if (ok && !mbar_wait(&d_full[db], dph)) atomicExch(args.status, kStatusWaitFullTimeout), ok = false;
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
          } else {  // down: the two issuers' halves of the group
            acc0[16 * c + j] = fmaf(s0, g[j] + v[j], acc0[16 * c + j]);
          }
        }
      }
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&d_empty[db]);
    if (++db == 2) {
      db = 0;
      dph ^= 1;
    }
    const bool piece_end = (kk == KI - 1) || (it == it_end - 1);
    if (++kk == KI) kk = 0;
    if (!piece_end) continue;

    // ---------------- end of this CTA's piece of unit u ----------------
    const int64_t ub = u * KI;
    const int64_t ue = ub + KI;
    if (ub >= it_beg && ue <= it_end) {
      emit();
      continue;
    }
    auto cta_of = [&](int64_t i) -> int64_t { return ((i + 1) * NC - 1) / W; };
    const int64_t c_first = cta_of(ub);
    const int64_t c_last = cta_of(ue - 1);
    const int slot = (u == first_unit) ? 0 : 1;
    float* mine = args.partials + (cta * 2 + slot) * static_cast<int64_t>(kPartialFloats) + etid;
#pragma unroll
    for (int n = 0; n < N; ++n) {
      if (n < npad) {
        mine[n * kEpiThreads] = acc0[n];
        if (G::kGU) mine[(N + n) * kEpiThreads] = acc1[n];
      }
    }
    __threadfence();
    named_bar_sync(1, kEpiThreads);
    if (etid == 0) {
      const int old = atomicAdd(&args.counters[c_first], 1);
      const int last = (old == static_cast<int>(c_last - c_first));
      if (last) args.counters[c_first] = 0;  // leave the counter clean for the next launch
      s_misc[8] = last;
    }
    named_bar_sync(1, kEpiThreads);
    if (s_misc[8] != 0) {
      __threadfence();
      zero();
      for (int64_t c = c_first; c <= c_last; ++c) {  // fixed order: the result is deterministic
        const int64_t c_first_unit = (c * W / NC) / KI;
        const int cslot = (u == c_first_unit) ? 0 : 1;
        const float* src = args.partials + (c * 2 + cslot) * static_cast<int64_t>(kPartialFloats) + etid;
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

template <bool kInt8, bool kGateUp>
__global__ void __launch_bounds__(Geo<kInt8, kGateUp>::kThreads, 1)
    expert_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB, const Args args) {
  using G = Geo<kInt8, kGateUp>;
  constexpr int kThreads = G::kThreads;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::kStages * G::kStage);
  uint64_t* empty = full + G::kStages;
  uint64_t* acc_full = empty + G::kStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2]
  uint64_t* mma_done = acc_empty + 2;       // [2] one per issuer
  uint64_t* a_full = mma_done + 2;          // [kABufs] INT8 operand buffer written (converters)
  uint64_t* a_empty = a_full + G::kABufs;   // [kABufs] INT8 operand buffer read (MMA commit)
  int* t_e = reinterpret_cast<int*>(a_empty + G::kABufs);
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
      mbar_init(&full[s], 1);                          // producer expect_tx
      mbar_init(&empty[s], G::kIssuers + (kInt8 ? kConvWarps : 0));  // MMA commits (+ converter warps)
    }
    for (int b = 0; b < G::kABufs; ++b) {
      mbar_init(&a_full[b], kConvWarps);
      mbar_init(&a_empty[b], G::kIssuers);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], G::kIssuers);  // MMA commits
      mbar_init(&acc_empty[b], 4);           // one arrival per epilogue warp
    }
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    if (kGateUp) tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, G::kTmemCols);

  // ---- schedule tables (threads 0..191 cover experts 0..191; experts 192..255 by the loop)
  // They are read before waiting for the preceding kernel: every kernel of this library waits
  // for its predecessor before it lets its successor start, so all work two launches back has
  // completed, and the routing tables are always at least that far back.
  int A = *args.num_active;
  A = A < 0 ? 0 : (A > args.E ? args.E : A);
  for (int a = tid; a < kTable; a += kThreads) {
    int passes = 0;
    if (a < A) {
      const int e = args.active[a];
      int tok0 = 0, ntok = 0;
      if (e >= 0 && e < args.E) {
        tok0 = args.offsets[e];
        ntok = args.offsets[e + 1] - tok0;
      }
      if (tok0 < 0 || ntok < 0 || static_cast<int64_t>(tok0) + ntok > args.P) ntok = 0;
      t_e[a] = e;
      t_tok0[a] = tok0;
      t_ntok[a] = ntok;
      passes = (ntok + G::kNMax - 1) / G::kNMax;
    }
    t_pp[a + 1] = passes;
  }
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
  const uint32_t tmem_base = *tmem_slot;

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
    constexpr int kHalves = kInt8 ? 2 : 1;  // 64-element halves of a stage's token tile
    auto bbytes = [](const Unit& w) { return kHalves * ((w.ntok + 15) >> 4) * 16 * 128; };
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
      const int n16 = (w.ntok + 15) >> 4;
      for (int h = 0; h < kHalves; ++h)
        for (int j = 0; j < n16; ++j)
          tma_load_2d(sb + h * G::kBHalf + j * 2048, &tmB, &full[stg], kk * G::kKStage + 64 * h, w.tok0 + 16 * j);
    };
    // weights first (they do not depend on the preceding kernel), token tiles after the wait
    const int64_t npre = (it_end - it_beg) < G::kStages ? (it_end - it_beg) : G::kStages;
    {
      int64_t pu = u;
      int pk = kk0;
      Unit pun = un;
      for (int64_t q = 0; q < npre; ++q) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[q], G::kWBytes + bbytes(pun));
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
          mbar_arrive_expect_tx(&full[stage], G::kWBytes + bbytes(un));
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
  } else if (warp == 1 || (kInt8 && warp == kIssuer1Warp)) {
    // =========================== MMA issuer(s) ===========================
    pdl_wait_predecessor();
    pdl_allow_successor();
    const int which = warp == 1 ? 0 : 1;
    if (lane == 0) {
      bool ok = true;
      int stage = 0;
      uint32_t phase = 0;
      int64_t piece = 0;
      int64_t u = it_beg / KI;
      int kk = static_cast<int>(it_beg - u * KI);
      Unit un{};
      if (it_beg < it_end) un = decode(u);
      const uint32_t smem_base = smem_addr(smem);
      int ab = 0;  // INT8 operand buffer of this stage
      uint32_t aph = 0;
      for (int64_t it = it_beg; it < it_end; ++it) {
        if (kk == 0 && it != it_beg) un = decode(++u);
        // BF16: one accumulator buffer per unit piece; INT8: one per stage (a scale group)
        const bool first = kInt8 || (it == it_beg) || (kk == 0);
        const bool last = kInt8 || (kk == KI - 1) || (it == it_end - 1);
        const int b = static_cast<int>(piece & 1);
        if (first && ok) {
          if (!mbar_wait(&acc_empty[b], static_cast<uint32_t>(((piece >> 1) & 1) ^ 1))) {
            ok = false;
            atomicExch(args.status, kStatusWaitEmptyTimeout);
          }
          tc_fence_after_sync();
        }
        // INT8: the converters arrive on a_full after they saw the stage land, so that wait also
        // covers the token tile the MMAs read
        if (!kInt8 && ok && !mbar_wait(&full[stage], phase)) {
          ok = false;
          atomicExch(args.status, kStatusWaitFullTimeout);
        }
        if (kInt8 && ok && !mbar_wait(&a_full[ab], aph)) {
          ok = false;
          atomicExch(args.status, kStatusWaitFullTimeout);
        }
        if (ok) {
          tc_fence_after_sync();
          const int npad = ((un.ntok + 15) >> 4) * 16;
          const uint32_t st = smem_base + stage * G::kStage;
          const uint32_t d = tmem_base + b * G::kAccCols;
          if constexpr (kInt8) {
            // A: the converters' fp16 rows in TMEM (column c holds elements 2c, 2c+1 of the
            // stage); B: the two 64-element halves of the fp16 token tile. Issuer 0 takes the
            // gate rows (or the first half of a down stage) into the first accumulator, issuer 1
            // the up rows (or the second half) into the second.
            const uint32_t idesc = umma_idesc_f16_m128(npad);
            const uint32_t a = tmem_base + G::kABase + ab * G::kACols + (kGateUp ? 64 * which : 0);
            const uint32_t dw = d + G::kNMax * which;
            constexpr int kSteps = kGateUp ? 8 : 4;
#pragma unroll
            for (int q = 0; q < kSteps; ++q) {
              const int s = kGateUp ? q : 4 * which + q;  // 16-element step within the stage
              const uint64_t db = umma_desc_sw128(st + G::kWBytes + (s >> 2) * G::kBHalf + 32 * (s & 3));
              umma_f16_tmem_a(dw, a + 8 * s, db, idesc, !(first && q == 0));
            }
          } else {
            const uint32_t idesc = umma_idesc_bf16_m128(npad);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const uint64_t db = umma_desc_sw128(st + G::kWBytes + 32 * s);
              const bool acc = !(first && s == 0);
              umma_bf16(d, umma_desc_sw128(st + 32 * s), db, idesc, acc);
              if (kGateUp) umma_bf16(d + G::kNMax, umma_desc_sw128(st + 16384 + 32 * s), db, idesc, acc);
            }
          }
        }
        umma_commit(&empty[stage]);  // frees the stage once these MMAs have read it
        if constexpr (kInt8) {
          umma_commit(&a_empty[ab]);  // and the operand buffer
          if (++ab == G::kABufs) {
            ab = 0;
            aph ^= 1;
          }
        }
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
      umma_commit(&mma_done[which]);
      if (!mbar_wait(&mma_done[which], 0)) atomicExch(args.status, kStatusDrainTimeout);
    }
    __syncwarp();
  } else if (warp >= kConvWarp0) {
    // =========================== INT8 converters (warps 6..13) ===========================
    if constexpr (kInt8) convert_stages<G>(smem, full, empty, a_full, a_empty, tmem_base, args, it_beg, it_end);
  } else if constexpr (kInt8) {
    // =========================== INT8 scale promotion + epilogue (warps 2..5) =================
    promote_stages<G>(smem, acc_full, acc_empty, tmem_base, args, it_beg, it_end, KI, W, NC, s_misc, decode);
  } else {
    // =========================== BF16 epilogue (warps 2..5) ===========================
    pdl_wait_predecessor();
    pdl_allow_successor();
    const int etid = tid - 64;                 // 0..127
    const int quarter = warp & 3;              // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;         // weight row within the 128-row block
    bool ok = true;
    int64_t piece = 0;
    const int64_t first_unit = it_beg / KI;
    int64_t u = first_unit;
    int kk = static_cast<int>(it_beg - u * KI);
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
