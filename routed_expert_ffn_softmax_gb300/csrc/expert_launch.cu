// Host side of the expert kernels: TMA descriptors and launches (BF16: expert_tc.cuh on single
// CTAs; INT8: expert_pair.cuh on CTA pairs, after an fp16 copy of the token rows).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "expert_pair.cuh"
#include "expert_tc.cuh"
#include "moe_launch.h"

namespace moe {

TensorMapEncodeFn tensor_map_encoder() {
  static TensorMapEncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TensorMapEncodeFn>(p);
  });
  return fn;
}

// Weights of all experts as a 3-D tensor {K (contiguous), rows, E}; box = one stage's 128 bytes of
// `box_rows` rows of one expert (64 bf16 or 128 int8 elements, one INT8 scale group), with the
// 128-byte swizzle the MMA descriptors and the converters expect.
bool encode_weights(CUtensorMap* map, const void* W, bool int8, int K, int rows, int E, int box_rows) {
  const cuuint64_t eb = int8 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(E)};
  cuuint64_t strides[2] = {K * eb, static_cast<cuuint64_t>(K) * rows * eb};
  cuuint32_t box[3] = {int8 ? 128u : 64u, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = tensor_map_encoder()(map, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                    const_cast<void*>(W), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                    CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// Token block {K (contiguous), P rows} bf16 or fp16; box = 64 elements x `box_rows` rows;
// 128-byte swizzle.
bool encode_tokens(CUtensorMap* map, const void* X, int K, int P, bool fp16 = false, int box_rows = 8) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(P)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = tensor_map_encoder()(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                    const_cast<void*>(X), dims, strides,
                                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp16 copy of bf16 rows for the INT8 path: each row is multiplied by 2^-k, with k chosen so that
// its largest magnitude lands in [2^14, 2^15) (inside fp16's range, k clamped to [-100, 127]),
// and row_scale[p] = 2^k restores it after the MMA. Every value within 2^-31 of the row's
// largest keeps its bf16 bits exactly in fp16; smaller ones round to fp16's subnormal grid.
// With src_rows, output row p is source row src_rows[p]: the token gather and the fp16 copy in
// one pass (the forward path's INT8 gather).
constexpr int kRowThreads = 256;

__global__ void __launch_bounds__(kRowThreads)
    rows_to_f16_kernel(const uint4* __restrict__ src, int K8, int64_t P, uint4* __restrict__ dst,
                       float* __restrict__ row_scale, const int32_t* __restrict__ src_rows,
                       int64_t src_prefetch_bytes) {
  __shared__ float s_max[kRowThreads / 32];
  prefetch_l2_grid(src, src_prefetch_bytes);
  pdl_wait_predecessor();
  pdl_allow_successor();
  const int tid = threadIdx.x;
  for (int64_t p = blockIdx.x; p < P; p += gridDim.x) {
    const uint4* s4 = src + (src_rows != nullptr ? static_cast<int64_t>(src_rows[p]) : p) * K8;
    float m = 0.0f;
    for (int c = tid; c < K8; c += kRowThreads) {
      const uint4 v = s4[c];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
        m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xffff0000u)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0) s_max[tid >> 5] = m;
    __syncthreads();
    m = s_max[0];
#pragma unroll
    for (int i = 1; i < kRowThreads / 32; ++i) m = fmaxf(m, s_max[i]);
    int k = 0;
    if (m > 0.0f && m <= 3.0e38f) {
      int e = 0;
      frexpf(m, &e);  // m = f * 2^e, 0.5 <= f < 1
      k = e - 15;
      k = k < -100 ? -100 : (k > 127 ? 127 : k);
    }
    const float down = ldexpf(1.0f, -k);
    uint4* d4 = dst + p * K8;
    for (int c = tid; c < K8; c += kRowThreads) {
      const uint4 v = s4[c];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h2 = __floats2half2_rn(__uint_as_float(w[i] << 16) * down,
                                             __uint_as_float(w[i] & 0xffff0000u) * down);
        o[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      d4[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (tid == 0) row_scale[p] = ldexpf(1.0f, k);
    __syncthreads();  // s_max is reused by the next row
  }
}

cudaError_t launch_rows_to_f16(const uint16_t* src, int K, int P, uint16_t* dst, float* row_scale, int num_sms,
                               cudaStream_t s, const int32_t* src_rows = nullptr, int64_t src_prefetch_bytes = 0) {
  int blocks = P < num_sms * 4 ? P : num_sms * 4;
  if (blocks < 1) blocks = 1;
  return launch_pdl(rows_to_f16_kernel, dim3(blocks), dim3(kRowThreads), 0, s, reinterpret_cast<const uint4*>(src),
                    K / 8, static_cast<int64_t>(P), reinterpret_cast<uint4*>(dst), row_scale, src_rows,
                    src_prefetch_bytes);
}

// Per device: the shared-memory attribute set, and (CTA pairs) the clusters that can be resident
// at once (a persistent grid must not be larger, or the late CTAs would run after the others).
template <int kKind, int kN, bool kPair>
cudaError_t prepare_tc_kernel(int* resident) {
  using G = tc::Geo<kKind, kN, kPair>;
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDev) {
    const int c = cache[dev].load(std::memory_order_acquire);
    if (c > 0) {
      *resident = c;
      return cudaSuccess;
    }
  }
  e = cudaFuncSetAttribute(tc::expert_tc_kernel<kKind, kN, kPair>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           G::kSmem);
  if (e != cudaSuccess) return e;
  int n = kPartialCtas;
  if (kPair) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kPartialCtas);
    cfg.blockDim = dim3(G::kThreads);
    cfg.dynamicSmemBytes = G::kSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&n, tc::expert_tc_kernel<kKind, kN, kPair>, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorNotSupported;
  }
  if (dev < kMaxDev) cache[dev].store(n, std::memory_order_release);
  *resident = n;
  return cudaSuccess;
}

template <int kKind, int kN, bool kPair>
cudaError_t launch_tc_kernel(const CUtensorMap& a0, const CUtensorMap& a1, const void* tokens, int K, int P,
                             const tc::Args& args, int num_ctas, cudaStream_t s) {
  using G = tc::Geo<kKind, kN, kPair>;
  tc::TokenMaps tb;
  for (int m = 0; m < 4; ++m)
    if (!encode_tokens(&tb.m[m], tokens, K, P, false, (kPair && m == 0) ? G::kBRows : 128 >> m))
      return cudaErrorInvalidValue;
  int resident = 0;
  cudaError_t e = prepare_tc_kernel<kKind, kN, kPair>(&resident);
  if (e != cudaSuccess) return e;
  if (!kPair)
    return launch_pdl(tc::expert_tc_kernel<kKind, kN, kPair>, dim3(num_ctas), dim3(G::kThreads), G::kSmem, s, a0,
                      a1, tb, args);
  int pairs = num_ctas / 2 < resident ? num_ctas / 2 : resident;
  if (pairs < 1) pairs = 1;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(G::kThreads);
  cfg.dynamicSmemBytes = G::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tc::expert_tc_kernel<kKind, kN, kPair>, a0, a1, tb, args);
}

// Launch the kernel of `pass` tokens per pass (64 on single CTAs; 128, 192 or 256 on CTA pairs), or of
// 64 where its partial slots would not fit in `slot` fp32.
template <bool kGateUp>
cudaError_t launch_tc_pass(int pass, int64_t slot, const CUtensorMap& a0, const CUtensorMap& a1, const void* tokens,
                           int K, int P, tc::Args args, int num_ctas, cudaStream_t s) {
  if (partial_slot_floats(pass, kGateUp) > slot) pass = 64;
  args.partial_stride = partial_slot_floats(pass, kGateUp);
  // on pairs down takes two 128-row tiles per stage (tc::kDown2), like gate and up
  constexpr int kPairKind = kGateUp ? tc::kGateUp : tc::kDown2;
  if (pass == 256) return launch_tc_kernel<kPairKind, 256, true>(a0, a1, tokens, K, P, args, num_ctas, s);
  if (pass == 192) return launch_tc_kernel<kPairKind, 192, true>(a0, a1, tokens, K, P, args, num_ctas, s);
  if (pass == 128) return launch_tc_kernel<kPairKind, 128, true>(a0, a1, tokens, K, P, args, num_ctas, s);
  args.partial_stride = kPartialSlotFloats;
  return launch_tc_kernel<kGateUp ? tc::kGateUp : tc::kDownK2, 64, false>(a0, a1, tokens, K, P, args, num_ctas, s);
}

std::atomic<int> g_pass_gate_up{0}, g_pass_down{0};
// Above 96 tokens per expert on average: 192-token passes when the largest expert (estimated as
// mean + 2 sqrt(mean)) needs no more ranks at 192 than at 256 (its token slots then load as one
// box with nothing past the ranks' shares; measured on GB300 +1-4% at 256 and 512 tokens per
// expert), else 256 (one rank more cost 8% at 1024 tokens per expert).
int pass_by_mean(int64_t P, int E) {
  const int64_t mean = (P + E - 1) / (E > 0 ? E : 1);
  if (mean <= 40) return 64;
  if (mean <= 96) return 128;
  const double est = static_cast<double>(mean) + 2.0 * std::sqrt(static_cast<double>(mean));
  const int64_t g256 = static_cast<int64_t>(std::ceil(est / 256.0));
  const int64_t g192 = static_cast<int64_t>(std::ceil(est / 192.0));
  return g192 == g256 ? 192 : 256;
}
int valid_pass(int n) { return n == 64 || n == 128 || n == 192 || n == 256 ? n : 0; }

// BF16: weight boxes of 128 rows by 128 bytes; token boxes of 64/32/16 rows (single CTAs) or one box of a
// pair CTA's whole token slot (tc::TokenMaps).
cudaError_t launch_tc(const ExpertFfnPlan& p, cudaStream_t s) {
  CUtensorMap tg, tu, td;
  if (!tensor_map_encoder()) return cudaErrorNotSupported;
  if (!encode_weights(&tg, p.W_gate, false, p.H, p.I, p.E, 128) ||
      !encode_weights(&tu, p.W_up, false, p.H, p.I, p.E, 128) ||
      !encode_weights(&td, p.W_down, false, p.I, p.H, p.E, 128))
    return cudaErrorInvalidValue;
  const int64_t slot = p.partial_slot > kPartialSlotFloats ? p.partial_slot : kPartialSlotFloats;
  tc::Args a{};
  a.wait_ns = p.wait_ns;
  a.offsets = p.offsets;
  a.active = p.active;
  a.num_active = p.num_active;
  a.partials = p.partials;
  a.counters = p.counters;
  a.status = p.status;
  a.E = p.E;
  a.P = p.P;
  tc::Args gu = a;
  gu.out = p.h;
  gu.out_ld = p.I;
  gu.rows = p.I;
  gu.K = p.H;
  cudaError_t e = launch_tc_pass<true>(p.passes.gate_up, slot, tg, tu, p.xg, p.H, p.P, gu, p.num_ctas, s);
  if (e != cudaSuccess) return e;
  tc::Args dn = a;
  dn.out = p.Y;
  dn.out_ld = p.H;
  dn.rows = p.H;
  dn.K = p.I;
  return launch_tc_pass<false>(p.passes.down, slot, td, td, p.h, p.I, p.P, dn, p.num_ctas, s);
}

// ---- INT8 on CTA pairs
template <bool kGateUp, int kN>
cudaError_t prepare_pair_kernel() {
  constexpr int kMaxDev = 64;
  static std::atomic<bool> done[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDev && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(pair::expert_pair_kernel<kGateUp, kN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           pair::Geo<kGateUp, kN>::kSmem);
  if (e == cudaSuccess && dev < kMaxDev) done[dev].store(true, std::memory_order_release);
  return e;
}

// Pairs of the pair kernel that can be resident at once on this device (a persistent stream-K
// grid must not be larger, or the late pairs would run after the others instead of beside them).
template <bool kGateUp, int kN>
cudaError_t resident_pairs(int* pairs) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDev) {
    const int c = cache[dev].load(std::memory_order_acquire);
    if (c > 0) {
      *pairs = c;
      return cudaSuccess;
    }
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kPartialCtas);
  cfg.blockDim = dim3(pair::kThreads);
  cfg.dynamicSmemBytes = pair::Geo<kGateUp, kN>::kSmem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, pair::expert_pair_kernel<kGateUp, kN>, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorNotSupported;
  if (dev < kMaxDev) cache[dev].store(n, std::memory_order_release);
  *pairs = n;
  return cudaSuccess;
}

// Launch on `pairs` clusters of two CTAs, with programmatic dependent launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pairs_pdl(void (*kernel)(KArgs...), int pairs, size_t smem, cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(pair::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// INT8: fp16 token copy, gate+up on pairs, fp16 copy of h, down on pairs. Weight boxes are one
// CTA's 128 rows by 128 bytes; token boxes are 8 rows (a CTA holds half of a pass's tokens).
template <int kN>
cudaError_t launch_pair_int8_n(const ExpertFfnPlan& p, cudaStream_t s) {
  CUtensorMap tg, tu, td, txg, th;
  if (!tensor_map_encoder()) return cudaErrorNotSupported;
  if (!encode_weights(&tg, p.W_gate, true, p.H, p.I, p.E, 128) ||
      !encode_weights(&tu, p.W_up, true, p.H, p.I, p.E, 128) ||
      !encode_weights(&td, p.W_down, true, p.I, p.H, p.E, 128) ||
      !encode_tokens(&txg, p.xg16, p.H, p.P, true, 8) || !encode_tokens(&th, p.h16, p.I, p.P, true, 8))
    return cudaErrorInvalidValue;
  // residual split: gate and up run over W^Q then W^R (the maps are unused otherwise)
  const bool residual = p.W_gate_r != nullptr;
  CUtensorMap tgr = tg, tur = tu;
  if (residual && (!encode_weights(&tgr, p.W_gate_r, true, p.H, p.I, p.E, 128) ||
                   !encode_weights(&tur, p.W_up_r, true, p.H, p.I, p.E, 128)))
    return cudaErrorInvalidValue;
  cudaError_t e = prepare_pair_kernel<true, kN>();
  if (e == cudaSuccess) e = prepare_pair_kernel<false, kN>();
  int pairs_gu = 0, pairs_dn = 0;
  if (e == cudaSuccess) e = resident_pairs<true, kN>(&pairs_gu);
  if (e == cudaSuccess) e = resident_pairs<false, kN>(&pairs_dn);
  if (e != cudaSuccess) return e;
  const int max_pairs = p.num_ctas / 2 > 0 ? p.num_ctas / 2 : 1;
  pairs_gu = pairs_gu < max_pairs ? pairs_gu : max_pairs;
  pairs_dn = pairs_dn < max_pairs ? pairs_dn : max_pairs;
  tc::Args a{};
  a.offsets = p.offsets;
  a.active = p.active;
  a.num_active = p.num_active;
  a.partials = p.partials;
  a.counters = p.counters;
  a.status = p.status;
  a.E = p.E;
  a.P = p.P;
  if (!p.xg16_ready) {
    e = launch_rows_to_f16(p.xg, p.H, p.P, p.xg16, p.xg_scale, p.num_ctas, s);
    if (e != cudaSuccess) return e;
  }
  tc::Args gu = a;
  gu.out = p.h;
  gu.out_ld = p.I;
  gu.rows = p.I;
  gu.K = p.H;
  gu.s0 = p.s_gate;
  gu.s1 = p.s_up;
  gu.row_scale = p.xg_scale;
  if (residual) {
    gu.s0r = p.s_gate_r;
    gu.s1r = p.s_up_r;
    gu.kq = p.H / 128;
  }
  e = launch_pairs_pdl(pair::expert_pair_kernel<true, kN>, pairs_gu, pair::Geo<true, kN>::kSmem, s, tg, tu, txg, tgr,
                       tur, gu);
  if (e != cudaSuccess) return e;
  e = launch_rows_to_f16(p.h, p.I, p.P, p.h16, p.h_scale, p.num_ctas, s);
  if (e != cudaSuccess) return e;
  tc::Args dn = a;
  dn.out = p.Y;
  dn.out_ld = p.H;
  dn.rows = p.H;
  dn.K = p.I;
  dn.s0 = p.s_down;
  dn.s1 = p.s_down;
  dn.row_scale = p.h_scale;
  return launch_pairs_pdl(pair::expert_pair_kernel<false, kN>, pairs_dn, pair::Geo<false, kN>::kSmem, s, td, td, th,
                          td, td, dn);
}

// Passes of 16 tokens (three TMEM operand buffers instead of two, half the promotion work) while
// the experts see at most about nine tokens each on average, passes of 32 above: measured on GB300
// (Qwen3-235B shapes), the shorter passes are 2-10% faster up to 8 assignments per expert, 1%
// slower at 10, 5% slower at 12 (experts past 16 tokens take two passes and stream their weights
// twice).
cudaError_t launch_pair_int8(const ExpertFfnPlan& p, cudaStream_t s) {
  if (static_cast<int64_t>(p.P) <= 9LL * p.E) return launch_pair_int8_n<16>(p, s);
  return launch_pair_int8_n<32>(p, s);
}

}  // namespace

cudaError_t launch_gather_f16(const uint16_t* x, int T, int H, int P, const int32_t* sorted_token, uint16_t* xg16,
                              float* xg_scale, int num_sms, cudaStream_t stream) {
  // a decode batch's token rows (at most a few MB) are warmed in L2 before the wait for routing
  const int64_t x_bytes = static_cast<int64_t>(T) * H * 2;
  return launch_rows_to_f16(x, H, P, xg16, xg_scale, num_sms, stream, sorted_token,
                            x_bytes <= kPrefetchMaxBytes ? x_bytes : int64_t{0});
}

PassTokens pass_tokens(int64_t P, int E) {
  const int auto_pass = pass_by_mean(P, E);
  const int gu = valid_pass(g_pass_gate_up.load(std::memory_order_relaxed));
  const int dn = valid_pass(g_pass_down.load(std::memory_order_relaxed));
  return PassTokens{gu ? gu : auto_pass, dn ? dn : auto_pass};
}

void set_pass_tokens(int gate_up, int down) {
  g_pass_gate_up.store(valid_pass(gate_up), std::memory_order_relaxed);
  g_pass_down.store(valid_pass(down), std::memory_order_relaxed);
}

cudaError_t launch_expert_ffn(const ExpertFfnPlan& plan, cudaStream_t stream) {
  return plan.int8 ? launch_pair_int8(plan, stream) : launch_tc(plan, stream);
}

}  // namespace moe
