// Host side of the weight-streaming expert kernels: TMA descriptors and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "expert_stream.cuh"
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

namespace {

// Weights of all experts as a 3-D tensor {K (contiguous), rows, E}; box = one stage of
// 128 bytes along K by `box_rows` rows of one expert; 128-byte swizzle.
bool encode_weights(CUtensorMap* map, const void* W, bool int8, int K, int rows, int E, int box_rows) {
  const cuuint64_t eb = int8 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(E)};
  cuuint64_t strides[2] = {K * eb, static_cast<cuuint64_t>(K) * rows * eb};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = tensor_map_encoder()(map, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                    const_cast<void*>(W), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Token block {K (contiguous), P rows} bf16; box = 64 elements x 8 rows; 128-byte swizzle.
bool encode_tokens(CUtensorMap* map, const void* X, int K, int P) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(P)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {64, 8};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = tensor_map_encoder()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides,
                                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool kInt8, bool kGateUp>
cudaError_t prepare_kernel() {
  // the dynamic shared-memory opt-in is per device
  constexpr int kMaxDev = 64;
  static std::atomic<bool> done[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDev && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(stream::expert_stream_kernel<kInt8, kGateUp>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, stream::Geometry<kInt8>::kSmem);
  if (e == cudaSuccess && dev < kMaxDev) done[dev].store(true, std::memory_order_release);
  return e;
}

template <bool kInt8>
cudaError_t launch_both(const ExpertFfnPlan& p, cudaStream_t s) {
  using G = stream::Geometry<kInt8>;
  CUtensorMap tg, tu, td, txg, th;
  if (!tensor_map_encoder()) return cudaErrorNotSupported;
  if (!encode_weights(&tg, p.W_gate, kInt8, p.H, p.I, p.E, 64) ||
      !encode_weights(&tu, p.W_up, kInt8, p.H, p.I, p.E, 64) ||
      !encode_weights(&td, p.W_down, kInt8, p.I, p.H, p.E, 128) || !encode_tokens(&txg, p.xg, p.H, p.P) ||
      !encode_tokens(&th, p.h, p.I, p.P))
    return cudaErrorInvalidValue;
  cudaError_t e = prepare_kernel<kInt8, true>();
  if (e != cudaSuccess) return e;
  e = prepare_kernel<kInt8, false>();
  if (e != cudaSuccess) return e;

  stream::Args a{};
  a.offsets = p.offsets;
  a.active = p.active;
  a.num_active = p.num_active;
  a.partials = p.partials;
  a.counters = p.counters;
  a.status = p.status;
  a.E = p.E;
  a.P = p.P;

  stream::Args gu = a;
  gu.s0 = p.s_gate;
  gu.s1 = p.s_up;
  gu.out = p.h;
  gu.out_ld = p.I;
  gu.rows = p.I;
  gu.K = p.H;
  e = launch_pdl(stream::expert_stream_kernel<kInt8, true>, dim3(p.num_ctas), dim3(stream::kThreads), G::kSmem, s,
                 tg, tu, txg, gu);
  if (e != cudaSuccess) return e;

  stream::Args dn = a;
  dn.s0 = p.s_down;
  dn.s1 = p.s_down;
  dn.out = p.Y;
  dn.out_ld = p.H;
  dn.rows = p.H;
  dn.K = p.I;
  return launch_pdl(stream::expert_stream_kernel<kInt8, false>, dim3(p.num_ctas), dim3(stream::kThreads), G::kSmem,
                    s, td, td, th, dn);
}

}  // namespace

cudaError_t launch_expert_ffn(const ExpertFfnPlan& plan, cudaStream_t stream) {
  return plan.int8 ? launch_both<true>(plan, stream) : launch_both<false>(plan, stream);
}

}  // namespace moe
