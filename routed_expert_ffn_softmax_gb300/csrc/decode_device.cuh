// Device-side building blocks of the fused decode step (decode_step.cu): contiguous bulk copies,
// proxy fences, scoped loads and stores for the grid barrier and tagged partial sums, and the mixed-precision
// FMA that takes bf16 operands with an fp32 accumulator.
#pragma once

#include "moe_device.cuh"

namespace moe {

// Status code of the fused decode step: the grid-wide barrier did not open in time.
constexpr int32_t kStatusGridTimeout = 5;
}  // namespace moe

namespace moe {

// ---------------------------------------------------------------- bulk copies and proxies
// Contiguous global -> shared copy by the async proxy (cp.async.bulk), completion signalled on
// `bar` as transaction bytes. Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// 3-D tiled tensor load with the default L2 policy.
__device__ __forceinline__ void tma_load_3d_plain(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                                  int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Order this thread's generic-proxy global writes before later async-proxy (bulk copy) reads, and
// the acquire of another CTA's release before this thread's later async-proxy reads.
// mbarrier try_wait that suspends for at most ~64 ns: for a thread that must also poll something else
// (a plain try_wait may suspend for microseconds before it returns false).
__device__ __forceinline__ bool mbar_try_wait_short(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(64)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ int ld_relaxed_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 64-bit relaxed load and store at GPU scope. A naturally aligned 64-bit access is single-copy atomic,
// so a value stored together with a tag is read either whole or not at all.
__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---------------------------------------------------------------- mixed-precision FMAs
// acc += lo(w) * lo(x) + hi(w) * hi(x) for two packed bf16 pairs, each product exact and added to the
// fp32 accumulator with one rounding (fma.rn.f32.bf16).
__device__ __forceinline__ float fma2_bf16(uint32_t w2, uint32_t x2, float acc) {
  asm("{.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\tfma.rn.f32.bf16 %0, wh, xh, %0;}"
      : "+f"(acc)
      : "r"(w2), "r"(x2));
  return acc;
}

}  // namespace moe
