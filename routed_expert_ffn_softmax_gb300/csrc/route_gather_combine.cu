// Routing (softmax top-k, renormalised), token gather and weighted combine.
//
// Routing follows HiNa-MoE (arXiv 2610.05123) §2.1 (the gate routes each token to a
// small subset of experts) and §8.1 Table 3 (Top-2 / Top-8); the pages print no gating
// formula, and the reading implemented is softmax over the E logits, top-k, renormalised
// over the kept k: w_j = exp(l_j - m) / sum_kept exp(l_i - m), m the largest kept logit.
// Slot j is the j-th largest logit; equal logits go to the lower expert id.
// The gather builds the per-expert intermediate matrix I of §4.1 (Figure 5); the
// combine writes the weighted expert outputs back in row-major token order.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>

#include <cstdint>

#include "moe_device.cuh"
#include "moe_launch.h"
#include "route_topk.cuh"

namespace moe {

// ---------------------------------------------------------------------------------
// Top-k per token: one warp per token (topk_tokens, route_topk.cuh).
constexpr int kTopkWarpsPerBlock = 8;

__global__ void __launch_bounds__(kTopkWarpsPerBlock * 32)
    route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                      int32_t* __restrict__ ids, float* __restrict__ w) {
  pdl_wait_predecessor();
  pdl_allow_successor();
  __shared__ float s_sv[kTopkWarpsPerBlock][256];
  __shared__ int s_si[kTopkWarpsPerBlock][256];
  const int tok = blockIdx.x * kTopkWarpsPerBlock + (threadIdx.x >> 5);
  topk_tokens<8, 1>(logits, tok, 0, T, E, k, ids, w, s_sv[threadIdx.x >> 5], s_si[threadIdx.x >> 5], 0);
}

// ---------------------------------------------------------------------------------
// Histogram, exclusive scan, stable permutation, active list: one CTA.
// Tokens are taken 1024 at a time; within a chunk an expert's rank is found from
// a per-expert bitmask over the chunk's tokens (smem), so ranks follow token order.
constexpr int kScanThreads = 1024;
constexpr int kScanWarps = kScanThreads / 32;

struct ScanShared {
  int cnt[256];
  int off[256];
  int run[256];
  int wsum[kScanWarps];
  uint32_t mask[256 * kScanWarps];
};

// `ids` may have been written earlier in the same launch (route_fused_kernel), so it is read
// through ordinary loads, not the read-only path.
__device__ __forceinline__ void scan_block(ScanShared& sh, const int32_t* ids, int T, int E, int k,
                                           int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                           int32_t* __restrict__ sorted_token, int32_t* __restrict__ inv_pos,
                                           int32_t* __restrict__ active, int32_t* __restrict__ num_active,
                                           int32_t* __restrict__ zero_words, int n_zero) {
  int* s_cnt = sh.cnt;
  int* s_off = sh.off;
  int* s_run = sh.run;
  int* s_wsum = sh.wsum;
  uint32_t* s_mask = sh.mask;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  for (int i = tid; i < n_zero; i += kScanThreads) zero_words[i] = 0;
  if (tid < 256) {
    s_cnt[tid] = 0;
    s_run[tid] = 0;
  }
  __syncthreads();
  const int64_t P = static_cast<int64_t>(T) * k;
  for (int64_t a = tid; a < P; a += kScanThreads) atomicAdd(&s_cnt[ids[a]], 1);
  __syncthreads();

  // exclusive scan of counts (E <= 256) and of the active flags
  auto block_scan256 = [&](int x) -> int {  // inclusive scan over threads 0..255
    int v = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (tid < 256 && lane == 31) s_wsum[warp] = v;
    __syncthreads();
    int add = 0;
    if (tid < 256)
      for (int w2 = 0; w2 < warp; ++w2) add += s_wsum[w2];
    __syncthreads();
    return v + add;
  };
  const int c = (tid < E) ? s_cnt[tid] : 0;
  const int cinc = block_scan256(c);
  if (tid < E) {
    s_off[tid] = cinc - c;
    counts[tid] = c;
    offsets[tid] = cinc - c;
    if (tid == E - 1) offsets[E] = cinc;
  }
  const int f = (tid < E && c > 0) ? 1 : 0;
  const int finc = block_scan256(f);
  if (f) active[finc - 1] = tid;
  if (tid == E - 1) *num_active = finc;
  __syncthreads();

  // stable placement, 1024 tokens per chunk
  for (int base = 0; base < T; base += kScanThreads) {
    for (int i = tid; i < 256 * kScanWarps; i += kScanThreads) s_mask[i] = 0;
    __syncthreads();
    const int t = base + tid;
    if (t < T)
      for (int j = 0; j < k; ++j) atomicOr(&s_mask[ids[static_cast<int64_t>(t) * k + j] * kScanWarps + warp], 1u << lane);
    __syncthreads();
    if (t < T) {
      for (int j = 0; j < k; ++j) {
        const int e = ids[static_cast<int64_t>(t) * k + j];
        const uint32_t* m = s_mask + e * kScanWarps;
        int r = s_run[e] + __popc(m[warp] & ((1u << lane) - 1u));
        for (int w2 = 0; w2 < warp; ++w2) r += __popc(m[w2]);
        const int p = s_off[e] + r;
        sorted_token[p] = t;
        inv_pos[static_cast<int64_t>(t) * k + j] = p;
      }
    }
    __syncthreads();
    if (tid < E) {
      int add = 0;
      for (int w2 = 0; w2 < kScanWarps; ++w2) add += __popc(s_mask[tid * kScanWarps + w2]);
      s_run[tid] += add;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kScanThreads)
    route_scan_kernel(const int32_t* __restrict__ ids, int T, int E, int k,
                      int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                      int32_t* __restrict__ sorted_token, int32_t* __restrict__ inv_pos,
                      int32_t* __restrict__ active, int32_t* __restrict__ num_active,
                      int32_t* __restrict__ zero_words, int n_zero) {
  __shared__ ScanShared sh;
  pdl_wait_predecessor();
  pdl_allow_successor();
  scan_block(sh, ids, T, E, k, counts, offsets, sorted_token, inv_pos, active, num_active, zero_words, n_zero);
}

// Decode-sized batches (T <= 64, T * k <= 1024): one launch instead of two. The CTA's warps take
// the tokens' top-k (kept in shared memory as well) and mark each expert's tokens in a 64-bit
// mask; warp 0 builds the exclusive offsets and the active list; then every assignment (t, j)
// finds its place in the stable expert-major order as offset[e] + the number of earlier tokens in
// e's mask. The general scan above needs many more block-wide barriers.
constexpr int kFusedRouteMaxT = 64;
constexpr int kFusedRouteMaxP = 1024;

__global__ void __launch_bounds__(kScanThreads)
    route_fused_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* ids, float* w,
                       int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                       int32_t* __restrict__ sorted_token, int32_t* __restrict__ inv_pos,
                       int32_t* __restrict__ active, int32_t* __restrict__ num_active,
                       int32_t* __restrict__ zero_words, int n_zero) {
  __shared__ int s_ids[kFusedRouteMaxP];  // token t's experts at t * k .. t * k + k - 1
  __shared__ float s_val[kFusedRouteMaxP];
  __shared__ int s_cnt[256];
  __shared__ int s_off[256];
  __shared__ unsigned long long s_tok[256];  // bit t: token t routed to the expert
  prefetch_l2_grid(logits, static_cast<int64_t>(T) * E * 4);
  pdl_wait_predecessor();
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  for (int i = tid; i < n_zero; i += kScanThreads) zero_words[i] = 0;
  if (tid < 256) {
    s_cnt[tid] = 0;
    s_tok[tid] = 0ull;
  }
  __syncthreads();
  {  // warp v takes tokens v and v + 32 (T <= 64): both at once where there are two and the
     // registers allow (a dummy second token would only lengthen the single token's chain)
    const int v = tid >> 5;
    if (E <= 128 && T > kScanWarps) {
      topk_tokens<4, 2>(logits, v, kScanWarps, T, E, k, ids, w, s_val + v * k, s_ids + v * k, kScanWarps * k);
    } else {
      for (int tok = v; tok < T; tok += kScanWarps)
        topk_tokens<8, 1>(logits, tok, 0, T, E, k, ids, w, s_val + tok * k, s_ids + tok * k, 0);
    }
  }
  __syncthreads();
  const int P = T * k;
  for (int a = tid; a < P; a += kScanThreads) {
    const int e = s_ids[a];
    atomicAdd(&s_cnt[e], 1);
    atomicOr(&s_tok[e], 1ull << (a / k));
  }
  __syncthreads();
  if (tid < 32) {  // warp 0
    // exclusive scan of the counts and the active list, 32 experts at a time
    int run = 0, nact = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int c = e < E ? s_cnt[e] : 0;
      int incl = c;
  #pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      const uint32_t act = __ballot_sync(0xffffffffu, c > 0);
      if (e < E) {
        s_off[e] = run + incl - c;
        counts[e] = c;
        offsets[e] = run + incl - c;
        if (c > 0) active[nact + __popc(act & ((1u << lane) - 1u))] = e;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      nact += __popc(act);
    }
    if (lane == 0) {
      offsets[E] = run;
      *num_active = nact;
    }
  }
  __syncthreads();
  // stable placement: tokens of an expert in token order
  for (int a = tid; a < P; a += kScanThreads) {
    const int t = a / k;
    const int e = s_ids[a];
    const int p = s_off[e] + __popcll(s_tok[e] & ((1ull << t) - 1ull));
    sorted_token[p] = t;
    inv_pos[a] = p;
  }
  // the successor is let go only now: launched early, its blocks could do nothing but wait
  // (measured on GB300 together with the shared-memory selection above: routing 1 µs shorter)
  pdl_allow_successor();
}

// ---------------------------------------------------------------------------------
// xg[p, :] = x[sorted_token[p], :], 16 bytes per thread.
__global__ void __launch_bounds__(256)
    gather_kernel(const uint4* __restrict__ x, int H8, const int32_t* __restrict__ sorted_token,
                  int64_t P, uint4* __restrict__ xg, int64_t x_prefetch_bytes) {
  prefetch_l2_grid(x, x_prefetch_bytes);
  pdl_wait_predecessor();
  pdl_allow_successor();
  const int64_t n = P * H8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = i / H8;
    const int64_t c = i - p * H8;
    xg[i] = x[static_cast<int64_t>(sorted_token[p]) * H8 + c];
  }
}

// ---------------------------------------------------------------------------------
// out[t, r] = bf16( sum_j w[t,j] * Y[inv_pos[t,j], r] ), fp32, slot order, 4 columns per thread.
__global__ void __launch_bounds__(256)
    combine_kernel(const float4* __restrict__ Y, const int32_t* __restrict__ inv_pos,
                   const float* __restrict__ w, int T, int k, int H4, uint2* __restrict__ out) {
  pdl_wait_predecessor();
  pdl_allow_successor();
  const int64_t n = static_cast<int64_t>(T) * H4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / H4;
    const int64_t c = i - t * H4;
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    for (int j = 0; j < k; ++j) {
      const float wj = w[t * k + j];
      const float4 y = Y[static_cast<int64_t>(inv_pos[t * k + j]) * H4 + c];
      a0 = __fadd_rn(a0, __fmul_rn(wj, y.x));
      a1 = __fadd_rn(a1, __fmul_rn(wj, y.y));
      a2 = __fadd_rn(a2, __fmul_rn(wj, y.z));
      a3 = __fadd_rn(a3, __fmul_rn(wj, y.w));
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a0, a1);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(a2, a3);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&lo);
    o.y = *reinterpret_cast<const uint32_t*>(&hi);
    out[i] = o;
  }
}

// ---------------------------------------------------------------------------------
// launchers (programmatic dependent launch on every kernel)
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         int32_t* counts, int32_t* offsets, int32_t* sorted_token, int32_t* inv_pos,
                         int32_t* active, int32_t* num_active, int32_t* zero_words, int n_zero,
                         cudaStream_t stream) {
  if (T <= kFusedRouteMaxT && static_cast<int64_t>(T) * k <= kFusedRouteMaxP)
    return launch_pdl(route_fused_kernel, dim3(1), dim3(kScanThreads), 0, stream, logits, T, E, k, ids, w, counts,
                      offsets, sorted_token, inv_pos, active, num_active, zero_words, n_zero);
  const int blocks = (T + kTopkWarpsPerBlock - 1) / kTopkWarpsPerBlock;
  cudaError_t err = launch_pdl(route_topk_kernel, dim3(blocks), dim3(kTopkWarpsPerBlock * 32), 0, stream,
                               logits, T, E, k, ids, w);
  if (err != cudaSuccess) return err;
  return launch_pdl(route_scan_kernel, dim3(1), dim3(kScanThreads), 0, stream, (const int32_t*)ids, T, E, k,
                    counts, offsets, sorted_token, inv_pos, active, num_active, zero_words, n_zero);
}

cudaError_t launch_gather(const uint16_t* x, int T, int H, int k, const int32_t* sorted_token, uint16_t* xg,
                          int num_sms, cudaStream_t stream) {
  const int64_t P = static_cast<int64_t>(T) * k;
  const int H8 = H / 8;
  const int64_t n = P * H8;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  // a decode batch's token rows (at most a few MB) are warmed in L2 before the wait for routing
  const int64_t x_bytes = static_cast<int64_t>(T) * H * 2;
  return launch_pdl(gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                    reinterpret_cast<const uint4*>(x), H8, sorted_token, P, reinterpret_cast<uint4*>(xg),
                    x_bytes <= kPrefetchMaxBytes ? x_bytes : int64_t{0});
}

cudaError_t launch_combine(const float* Y, const int32_t* inv_pos, const float* w, int T, int k, int H,
                           uint16_t* out, int num_sms, cudaStream_t stream) {
  const int H4 = H / 4;
  const int64_t n = static_cast<int64_t>(T) * H4;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                    reinterpret_cast<const float4*>(Y), inv_pos, w, T, k, H4, reinterpret_cast<uint2*>(out));
}

}  // namespace moe
