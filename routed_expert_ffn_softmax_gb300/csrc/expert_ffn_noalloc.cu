// moe_expert_ffn_noalloc: the grouped expert FFN for callers that cannot provide a workspace.
//
// Some callers of this library cannot allocate device memory when they call it: a plugin
// running inside another runtime whose device memory belongs to that runtime's own pool,
// or a decode loop that must not call cudaMalloc mid-step (the call synchronises the device
// and may fail once memory is fragmented). This entry point runs the same gate+up and down
// kernels as moe_expert_ffn, but their scratch (status word, stream-K counters and partial
// sums, and the bf16 intermediate h) lives in one fixed array of this library,
// g_expert_ffn_scratch below, instead of a caller-supplied workspace.
//
// Costs and limits, for users:
//   * Every GPU on which this library is loaded reserves kScratchBytes (48 MiB) for the
//     array, from module load until the process exits, whether or not this entry point
//     is ever called.
//   * The token block must fit: P * I * 2 bytes of intermediate (BF16 weights), or
//     P * (4 * I + 2 * H + 8) bytes (INT8 weights: h plus fp16 copies of h and of the token
//     block with their row scales), at most kHMaxBytes (about 28 MiB; BF16: up to about 7100
//     rows at I = 2048, or 1000 rows at I = 14336); larger requests return MOE_ERR_WORKSPACE
//     and launch nothing.
//   * At most kCtas (160) CTAs take part, one per SM, whatever the SM count.
//   * All calls share the one array, which keeps what the last call left in it. Calls whose
//     kernels overlap on the GPU (different streams, or different host threads, on the same
//     device) race on it and produce wrong results; serialise them.
//   * The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current and keeps it until the process exits;
//     make that first call before any stream capture begins on the device, and keep the
//     device's primary context alive (no cudaDeviceReset) between calls.
//   * A kernel that gives up on a bounded wait writes a nonzero code into the status word at
//     the start of the array; moe_expert_ffn_noalloc_status copies it out. Every call clears
//     it first.
// The paper has no counterpart of this entry point: it concerns memory ownership only.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "moe.h"
#include "moe_launch.h"

namespace {

constexpr size_t kScratchBytes = size_t(48) << 20;
constexpr int kCtas = 160;                 // partial-slot capacity
constexpr size_t kCountersOffset = 256;    // status word at byte 0, counters at 256
constexpr size_t kZeroBytes = kCountersOffset + 4 * moe::kPartialCtas;
constexpr size_t kPartialsOffset = 2048;
constexpr size_t kPartialsBytes = size_t(kCtas) * 2 * moe::kPartialSlotFloats * sizeof(float);
constexpr size_t kHOffset = kPartialsOffset + kPartialsBytes;
constexpr size_t kHMaxBytes = kScratchBytes - kHOffset;
static_assert(kZeroBytes <= kPartialsOffset, "control words overlap the partials");
static_assert(kHOffset % 256 == 0, "h must stay 256-byte aligned");

}  // namespace

// The scratch itself. In host code this name is only a stand-in for the symbol: the kernels
// must be given the device address returned by cudaGetSymbolAddress, never this name.
static __device__ __align__(256) unsigned char g_expert_ffn_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

// Device address of the scratch array and the SM count, for the current device; looked up
// once per device.
cudaError_t scratch_for_current_device(char** ptr, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_expert_ffn_scratch);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (p == nullptr || n < 1) return cudaErrorInvalidValue;
    g_scratch_ptr[dev] = p;
    g_sms[dev] = n;
  }
  *ptr = static_cast<char*>(g_scratch_ptr[dev]);
  *sms = g_sms[dev];
  return cudaSuccess;
}

bool is_aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" moe_status_t moe_expert_ffn_noalloc(const uint16_t* xg, const int32_t* expert_offsets,
                                               const int32_t* active_experts, const int32_t* num_active,
                                               const void* W_gate, const void* W_up, const void* W_down,
                                               const float* s_gate, const float* s_up, const float* s_down,
                                               moe_wtype_t wtype, int H, int I, int E, int P, float* Y,
                                               moe_stream_t stream) {
  // the same argument rules as moe_expert_ffn
  if (P < 0 || H < 1 || I < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (wtype != MOE_W_BF16 && wtype != MOE_W_INT8_G128) return MOE_ERR_INVALID_ARG;
  if (E > 256) return MOE_ERR_UNSUPPORTED;
  const int m = wtype == MOE_W_INT8_G128 ? 128 : 8;
  if (H % m || I % m) return MOE_ERR_INVALID_ARG;
  if (P == 0) return MOE_OK;
  if (!xg || !expert_offsets || !active_experts || !num_active || !Y) return MOE_ERR_INVALID_ARG;
  if (!is_aligned(xg, 16) || !is_aligned(Y, 16) || !is_aligned(expert_offsets, 4) ||
      !is_aligned(active_experts, 4) || !is_aligned(num_active, 4))
    return MOE_ERR_INVALID_ARG;
  if (!W_gate || !W_up || !W_down || !is_aligned(W_gate, 16) || !is_aligned(W_up, 16) || !is_aligned(W_down, 16))
    return MOE_ERR_INVALID_ARG;
  if (wtype == MOE_W_INT8_G128 && (!s_gate || !s_up || !s_down || !is_aligned(s_gate, 4) ||
                                   !is_aligned(s_up, 4) || !is_aligned(s_down, 4)))
    return MOE_ERR_INVALID_ARG;
  // the fixed scratch must hold the intermediate h [P, I] bf16 (and, for INT8, the fp16 copies)
  const bool int8 = wtype == MOE_W_INT8_G128;
  auto up256 = [](uint64_t x) { return (x + 255) / 256 * 256; };
  const uint64_t h_bytes = up256(uint64_t(P) * uint64_t(I) * 2u);
  const uint64_t h16_bytes = int8 ? h_bytes : 0;
  const uint64_t xg16_bytes = int8 ? up256(uint64_t(P) * uint64_t(H) * 2u) : 0;
  const uint64_t scale_bytes = int8 ? up256(uint64_t(P) * 4u) : 0;
  if (h_bytes + h16_bytes + xg16_bytes + 2 * scale_bytes > kHMaxBytes) return MOE_ERR_WORKSPACE;

  char* scratch = nullptr;
  int sms = 0;
  if (scratch_for_current_device(&scratch, &sms) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the status word and the stream-K counters must start at zero on every call
  if (cudaMemsetAsync(scratch, 0, kZeroBytes, s) != cudaSuccess) return MOE_ERR_CUDA;

  moe::ExpertFfnPlan plan{};
  plan.xg = xg;
  plan.offsets = expert_offsets;
  plan.active = active_experts;
  plan.num_active = num_active;
  plan.W_gate = W_gate;
  plan.W_up = W_up;
  plan.W_down = W_down;
  plan.s_gate = s_gate;
  plan.s_up = s_up;
  plan.s_down = s_down;
  plan.int8 = int8;
  plan.H = H;
  plan.I = I;
  plan.E = E;
  plan.P = P;
  plan.h = reinterpret_cast<uint16_t*>(scratch + kHOffset);
  plan.h16 = reinterpret_cast<uint16_t*>(scratch + kHOffset + h_bytes);
  plan.xg16 = reinterpret_cast<uint16_t*>(scratch + kHOffset + h_bytes + h16_bytes);
  plan.h_scale = reinterpret_cast<float*>(scratch + kHOffset + h_bytes + h16_bytes + xg16_bytes);
  plan.xg_scale = reinterpret_cast<float*>(scratch + kHOffset + h_bytes + h16_bytes + xg16_bytes + scale_bytes);
  plan.Y = Y;
  plan.partials = reinterpret_cast<float*>(scratch + kPartialsOffset);
  plan.partial_slot = moe::kPartialSlotFloats;
  plan.passes = moe::PassTokens{64, 64};
  plan.wait_ns = 0;
  plan.counters = reinterpret_cast<int32_t*>(scratch + kCountersOffset);
  plan.status = reinterpret_cast<int32_t*>(scratch);
  plan.num_ctas = sms < kCtas ? sms : kCtas;
  return moe::launch_expert_ffn(plan, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t moe_expert_ffn_noalloc_status(int32_t* status_out, moe_stream_t stream) {
  if (status_out == nullptr) return MOE_ERR_INVALID_ARG;
  char* scratch = nullptr;
  int sms = 0;
  if (scratch_for_current_device(&scratch, &sms) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t word = 0;  // pageable host memory: the copy completes before cudaStreamSynchronize returns
  if (cudaMemcpyAsync(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  *status_out = word;
  return MOE_OK;
}
