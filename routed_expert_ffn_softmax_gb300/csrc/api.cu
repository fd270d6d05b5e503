// C ABI of the routed-expert FFN library (declared in include/moe.h) and of decode-phase GQA
// attention (include/moe_gqa.h).
// Host-side argument checks, workspace layout and the launch sequence.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include <cmath>

#include "moe.h"
#include "moe_gqa.h"
#include "moe_launch.h"

namespace {

constexpr int kMaxCtas = moe::kPartialCtas;

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Workspace layout, in order (each section 256-byte aligned):
//   ctrl      status word (byte 0), the fused decode step's grid barrier (bytes 8..15), stream-K
//             counters at byte 256, the fused decode step's row-block counters at byte 2048
//   partials  stream-K partial slots
//   h         [P, I] bf16 (gate+up output)
//   INT8 only: h16 [P, I] fp16, xg16 [P, H] fp16, h_scale [P], xg_scale [P] f32
//   --- moe_ffn_forward only ---
//   ids, w, counts, offsets, sorted_token, inv_pos, active, num_active, xg [P,H] bf16, Y [P,H] f32,
//   INT8 only: hrec: the fused decode step's token records of 400 bytes (digit planes), [P, H/128] for
//   the token rows (T <= P of them used) then [P, I/128] for h
constexpr size_t kCtrlBytes = 4096;
constexpr size_t kGridBarrierOffset = 8;
constexpr size_t kCountersOffset = 256;
constexpr size_t kRowCountersOffset = 2048;
constexpr int kMaxRowBlocks = static_cast<int>((kCtrlBytes - kRowCountersOffset) / 4);  // H <= 65536
constexpr int kZeroWords = static_cast<int>((kCountersOffset + 4 * kMaxCtas) / 4);

struct Layout {
  size_t ctrl, partials, h, h16, xg16, h_scale, xg_scale, ids, w, counts, offsets, sorted_token, inv_pos, active,
      num_active, xg, Y, hrec, total;
  int64_t partial_slot;      // fp32 per stream-K partial slot
  moe::PassTokens passes;    // BF16 tokens per pass the slots are sized for
};

Layout layout(int64_t P, int H, int I, int E, bool int8) {
  Layout L{};
  L.passes = int8 ? moe::PassTokens{64, 64} : moe::pass_tokens(P, E);
  L.partial_slot = moe::kPartialSlotFloats;
  if (!int8) {
    const int64_t gu = moe::partial_slot_floats(L.passes.gate_up, true);
    const int64_t dn = moe::partial_slot_floats(L.passes.down, false);
    L.partial_slot = gu > L.partial_slot ? gu : L.partial_slot;
    L.partial_slot = dn > L.partial_slot ? dn : L.partial_slot;
  }
  size_t o = 0;
  L.ctrl = o;
  o += kCtrlBytes;
  L.partials = o;
  o = align_up(o + sizeof(float) * static_cast<size_t>(kMaxCtas) * 2 * static_cast<size_t>(L.partial_slot));
  L.h = o;
  o = align_up(o + 2 * static_cast<size_t>(P) * I);
  L.h16 = L.xg16 = L.h_scale = L.xg_scale = o;
  if (int8) {
    L.h16 = o;
    o = align_up(o + 2 * static_cast<size_t>(P) * I);
    L.xg16 = o;
    o = align_up(o + 2 * static_cast<size_t>(P) * H);
    L.h_scale = o;
    o = align_up(o + 4 * static_cast<size_t>(P));
    L.xg_scale = o;
    o = align_up(o + 4 * static_cast<size_t>(P));
  }
  L.ids = o;
  o = align_up(o + 4 * static_cast<size_t>(P));
  L.w = o;
  o = align_up(o + 4 * static_cast<size_t>(P));
  L.counts = o;
  o = align_up(o + 4 * static_cast<size_t>(E));
  L.offsets = o;
  o = align_up(o + 4 * static_cast<size_t>(E + 1));
  L.sorted_token = o;
  o = align_up(o + 4 * static_cast<size_t>(P));
  L.inv_pos = o;
  o = align_up(o + 4 * static_cast<size_t>(P));
  L.active = o;
  o = align_up(o + 4 * static_cast<size_t>(E));
  L.num_active = o;
  o = align_up(o + 4);
  L.xg = o;
  o = align_up(o + 2 * static_cast<size_t>(P) * H);
  L.Y = o;
  o = align_up(o + 4 * static_cast<size_t>(P) * H);
  L.hrec = o;
  if (int8) o = align_up(o + 400 * static_cast<size_t>(P) * (H / 128 + I / 128));
  L.total = o;
  return L;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Size checks shared by the entry points. Returns MOE_OK or the error to report.
moe_status_t check_sizes(int T, int H, int I, int E, int top_k, moe_wtype_t wtype) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || top_k < 1) return MOE_ERR_INVALID_ARG;
  if (wtype != MOE_W_BF16 && wtype != MOE_W_INT8_G128) return MOE_ERR_INVALID_ARG;
  if (top_k > E) return MOE_ERR_INVALID_ARG;
  if (E > 256) return MOE_ERR_UNSUPPORTED;
  const int m = wtype == MOE_W_INT8_G128 ? 128 : 8;
  if (H % m || I % m) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * top_k > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int sm_count() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev < kMaxDev) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return -1;
  if (dev < kMaxDev) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// moe_set_decode_step_policy: 0 = by batch shape, 1 = never, 2 = whenever the sizes allow it.
std::atomic<int> g_decode_policy{0};
// moe_test_expire_grid_barrier: extra arrivals the decode step's grid barrier waits for, and its wait limit.
std::atomic<int> g_grid_extra{0};
std::atomic<unsigned long long> g_grid_wait_ns{2000000000ull};
// moe_test_expert_wait_limit: limit of the BF16 single-CTA expert kernels' pipeline waits (0 = normal).
std::atomic<unsigned long long> g_expert_wait_ns{0};

// Whether moe_ffn_forward runs the fused one-launch decode step for these sizes: by batch shape
// (policy 0) INT8 weights while the batch has at most one assignment per two experts (T <= 8 at
// Qwen3-235B shapes), BF16 weights up to two tokens. Measured on GB300 against the separate
// launches (the same box, GB/s): INT8 3480 vs 2837 at T = 1, 5160 vs 4919 at T = 4, 5720 vs 5689
// at T = 8, behind at T = 16; BF16 at T = 1 5920 vs 5730 (Mixtral-8x7B), 5754 vs 5611
// (DeepSeek-V3), 6375 vs 6201 (Mixtral-8x22B), at T = 2 +0.7-2%, level at T = 4, behind at T = 8.
bool use_decode_step(int T, int H, int I, int E, int top_k, moe_wtype_t wtype, bool residual) {
  const int policy = g_decode_policy.load(std::memory_order_relaxed);
  if (policy == 1 || residual) return false;
  if (!moe::decode_step_supported(T, H, I, E, top_k, wtype == MOE_W_INT8_G128)) return false;
  if (H / 128 > kMaxRowBlocks) return false;
  if (policy == 2) return true;
  return wtype == MOE_W_INT8_G128 ? static_cast<int64_t>(T) * top_k * 2 <= E : T <= 2;
}

// Residual-split parts of gate and up (INT8 only); all null when the weights are not split.
struct Residual {
  const void* Wg = nullptr;
  const void* Wu = nullptr;
  const float* sg = nullptr;
  const float* su = nullptr;
};

bool residual_ok(const Residual& r) {
  return r.Wg && r.Wu && r.sg && r.su && aligned(r.Wg, 16) && aligned(r.Wu, 16) && aligned(r.sg, 4) &&
         aligned(r.su, 4);
}

moe_status_t run_expert_ffn(const uint16_t* xg, const int32_t* offsets, const int32_t* active,
                            const int32_t* num_active, const void* Wg, const void* Wu, const void* Wd,
                            const float* sg, const float* su, const float* sd, moe_wtype_t wtype, int H, int I,
                            int E, int P, float* Y, char* ws, cudaStream_t stream, bool xg16_ready = false,
                            const Residual& res = Residual{}) {
  const int sms = sm_count();
  if (sms < 1) return MOE_ERR_CUDA;
  const Layout L = layout(P, H, I, E, wtype == MOE_W_INT8_G128);
  moe::ExpertFfnPlan plan{};
  plan.xg = xg;
  plan.offsets = offsets;
  plan.active = active;
  plan.num_active = num_active;
  plan.W_gate = Wg;
  plan.W_up = Wu;
  plan.W_down = Wd;
  plan.s_gate = sg;
  plan.s_up = su;
  plan.s_down = sd;
  plan.W_gate_r = res.Wg;
  plan.W_up_r = res.Wu;
  plan.s_gate_r = res.sg;
  plan.s_up_r = res.su;
  plan.int8 = wtype == MOE_W_INT8_G128;
  plan.H = H;
  plan.I = I;
  plan.E = E;
  plan.P = P;
  plan.h = reinterpret_cast<uint16_t*>(ws + L.h);
  plan.h16 = reinterpret_cast<uint16_t*>(ws + L.h16);
  plan.xg16 = reinterpret_cast<uint16_t*>(ws + L.xg16);
  plan.h_scale = reinterpret_cast<float*>(ws + L.h_scale);
  plan.xg_scale = reinterpret_cast<float*>(ws + L.xg_scale);
  plan.xg16_ready = xg16_ready;
  plan.Y = Y;
  plan.partials = reinterpret_cast<float*>(ws + L.partials);
  plan.partial_slot = L.partial_slot;
  plan.passes = L.passes;
  plan.wait_ns = g_expert_wait_ns.load(std::memory_order_relaxed);
  plan.counters = reinterpret_cast<int32_t*>(ws + L.ctrl + kCountersOffset);
  plan.status = reinterpret_cast<int32_t*>(ws + L.ctrl);
  plan.num_ctas = sms < kMaxCtas ? sms : kMaxCtas;
  return cuda_status(moe::launch_expert_ffn(plan, stream));
}

bool weights_ok(const void* Wg, const void* Wu, const void* Wd, const float* sg, const float* su,
                const float* sd, moe_wtype_t wtype) {
  if (!Wg || !Wu || !Wd || !aligned(Wg, 16) || !aligned(Wu, 16) || !aligned(Wd, 16)) return false;
  if (wtype == MOE_W_INT8_G128 &&
      (!sg || !su || !sd || !aligned(sg, 4) || !aligned(su, 4) || !aligned(sd, 4)))
    return false;
  return true;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: outside what this library implements";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA call or kernel launch failed";
  }
  return "unknown moe_status_t";
}

size_t moe_workspace_size(int T, int H, int I, int E, int top_k, moe_wtype_t wtype) {
  if (check_sizes(T, H, I, E, top_k, wtype) != MOE_OK) return 0;
  return layout(static_cast<int64_t>(T) * top_k, H, I, E, wtype == MOE_W_INT8_G128).total;
}

moe_status_t moe_route_topk(const float* logits, int T, int E, int top_k, int32_t* topk_ids, float* topk_w,
                            int32_t* expert_counts, int32_t* expert_offsets, int32_t* sorted_token,
                            int32_t* inv_pos, int32_t* active_experts, int32_t* num_active,
                            moe_stream_t stream) {
  const moe_status_t sz = check_sizes(T, 8, 8, E, top_k, MOE_W_BF16);
  if (sz != MOE_OK) return sz;
  if (T == 0) return MOE_OK;
  const void* ptrs[] = {logits, topk_ids, topk_w, expert_counts, expert_offsets,
                        sorted_token, inv_pos, active_experts, num_active};
  for (const void* p : ptrs)
    if (!p || !aligned(p, 4)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_route(logits, T, E, top_k, topk_ids, topk_w, expert_counts, expert_offsets,
                                       sorted_token, inv_pos, active_experts, num_active, nullptr, 0,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_gather(const uint16_t* x, int T, int H, int top_k, const int32_t* sorted_token, uint16_t* xg,
                        moe_stream_t stream) {
  if (T < 0 || H < 8 || H % 8 || top_k < 1) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * top_k > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !sorted_token || !xg || !aligned(x, 16) || !aligned(xg, 16) || !aligned(sorted_token, 4))
    return MOE_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms < 1) return MOE_ERR_CUDA;
  return cuda_status(
      moe::launch_gather(x, T, H, top_k, sorted_token, xg, sms, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

moe_status_t expert_ffn_impl(const uint16_t* xg, const int32_t* expert_offsets, const int32_t* active_experts,
                             const int32_t* num_active, const void* W_gate, const void* W_up, const void* W_down,
                             const float* s_gate, const float* s_up, const float* s_down, moe_wtype_t wtype, int H,
                             int I, int E, int P, float* Y, void* workspace, size_t ws_bytes, moe_stream_t stream,
                             const Residual& res) {
  if (P < 0) return MOE_ERR_INVALID_ARG;
  const moe_status_t sz = check_sizes(P, H, I, E, 1, wtype);
  if (sz != MOE_OK) return sz;
  if (P == 0) return MOE_OK;
  if (!xg || !expert_offsets || !active_experts || !num_active || !Y || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(xg, 16) || !aligned(Y, 16) || !aligned(workspace, kAlign) || !aligned(expert_offsets, 4) ||
      !aligned(active_experts, 4) || !aligned(num_active, 4))
    return MOE_ERR_INVALID_ARG;
  if (!weights_ok(W_gate, W_up, W_down, s_gate, s_up, s_down, wtype)) return MOE_ERR_INVALID_ARG;
  const Layout L = layout(P, H, I, E, wtype == MOE_W_INT8_G128);
  if (ws_bytes < L.ids) return MOE_ERR_WORKSPACE;  // ctrl + partials + h (+ INT8 fp16 copies)
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws + L.ctrl, 0, kCountersOffset + 4 * kMaxCtas, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return run_expert_ffn(xg, expert_offsets, active_experts, num_active, W_gate, W_up, W_down, s_gate, s_up, s_down,
                        wtype, H, I, E, P, Y, ws, s, false, res);
}

}  // namespace

extern "C" {

moe_status_t moe_expert_ffn(const uint16_t* xg, const int32_t* expert_offsets, const int32_t* active_experts,
                            const int32_t* num_active, const void* W_gate, const void* W_up, const void* W_down,
                            const float* s_gate, const float* s_up, const float* s_down, moe_wtype_t wtype, int H,
                            int I, int E, int P, float* Y, void* workspace, size_t ws_bytes,
                            moe_stream_t stream) {
  return expert_ffn_impl(xg, expert_offsets, active_experts, num_active, W_gate, W_up, W_down, s_gate, s_up, s_down,
                         wtype, H, I, E, P, Y, workspace, ws_bytes, stream, Residual{});
}

moe_status_t moe_expert_ffn_residual(const uint16_t* xg, const int32_t* expert_offsets,
                                     const int32_t* active_experts, const int32_t* num_active, const void* W_gate,
                                     const void* W_up, const void* W_down, const float* s_gate, const float* s_up,
                                     const float* s_down, const void* Wr_gate, const void* Wr_up,
                                     const float* sr_gate, const float* sr_up, int H, int I, int E, int P, float* Y,
                                     void* workspace, size_t ws_bytes, moe_stream_t stream) {
  Residual r;
  r.Wg = Wr_gate;
  r.Wu = Wr_up;
  r.sg = sr_gate;
  r.su = sr_up;
  if (P > 0 && !residual_ok(r)) return MOE_ERR_INVALID_ARG;
  return expert_ffn_impl(xg, expert_offsets, active_experts, num_active, W_gate, W_up, W_down, s_gate, s_up, s_down,
                         MOE_W_INT8_G128, H, I, E, P, Y, workspace, ws_bytes, stream, r);
}

moe_status_t moe_combine(const float* Y, const int32_t* inv_pos, const float* topk_w, int T, int top_k, int H,
                         uint16_t* out, moe_stream_t stream) {
  if (T < 0 || H < 8 || H % 8 || top_k < 1) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * top_k > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!Y || !inv_pos || !topk_w || !out || !aligned(Y, 16) || !aligned(out, 16) || !aligned(inv_pos, 4) ||
      !aligned(topk_w, 4))
    return MOE_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms < 1) return MOE_ERR_CUDA;
  return cuda_status(
      moe::launch_combine(Y, inv_pos, topk_w, T, top_k, H, out, sms, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

moe_status_t ffn_forward_impl(const uint16_t* x, const float* logits, const void* W_gate, const void* W_up,
                              const void* W_down, const float* s_gate, const float* s_up, const float* s_down,
                              moe_wtype_t wtype, int T, int H, int I, int E, int top_k, uint16_t* out,
                              void* workspace, size_t ws_bytes, moe_stream_t stream, const Residual& res) {
  const moe_status_t sz = check_sizes(T, H, I, E, top_k, wtype);
  if (sz != MOE_OK) return sz;
  if (T == 0) return MOE_OK;
  if (!x || !logits || !out || !workspace || !aligned(x, 16) || !aligned(out, 16) || !aligned(logits, 4) ||
      !aligned(workspace, kAlign))
    return MOE_ERR_INVALID_ARG;
  if (!weights_ok(W_gate, W_up, W_down, s_gate, s_up, s_down, wtype)) return MOE_ERR_INVALID_ARG;
  const int P = T * top_k;
  const Layout L = layout(P, H, I, E, wtype == MOE_W_INT8_G128);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  const int sms = sm_count();
  if (sms < 1) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  auto I32 = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  int32_t* ids = I32(L.ids);
  float* w = reinterpret_cast<float*>(ws + L.w);
  int32_t* offsets = I32(L.offsets);
  int32_t* sorted_token = I32(L.sorted_token);
  int32_t* inv_pos = I32(L.inv_pos);
  int32_t* active = I32(L.active);
  int32_t* num_active = I32(L.num_active);
  uint16_t* xg = reinterpret_cast<uint16_t*>(ws + L.xg);
  float* Y = reinterpret_cast<float*>(ws + L.Y);

  const bool int8 = wtype == MOE_W_INT8_G128;
  if (use_decode_step(T, H, I, E, top_k, wtype, res.Wg != nullptr)) {
    moe::DecodePlan plan{};
    moe::DecodeArgs& a = plan.args;
    a.x = x;
    a.logits = logits;
    a.out = out;
    a.x16 = reinterpret_cast<uint16_t*>(ws + L.hrec);
    a.h = int8 ? static_cast<void*>(ws + L.hrec + 400 * static_cast<size_t>(P) * (H / 128))
               : static_cast<void*>(ws + L.h);
    a.Y = Y;
    a.partials = reinterpret_cast<float*>(ws + L.partials);
    a.ccount = I32(L.ctrl + kRowCountersOffset);
    a.gbar = I32(L.ctrl + kGridBarrierOffset);
    a.status = I32(L.ctrl);
    a.ids = ids;
    a.w = w;
    a.counts = I32(L.counts);
    a.offsets = offsets;
    a.sorted_token = sorted_token;
    a.inv_pos = inv_pos;
    a.active = active;
    a.num_active = num_active;
    a.T = T;
    a.H = H;
    a.I = I;
    a.E = E;
    a.k = top_k;
    a.grid_extra = g_grid_extra.load(std::memory_order_relaxed);
    a.grid_wait_ns = g_grid_wait_ns.load(std::memory_order_relaxed);
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
    plan.max_ctas = sms < kMaxCtas ? sms : kMaxCtas;
    return cuda_status(moe::launch_decode_step(plan, s));
  }
  cudaError_t e = moe::launch_route(logits, T, E, top_k, ids, w, I32(L.counts), offsets, sorted_token, inv_pos,
                                    active, num_active, I32(L.ctrl), kZeroWords, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (int8)  // the INT8 kernels read only the fp16 copy of the gathered rows: write it directly
    e = moe::launch_gather_f16(x, T, H, P, sorted_token, reinterpret_cast<uint16_t*>(ws + L.xg16),
                               reinterpret_cast<float*>(ws + L.xg_scale), sms, s);
  else
    e = moe::launch_gather(x, T, H, top_k, sorted_token, xg, sms, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const moe_status_t st = run_expert_ffn(xg, offsets, active, num_active, W_gate, W_up, W_down, s_gate, s_up,
                                         s_down, wtype, H, I, E, P, Y, ws, s, int8, res);
  if (st != MOE_OK) return st;
  return cuda_status(moe::launch_combine(Y, inv_pos, w, T, top_k, H, out, sms, s));
}

}  // namespace

extern "C" {

moe_status_t moe_ffn_forward(const uint16_t* x, const float* logits, const void* W_gate, const void* W_up,
                             const void* W_down, const float* s_gate, const float* s_up, const float* s_down,
                             moe_wtype_t wtype, int T, int H, int I, int E, int top_k, uint16_t* out,
                             void* workspace, size_t ws_bytes, moe_stream_t stream) {
  return ffn_forward_impl(x, logits, W_gate, W_up, W_down, s_gate, s_up, s_down, wtype, T, H, I, E, top_k, out,
                          workspace, ws_bytes, stream, Residual{});
}

moe_status_t moe_set_decode_step_policy(int policy) {
  if (policy < 0 || policy > 2) return MOE_ERR_INVALID_ARG;
  g_decode_policy.store(policy, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status_t moe_set_expert_pass_tokens(int gate_up, int down) {
  auto ok = [](int n) { return n == 0 || n == 64 || n == 128 || n == 192 || n == 256; };
  if (!ok(gate_up) || !ok(down)) return MOE_ERR_INVALID_ARG;
  moe::set_pass_tokens(gate_up, down);
  return MOE_OK;
}

moe_status_t moe_test_expert_wait_limit(uint64_t wait_ns) {
  if (wait_ns != 0 && (wait_ns < 100ull || wait_ns > 2000000000ull)) return MOE_ERR_INVALID_ARG;
  g_expert_wait_ns.store(wait_ns, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status_t moe_test_expire_grid_barrier(int enable, uint64_t wait_ns) {
  if (enable != 0 && enable != 1) return MOE_ERR_INVALID_ARG;
  if (enable && (wait_ns < 1000ull || wait_ns > 2000000000ull)) return MOE_ERR_INVALID_ARG;
  g_grid_wait_ns.store(enable ? wait_ns : 2000000000ull, std::memory_order_relaxed);
  g_grid_extra.store(enable, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_ffn_forward_launches(int T, int H, int I, int E, int top_k, moe_wtype_t wtype) {
  if (check_sizes(T, H, I, E, top_k, wtype) != MOE_OK) return -1;
  if (T == 0) return 0;
  if (use_decode_step(T, H, I, E, top_k, wtype, false)) return 1;
  const int route = (T <= 64 && static_cast<int64_t>(T) * top_k <= 1024) ? 1 : 2;
  return route + 1 + (wtype == MOE_W_INT8_G128 ? 3 : 2) + 1;
}

moe_status_t moe_ffn_forward_residual(const uint16_t* x, const float* logits, const void* W_gate, const void* W_up,
                                      const void* W_down, const float* s_gate, const float* s_up,
                                      const float* s_down, const void* Wr_gate, const void* Wr_up,
                                      const float* sr_gate, const float* sr_up, int T, int H, int I, int E,
                                      int top_k, uint16_t* out, void* workspace, size_t ws_bytes,
                                      moe_stream_t stream) {
  Residual r;
  r.Wg = Wr_gate;
  r.Wu = Wr_up;
  r.sg = sr_gate;
  r.su = sr_up;
  if (T > 0 && !residual_ok(r)) return MOE_ERR_INVALID_ARG;
  return ffn_forward_impl(x, logits, W_gate, W_up, W_down, s_gate, s_up, s_down, MOE_W_INT8_G128, T, H, I, E, top_k,
                          out, workspace, ws_bytes, stream, r);
}

// ---------------------------------------------------------------- decode GQA attention
namespace {

constexpr size_t kGqaPartialBytes = sizeof(float) * static_cast<size_t>(kMaxCtas) * 2 * moe::kGqaSlotFloats;

moe_status_t gqa_check(int B, int h_q, int h_kv, int d, int L_cap) {
  if (B < 0 || h_q < 1 || h_kv < 1 || d < 1 || L_cap < 1 || h_q % h_kv) return MOE_ERR_INVALID_ARG;
  if (d != 128 || h_q / h_kv > 16 || B > moe::kGqaMaxSeqs) return MOE_ERR_UNSUPPORTED;
  // the kernel counts key tiles of 128 rows over all (sequence, key/value head) pairs in 32 bits
  if (static_cast<int64_t>(B) * h_q > INT32_MAX || static_cast<int64_t>(B) * h_kv * ((L_cap + 127) / 128) > INT32_MAX)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

size_t moe_gqa_workspace_size(int B, int h_q, int h_kv, int d, int L_cap) {
  if (gqa_check(B, h_q, h_kv, d, L_cap) != MOE_OK) return 0;
  return kCtrlBytes + align_up(kGqaPartialBytes);
}

moe_status_t moe_gqa_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* seq_lens, int B, int h_q, int h_kv, int d, int L_cap, float scale,
                            uint16_t* out, void* workspace, size_t ws_bytes, moe_stream_t stream) {
  const moe_status_t sz = gqa_check(B, h_q, h_kv, d, L_cap);
  if (sz != MOE_OK) return sz;
  if (!std::isfinite(scale)) return MOE_ERR_INVALID_ARG;
  if (B == 0) return MOE_OK;
  if (!q || !k_cache || !v_cache || !seq_lens || !out || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(seq_lens, 4) || !aligned(workspace, kAlign))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_gqa_workspace_size(B, h_q, h_kv, d, L_cap)) return MOE_ERR_WORKSPACE;
  const int sms = sm_count();
  if (sms < 1) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  // No clearing launch here: the merge counters are left zero by every call, so consecutive calls
  // are back-to-back kernels that overlap launch and prologue (programmatic dependent launch).
  moe::GqaPlan plan{};
  plan.q = q;
  plan.k_cache = k_cache;
  plan.v_cache = v_cache;
  plan.seq_lens = seq_lens;
  plan.out = out;
  plan.partials = reinterpret_cast<float*>(ws + kCtrlBytes);
  plan.counters = reinterpret_cast<int32_t*>(ws + kCountersOffset);
  plan.status = reinterpret_cast<int32_t*>(ws);
  plan.B = B;
  plan.h_q = h_q;
  plan.h_kv = h_kv;
  plan.L_cap = L_cap;
  plan.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  plan.num_ctas = sms < kMaxCtas ? sms : kMaxCtas;
  return cuda_status(moe::launch_gqa_decode(plan, s));
}

}  // extern "C"
