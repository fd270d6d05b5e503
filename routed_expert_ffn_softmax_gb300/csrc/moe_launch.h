// Host-side launch helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

// Launch with programmatic dependent launch enabled: the kernel may begin while its
// predecessor in the stream finishes; every kernel of this library waits for its
// predecessor (griddepcontrol.wait) before touching data the predecessor wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* counts,
                         int32_t* offsets, int32_t* sorted_token, int32_t* inv_pos, int32_t* active,
                         int32_t* num_active, int32_t* zero_words, int n_zero, cudaStream_t stream);

// The gathers warm the token rows in L2 before waiting for routing when they are at most this size.
constexpr int64_t kPrefetchMaxBytes = int64_t{4} << 20;

cudaError_t launch_gather(const uint16_t* x, int T, int H, int k, const int32_t* sorted_token, uint16_t* xg,
                          int num_sms, cudaStream_t stream);

cudaError_t launch_combine(const float* Y, const int32_t* inv_pos, const float* w, int T, int k, int H,
                           uint16_t* out, int num_sms, cudaStream_t stream);

// INT8 forward path: gather the token rows straight into their fp16 copy (see ExpertFfnPlan::xg16).
cudaError_t launch_gather_f16(const uint16_t* x, int T, int H, int P, const int32_t* sorted_token, uint16_t* xg16,
                              float* xg_scale, int num_sms, cudaStream_t stream);

// fp32 slots per CTA the expert kernels' stream-K partials need at 64-token passes (the larger of
// the two kernel families), and the CTA capacity the workspace provides.
constexpr int kPartialSlotFloats = 16384;
constexpr int kPartialCtas = 256;

// BF16 expert kernels: tokens per pass (64, 128, 192 or 256) of gate+up and of down, and the fp32 per
// stream-K partial slot a pass size needs (128 rows x the accumulator columns).
struct PassTokens {
  int gate_up, down;
};
// The passes a BF16 launch of P assignments over E experts takes: by the mean tokens per expert,
// unless set_pass_tokens forced a size. The workspace layout and the launch both call it.
PassTokens pass_tokens(int64_t P, int E);
void set_pass_tokens(int gate_up, int down);  // 0 = by batch shape
// Passes above 64 tokens run on CTA pairs, where down also holds two accumulator regions (two
// 128-row tiles per stage).
inline int64_t partial_slot_floats(int pass_tokens, bool gate_up) {
  return 128LL * ((gate_up || pass_tokens > 64) ? 2 : 1) * pass_tokens;
}

// Grouped expert FFN (gate+up then down) over an expert-sorted token block.
struct ExpertFfnPlan {
  const uint16_t* xg;  // [P, H]
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* num_active;
  const void* W_gate;
  const void* W_up;
  const void* W_down;
  const float* s_gate;
  const float* s_up;
  const float* s_down;
  // INT8 only, optional: residual-split parts of gate and up (W^Q + W^R) and their scales
  const void* W_gate_r;
  const void* W_up_r;
  const float* s_gate_r;
  const float* s_up_r;
  bool int8;
  int H, I, E, P;
  uint16_t* h;        // [P, I] scratch
  // INT8 only (scratch): fp16 copies of the token block and of h, and their row scales
  uint16_t* xg16;     // [P, H]
  uint16_t* h16;      // [P, I]
  float* xg_scale;    // [P]
  bool xg16_ready;    // INT8: xg16 / xg_scale were written by the gather (xg is then not read)
  float* h_scale;     // [P]
  float* Y;           // [P, H]
  float* partials;    // stream-K partial slots, [kPartialCtas][2][partial_slot]
  int64_t partial_slot;  // fp32 per slot (at least kPartialSlotFloats)
  PassTokens passes;     // BF16: tokens per pass; a size whose partials need more than partial_slot
                         // falls back to 64
  uint64_t wait_ns;      // BF16 single-CTA kernels: limit of their pipeline waits (0 = the normal 2 s)
  int32_t* counters;  // zeroed, kMaxCtas entries
  int32_t* status;
  int num_ctas;
};
cudaError_t launch_expert_ffn(const ExpertFfnPlan& plan, cudaStream_t stream);

// Decode-phase GQA attention (gqa_decode.cu) over a key/value cache [B, h_kv, L_cap, 128].
constexpr int kGqaMaxSeqs = 2048;  // sequences per call (the tile prefix lives in shared memory)
constexpr int kGqaSlotFloats = 16 * 128 + 2 * 16;  // one stream-K partial: o[16][128], m[16], l[16]
struct GqaPlan {
  const uint16_t* q;        // [B, h_q, 128] bf16
  const uint16_t* k_cache;  // [B, h_kv, L_cap, 128] bf16
  const uint16_t* v_cache;  // [B, h_kv, L_cap, 128] bf16
  const int32_t* seq_lens;  // [B]
  uint16_t* out;            // [B, h_q, 128] bf16
  float* partials;          // [kPartialCtas][2][kGqaSlotFloats]
  int32_t* counters;        // [kPartialCtas], zeroed
  int32_t* status;
  int B, h_q, h_kv, L_cap;
  float scale_log2;         // softmax scale * log2(e)
  int num_ctas;
};
cudaError_t launch_gqa_decode(const GqaPlan& plan, cudaStream_t stream);

// The whole decode step (routing, gate+up, down, combine) in one cooperative persistent launch
// (decode_step.cu), for small batches: at most kDecodeMaxT tokens and kDecodeMaxP assignments.
constexpr int kDecodeMaxT = 32;
constexpr int kDecodeMaxP = 256;
struct DecodeArgs {
  const uint16_t* x;     // [T, H] bf16
  const float* logits;   // [T, E]
  uint16_t* out;         // [T, H] bf16
  uint16_t* x16;         // INT8: [T, H / 128] records of 400 bytes, the token rows as digit planes (scratch)
  void* h;               // BF16: [P, I] bf16; INT8: [P, I / 128] records of 400 bytes (scratch)
  float* Y;              // [P, H] (scratch)
  float* partials;       // per CTA: its split-unit piece as (tag, value) pairs, [num CTAs][2][kPartialSlotFloats]
  int32_t* ccount;       // per 128-row block of H: units done, zero on entry, left zero
  int32_t* gbar;         // grid barrier: [0] arrivals (zero on entry, left zero), [1] release word
  int32_t* status;
  // the grid barrier opens after gridDim.x + grid_extra arrivals (grid_extra > 0 only in the
  // failure-detection test: it never opens, and every CTA's wait gives up after grid_wait_ns)
  int grid_extra;
  unsigned long long grid_wait_ns;
  // the routing tables (written by CTA 0)
  int32_t* ids;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_token;
  int32_t* inv_pos;
  int32_t* active;
  int32_t* num_active;
  int T, H, I, E, k;
};
struct DecodePlan {
  DecodeArgs args;
  const void* W_gate;
  const void* W_up;
  const void* W_down;
  const float* s_gate;
  const float* s_up;
  const float* s_down;
  bool int8;
  int H, I, E;
  int max_ctas;  // partial-slot capacity of the workspace
};
bool decode_step_supported(int T, int H, int I, int E, int k, bool int8);
cudaError_t launch_decode_step(const DecodePlan& plan, cudaStream_t stream);

// Weights of all experts as a 3-D tensor {K (contiguous), rows, E}; box = 128 bytes of `box_rows` rows
// of one expert (64 bf16 or 128 int8 elements), 128-byte swizzle.
bool encode_weights(CUtensorMap* map, const void* W, bool int8, int K, int rows, int E, int box_rows);

// Resolves cuTensorMapEncodeTiled through the runtime (no link-time libcuda).
using TensorMapEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                       const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                       CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                       CUtensorMapFloatOOBfill);
TensorMapEncodeFn tensor_map_encoder();

}  // namespace moe
