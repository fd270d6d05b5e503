/*
 * moe.h - C ABI of the routed-expert MoE FFN library for the GB300 (sm_103a).
 *
 * The operation (HiNa-MoE, arXiv 2610.05123):
 *   - a gating function routes each token to a small subset of experts (§2.1;
 *     Top-2 / Top-8 in §8.1 Table 3), read here as softmax over the E router
 *     logits, top-k, renormalised over the kept k;
 *   - the routed tokens are gathered into a per-expert intermediate matrix I
 *     (§4.1, Figure 5);
 *   - each expert computes FFN(I) = SiLU(I x W_gate) (.) (I x W_up) x W_down
 *     (§4.1, the FFN equation) with bf16 inputs and fp32 accumulation (§4.2.1);
 *     h = SiLU(g) * u is rounded to bf16 before the down projection;
 *   - the expert outputs are combined per token with the routing weights and
 *     written back row-major (§4.1, third layout transformation).
 * Expert weights stay in the general row-major layout, one output row per line
 * with the reduction contiguous (§2.2 Figure 3, "general layout"): W_gate and
 * W_up are [E, I, H], W_down is [E, H, I]. The INT8 variant (§8.1, Figure 11,
 * symmetric group-wise quantisation) stores int8 weights in the same layout
 * plus fp32 scales, one per 128 consecutive reduction elements:
 * s_gate/s_up [E, I, H/128], s_down [E, H, I/128]; w = q * s.
 *
 * Conventions shared by every entry point:
 *   - Every array pointer is a DEVICE pointer owned by the caller. The library
 *     allocates no memory and keeps no device state between calls, with one
 *     exception: moe_expert_ffn_noalloc uses a fixed scratch array inside the
 *     library (see there), which persists from load until the process exits.
 *   - Exception: the expert weights and scales (W_gate, W_up, W_down, s_gate,
 *     s_up, s_down) may also live in host memory the GPU can address (pinned or
 *     registered; on a GB300 node the Grace LPDDR5X), passed by that memory's
 *     device-visible address. The kernels then stream them in place over
 *     NVLink-C2C with the same results (bit-identical) as from HBM: the pages
 *     keep routed experts in CPU memory when they exceed GPU memory (§1) in
 *     one general layout that CPU and GPU share (§3.1). Throughput is then
 *     bounded by the host link instead of HBM.
 *   - bf16 arrays are passed as uint16_t bit patterns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; 0 = legacy
 *     default stream) and never synchronises the host. Calls on one stream may
 *     be captured in a CUDA graph.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns an error and launches nothing. A failed launch returns
 *     MOE_ERR_CUDA. No C++ exception crosses this boundary.
 *   - T = 0 is a valid no-op that returns MOE_OK.
 *   - Sizes: 1 <= top_k <= E <= 256. BF16: H and I multiples of 8.
 *     INT8: H and I multiples of 128. Device pointers must be 16-byte aligned;
 *     the workspace must be 256-byte aligned.
 *   - Router logits must be finite; with a NaN logit the routing is still a
 *     valid set of distinct experts but is otherwise unspecified.
 *
 * Notation: T tokens, H hidden size, I intermediate size, E experts,
 * P = T * top_k token-expert assignments.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so this header needs no CUDA header. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size, misalignment */
  MOE_ERR_UNSUPPORTED = 2, /* valid request outside what this build implements (E > 256, ...) */
  MOE_ERR_WORKSPACE = 3,   /* workspace smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4         /* a CUDA call or kernel launch failed */
} moe_status_t;

typedef enum {
  MOE_W_BF16 = 0,     /* bf16 weights, scale pointers ignored */
  MOE_W_INT8_G128 = 1 /* int8 weights + fp32 scales per 128 reduction elements */
} moe_wtype_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status_t status);

/*
 * Bytes of device workspace that moe_ffn_forward and moe_expert_ffn need for
 * these sizes (the same figure serves both). Returns 0 when the sizes are
 * invalid. Pure host computation; touches no device.
 *
 * A workspace must be zero-filled before its first use (cudaMemset to 0); every
 * call leaves its counters zero again, so it stays usable call after call.
 *
 * The first 4 bytes of a workspace are a status word: a kernel that gives up
 * on a bounded wait (which does not happen in correct operation) writes a
 * nonzero code there and returns early, leaving the outputs undefined. Each
 * moe_ffn_forward / moe_expert_ffn call clears it at its start. After a
 * nonzero status, zero the whole workspace again before the next call (a call
 * that gave up may leave counters behind).
 */
size_t moe_workspace_size(int T, int H, int I, int E, int top_k, moe_wtype_t wtype);

/*
 * Routing (HiNa-MoE §2.1, §8.1 Table 3; softmax -> top-k -> renormalise).
 *   logits          [T, E] f32, row-major
 *   topk_ids        [T, top_k] i32 out: slot j holds the j-th largest logit's expert,
 *                   ties broken toward the lower expert id
 *   topk_w          [T, top_k] f32 out: w_j = exp(l_j - m) / sum_i exp(l_i - m) over
 *                   the kept experts, m = the largest kept logit
 *   expert_counts   [E] i32 out: tokens routed to each expert
 *   expert_offsets  [E + 1] i32 out: exclusive prefix sum of expert_counts
 *   sorted_token    [P] i32 out: token of each assignment in (expert, token) order,
 *                   i.e. expert e's tokens in ascending order at
 *                   [expert_offsets[e], expert_offsets[e + 1])
 *   inv_pos         [T, top_k] i32 out: position of assignment (t, j) in sorted_token
 *   active_experts  [E] i32 out: experts with expert_counts > 0, ascending; entries
 *                   past *num_active are left unwritten
 *   num_active      [1] i32 out
 * Integer outputs are deterministic and bit-identical to the definition above.
 */
moe_status_t moe_route_topk(const float* logits, int T, int E, int top_k, int32_t* topk_ids,
                            float* topk_w, int32_t* expert_counts, int32_t* expert_offsets,
                            int32_t* sorted_token, int32_t* inv_pos, int32_t* active_experts,
                            int32_t* num_active, moe_stream_t stream);

/*
 * Token gather into the per-expert intermediate matrix (HiNa-MoE §4.1, Figure 5):
 *   xg[p, :] = x[sorted_token[p], :] for p < P = T * top_k.
 *   x  [T, H] bf16, row-major;  xg [P, H] bf16 out, row-major, expert-sorted.
 * The rows of one expert are contiguous, which is the operand layout the expert
 * kernels load tile by tile (the first layout transformation of §4.1 is done by
 * this copy: the token block is reshaped, the weights are not).
 */
moe_status_t moe_gather(const uint16_t* x, int T, int H, int top_k, const int32_t* sorted_token,
                        uint16_t* xg, moe_stream_t stream);

/*
 * Expert FFN over the gathered token block (HiNa-MoE §4.1 FFN equation):
 *   for every active expert e and every row p of its block
 *   [expert_offsets[e], expert_offsets[e + 1]):
 *     h[p, i] = bf16( SiLU(g) * u ),  g = sum_c xg[p, c] W_gate[e, i, c],
 *                                      u = sum_c xg[p, c] W_up[e, i, c]   (fp32)
 *     Y[p, r] = sum_i h[p, i] W_down[e, r, i]                              (fp32)
 *   xg              [P, H] bf16 (expert-sorted, as written by moe_gather)
 *   expert_offsets  [E + 1] i32, active_experts [E] i32, num_active [1] i32 (device,
 *                   as written by moe_route_topk; the host never reads them)
 *   W_gate, W_up    [E, I, H] bf16 or int8;  W_down [E, H, I] bf16 or int8
 *   s_gate, s_up    [E, I, H/128] f32;  s_down [E, H, I/128] f32 (INT8 only, else ignored)
 *   P               = T * top_k, the number of rows of xg and Y
 *   Y               [P, H] f32 out, expert-sorted rows
 *   workspace       >= moe_workspace_size(T, H, I, E, top_k, wtype) bytes (device)
 * Only the weights of active experts are read. BF16 weights stream once per pass of an
 * expert's tokens: 64-token passes when the mean tokens per expert P / E is at most 40,
 * 128 up to 96, 192 or 256 above (moe_set_expert_pass_tokens can force a size). At 128- to
 * 256-token passes (on CTA pairs) an expert with more tokens than one pass has them split
 * evenly over up to 8 passes that run the same weight blocks side by side, so its weights
 * come from HBM once and from L2 for the others (up to 8 passes' worth of tokens per expert;
 * more take further rounds). INT8 weights stream once per 16 or 32 tokens.
 * The result is deterministic for a given device and pass size.
 */
moe_status_t moe_expert_ffn(const uint16_t* xg, const int32_t* expert_offsets,
                            const int32_t* active_experts, const int32_t* num_active,
                            const void* W_gate, const void* W_up, const void* W_down,
                            const float* s_gate, const float* s_up, const float* s_down,
                            moe_wtype_t wtype, int H, int I, int E, int P, float* Y,
                            void* workspace, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_expert_ffn without a workspace, for callers that cannot allocate device memory when
 * they call this library (for example a plugin inside another runtime whose device memory
 * belongs to that runtime's pool, or a decode loop that must not call cudaMalloc mid-step).
 * The paper has no counterpart of this entry point; it changes only who owns the scratch.
 *   Computes exactly what moe_expert_ffn computes, with the same arguments minus the
 *   workspace; the result may differ from moe_expert_ffn's only in fp32 summation order
 *   when the device has more than 160 SMs.
 *   Scratch: one fixed 48 MiB array inside this library, reserved on every GPU that loads
 *   the library until the process exits. P * I * 2 bytes (the bf16 intermediate h; for
 *   INT8 weights P * (4 * I + 2 * H + 8) bytes) must fit in about 28 MiB of it; larger
 *   requests return MOE_ERR_WORKSPACE and launch nothing.
 *   All calls share that array and it keeps the last call's contents: calls whose kernels
 *   overlap on one GPU (several streams or host threads) race and give wrong results.
 *   The first call on a device looks up the array's device address with that device
 *   current and keeps it for the life of the process: make that first call before any
 *   stream capture starts on the device, and do not reset the device (cudaDeviceReset)
 *   or switch it to another context between calls.
 *   A kernel that gives up on a bounded wait records a nonzero code in the array's status
 *   word; read it with moe_expert_ffn_noalloc_status. Each call clears it at its start.
 *   Calls no cudaMalloc/cudaFree and no allocating library routine.
 */
moe_status_t moe_expert_ffn_noalloc(const uint16_t* xg, const int32_t* expert_offsets,
                                    const int32_t* active_experts, const int32_t* num_active,
                                    const void* W_gate, const void* W_up, const void* W_down,
                                    const float* s_gate, const float* s_up, const float* s_down,
                                    moe_wtype_t wtype, int H, int I, int E, int P, float* Y,
                                    moe_stream_t stream);

/*
 * The status word of moe_expert_ffn_noalloc's scratch, as the last call on `stream` left it:
 * waits until the stream's work so far is done, then copies the 4-byte word to *status_out
 * (0 = no kernel gave up a wait). Allocates nothing. The paper has no counterpart.
 * Returns MOE_ERR_INVALID_ARG for a null status_out, MOE_ERR_CUDA if the copy fails.
 */
moe_status_t moe_expert_ffn_noalloc_status(int32_t* status_out, moe_stream_t stream);

/*
 * Routing-weighted combine back to row-major token order (HiNa-MoE §4.1, third
 * layout transformation):
 *   out[t, r] = bf16( sum_{j < top_k} topk_w[t, j] * Y[inv_pos[t, j], r] ),
 *   summed in fp32 in slot order j = 0, 1, ... (deterministic, no atomics).
 *   Y [P, H] f32;  inv_pos, topk_w [T, top_k];  out [T, H] bf16.
 */
moe_status_t moe_combine(const float* Y, const int32_t* inv_pos, const float* topk_w, int T,
                         int top_k, int H, uint16_t* out, moe_stream_t stream);

/*
 * The whole routed-expert FFN in one call: route -> gather -> expert FFN -> combine.
 *   x [T, H] bf16;  logits [T, E] f32;  weights and scales as in moe_expert_ffn;
 *   out [T, H] bf16;  workspace >= moe_workspace_size(T, H, I, E, top_k, wtype).
 * The routing, the gathered block, h and Y live in the workspace; the host never
 * learns the routing, so the call is free of host synchronisation.
 * It runs the routing, gather, tensor-core expert kernels and combine as separate launches
 * (linked by programmatic dependent launch), except for INT8 weights while the batch has at
 * most one assignment per two experts (2 * T * top_k <= E) and BF16 weights up to two tokens
 * (T <= 2): that step runs as ONE cooperative kernel that routes, streams both projections on
 * CUDA-core dot products (INT8: integer) and combines (measured faster on GB300 there, level
 * or slower at larger batches). moe_set_decode_step_policy can force either way for
 * small decode batches (T <= 32, T * top_k <= 256, H <= 16384, I <= 32768, H and I multiples
 * of 128, for INT8 multiples of 512). Both give results within the same tolerance of the
 * definition; the routing tables in the workspace are the same.
 */
moe_status_t moe_ffn_forward(const uint16_t* x, const float* logits, const void* W_gate,
                             const void* W_up, const void* W_down, const float* s_gate,
                             const float* s_up, const float* s_down, moe_wtype_t wtype, int T,
                             int H, int I, int E, int top_k, uint16_t* out, void* workspace,
                             size_t ws_bytes, moe_stream_t stream);

/*
 * Which implementation moe_ffn_forward uses (process-wide; the default is 0):
 *   0  by batch shape (the one-launch step for INT8 weights with 2 * T * top_k <= E and for
 *      BF16 weights with T <= 2, else the separate launches);
 *   1  never the one-launch decode step;
 *   2  the one-launch decode step whenever the sizes allow it.
 * Returns MOE_ERR_INVALID_ARG for any other value. Affects only later calls.
 */
moe_status_t moe_set_decode_step_policy(int policy);

/*
 * Tokens per pass of the BF16 expert kernels, gate+up and down separately: 64, 128, 192 or 256,
 * or 0 for the rule of moe_expert_ffn (the default). A tuning and test control; the paper
 * has no counterpart. Process-wide, affects only later calls. moe_workspace_size sizes the
 * stream-K partial slots for the sizes in force when it is called; a call whose workspace
 * was sized for smaller passes runs 64-token passes instead. Results differ between pass
 * sizes only in fp32 summation order. Returns MOE_ERR_INVALID_ARG for other values.
 */
moe_status_t moe_set_expert_pass_tokens(int gate_up, int down);

/*
 * Failure-detection test hook; the paper has no counterpart. While enabled (enable = 1), the
 * one-launch decode step's grid-wide barrier waits for one more CTA than the launch has, so it
 * never opens: every CTA gives up after wait_ns nanoseconds (1 us .. 2 s), records status 5 in
 * the workspace status word, and the kernel runs to its end and returns (outputs undefined; the
 * GPU and the context stay usable). Zero the workspace before its next use, as after any nonzero
 * status. enable = 0 restores the normal barrier and its 2 s limit. Process-wide; affects only
 * later calls. Returns MOE_ERR_INVALID_ARG for other values.
 */
moe_status_t moe_test_expire_grid_barrier(int enable, uint64_t wait_ns);

/*
 * Failure-detection test hook; the paper has no counterpart. wait_ns (100 ns .. 2 s, or 0 for the
 * normal 2 s) limits the pipeline waits of the BF16 expert kernels that run on single CTAs (passes of
 * 64 tokens): a wait for a tile or an accumulator that runs out records a nonzero status in the
 * workspace status word, the CTA's MMA issuer stops, its producer drains the copies it issued (those
 * waits keep the full limit, so no copy outlives its CTA), and the kernel returns (outputs undefined;
 * the GPU and the context stay usable). Zero the workspace before its next use. Process-wide; affects
 * only later calls. Returns MOE_ERR_INVALID_ARG for other values.
 */
moe_status_t moe_test_expert_wait_limit(uint64_t wait_ns);

/*
 * Kernels one moe_ffn_forward call launches for these sizes under the current policy
 * (1 for the one-launch decode step), or -1 when the sizes are invalid. Host only.
 */
int moe_ffn_forward_launches(int T, int H, int I, int E, int top_k, moe_wtype_t wtype);

/*
 * Residual-split INT8 experts (RapidMoE, arXiv 2610.01265, "Residual-Split Representation" and
 * "GLU Architecture Adoption"): gate and up are held as a low-precision part W^Q and the quantised
 * residual W^R of W - W^Q, the high-precision weight being W^H = W^Q + W^R; the gate and up
 * preactivations are W^Q x + W^R x, summed before SiLU. Down keeps one separately quantised copy
 * (the pages' "dual quantization" of down_proj). Here every part is symmetric group-128 INT8:
 *   W_gate, W_up    [E, I, H] int8: W^Q;  s_gate, s_up [E, I, H/128] f32 its scales
 *   Wr_gate, Wr_up  [E, I, H] int8: W^R;  sr_gate, sr_up [E, I, H/128] f32 its scales
 *   W_down          [E, H, I] int8;       s_down [E, H, I/128] f32
 * i.e. w = q * s + qr * sr for gate and up. Everything else (sizes, workspace: the INT8 figure of
 * moe_workspace_size, conventions, the host-memory option for weights) is as in
 * moe_expert_ffn / moe_ffn_forward with MOE_W_INT8_G128; the gate and up weight stream doubles.
 * All residual pointers must be non-null (16-byte aligned parts, 4-byte aligned scales).
 */
moe_status_t moe_expert_ffn_residual(const uint16_t* xg, const int32_t* expert_offsets,
                                     const int32_t* active_experts, const int32_t* num_active,
                                     const void* W_gate, const void* W_up, const void* W_down,
                                     const float* s_gate, const float* s_up, const float* s_down,
                                     const void* Wr_gate, const void* Wr_up, const float* sr_gate,
                                     const float* sr_up, int H, int I, int E, int P, float* Y,
                                     void* workspace, size_t ws_bytes, moe_stream_t stream);

moe_status_t moe_ffn_forward_residual(const uint16_t* x, const float* logits, const void* W_gate,
                                      const void* W_up, const void* W_down, const float* s_gate,
                                      const float* s_up, const float* s_down, const void* Wr_gate,
                                      const void* Wr_up, const float* sr_gate, const float* sr_up,
                                      int T, int H, int I, int E, int top_k, uint16_t* out,
                                      void* workspace, size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
