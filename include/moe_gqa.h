/*
 * moe_gqa.h - C ABI of decode-phase grouped-query attention (libmoe.so, GB300 / sm_103a).
 *
 * The operation (HiNa-MoE, arXiv 2610.05123, §6.1 and Figure 9): each of B sequences has one
 * new query token, split into h_q heads of length d; its keys and values so far are split into
 * h_kv heads, each an l_seq x d matrix. A group of G = h_q / h_kv query heads shares one
 * key/value head; consecutive query heads share (query head hq reads key/value head hq / G,
 * a reading: the pages do not say which heads form a group). For every sequence b and query
 * head hq, with j = hq / G and n = seq_lens[b]:
 *     s_i = scale * sum_c q[b, hq, c] * K[b, j, i, c]          (i < n)
 *     out[b, hq, :] = bf16( sum_i softmax(s)_i * V[b, j, i, :] )
 * A sequence with n = 0 has nothing to attend to and gets out = 0.
 *
 * Numerics (the pages fix none): scores and softmax in fp32, the probabilities rounded to bf16
 * for the probability x value product, fp32 accumulation, the output rounded once to bf16
 * (round to nearest even). Against the exact result the error is within a few bf16 ulps of
 * the largest |V| entry attended to (see the parity tests).
 *
 * Conventions: those of moe.h (device pointers owned by the caller, asynchronous on `stream`,
 * host-side checks before any launch, no exceptions across the boundary, graph capturable).
 */
#ifndef MOE_GQA_H_
#define MOE_GQA_H_

#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Bytes of device workspace moe_gqa_decode needs (about 4.3 MB, independent of the sizes as long
 * as they are supported). Returns 0 when the sizes are invalid or unsupported. Pure host
 * computation.
 *
 * The workspace must be zero-filled before its first use (for example with cudaMemset); every
 * call leaves it ready for the next one, so calls need no clearing step between them. The first
 * 4 bytes are a status word that calls set and never clear: 4 means some seq_lens entry was
 * outside [0, L_cap] (that sequence's output is then 0; the workspace stays usable, zero the
 * word to reset it); 1-3 mean a kernel gave up a bounded wait (which does not happen in correct
 * operation; outputs undefined, and the whole workspace must be zero-filled again before reuse).
 */
size_t moe_gqa_workspace_size(int B, int h_q, int h_kv, int d, int L_cap);

/*
 * Decode-phase GQA attention over a key/value cache.
 *   q         [B, h_q, d] bf16 (row-major; the new token's query heads)
 *   k_cache   [B, h_kv, L_cap, d] bf16: rows i < seq_lens[b] of sequence b are its keys; rows
 *             at or past seq_lens[b] are never used (they may hold anything, even NaN)
 *   v_cache   [B, h_kv, L_cap, d] bf16, the values, same layout
 *   seq_lens  [B] int32 (device), 0 <= seq_lens[b] <= L_cap; the host never reads them
 *   scale     the softmax scale (1/sqrt(d) in the usual models); must be finite
 *   out       [B, h_q, d] bf16 out
 *   workspace >= moe_gqa_workspace_size(...) bytes (device, 256-byte aligned)
 * Supported: d = 128, 1 <= G = h_q / h_kv <= 16 (h_q a multiple of h_kv), 0 <= B <= 2048,
 * L_cap >= 1, B * h_kv * ceil(L_cap / 128) < 2^31; otherwise MOE_ERR_UNSUPPORTED (d, G, B, the
 * tile count) or MOE_ERR_INVALID_ARG. q, the caches and
 * out must be 16-byte aligned, seq_lens 4-byte aligned. B = 0 is a no-op.
 * Each key/value row attended to is read from memory once per call. The result is
 * deterministic for a given device and does not depend on timing.
 */
moe_status_t moe_gqa_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* seq_lens, int B, int h_q, int h_kv, int d, int L_cap,
                            float scale, uint16_t* out, void* workspace, size_t ws_bytes,
                            moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GQA_H_ */
