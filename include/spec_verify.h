/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding
 * verify-and-sample library.
 *
 * The operation (one decode step of speculative decoding, for a batch):
 * for every sequence b, K drafted tokens d_0..d_{K-1} are checked against the
 * target model's K+1 logit rows.
 *   - "Speculative decoding: draft models, VRAM economics, 3x" (tinycto.tv),
 *     section "Core mechanism": draft K tokens, score all positions in one
 *     target pass, accept in order with probability min(1, p(x)/q(x)), and on
 *     the first rejection draw a replacement from (p(x) - q(x))+ and drop the
 *     remaining drafts.
 *   - "after three fixes, Qwen3.5/3.6 MTP head reaches 1.4x on Apple Silicon"
 *     (deniz.in), sections "Verification under sampling was wrong" and
 *     "Truncation must match on both sides": greedy verification compares the
 *     draft with the target argmax; under sampling, both distributions get the
 *     same temperature, top-k and top-p truncation before the ratio is taken.
 *   - "MTPLX: native MTP speculative decoding on Apple Silicon", section 3.3:
 *     the output distribution equals plain sampling from the target.
 *
 * Exact rules used (readings where the pages are silent):
 *   p and q: softmax of logits/T restricted to the top_k best tokens
 *     (order: logit descending, token id ascending), renormalised, then to the
 *     shortest prefix of that order whose mass reaches top_p, renormalised
 *     again. top_k <= 0 or >= V: no top-k; top_p >= 1: no top-p.
 *   accept d_i iff u_i * q_i(d_i) < p_i(d_i), u_i uniform on the 2^-24 grid;
 *   n = number of leading accepted drafts;
 *   replacement (n < K): smallest token id j whose cumulative (p_n - q_n)+
 *     mass, in token-id order, exceeds v_n times the total; from p_n if that
 *     total is 0;
 *   bonus (n == K): the same inverse CDF over p_K with v_K;
 *   temperature == 0: greedy. a_i = argmax of target row i (lowest id on
 *     ties); n = leading i with d_i == a_i; emitted token a_n. Draft logits are
 *     not read for such a sequence.
 *   Uniforms: Philox4x32-10 (Salmon et al., SC'11) with key = (seed low, seed
 *   high) and counter = (i, b, offset low, offset high); word 0 -> u_i, word
 *   1 -> v_i, each as (word >> 8) * 2^-24. Randomness is a pure function of
 *   (seed, offset, b, i): a step can be replayed by passing the same values.
 *
 * Arithmetic: logits are read as bf16 or fp32 and converted to fp32 exactly.
 * Weights e = exp((z - max)/T) are fp32 (argument carried to ~2^-48); every
 * sum (normaliser, truncation mass, inverse-CDF scan) is an exact integer sum
 * of fixed-point weights, so results do not depend on summation order and
 * identical target and draft rows give identical p and q (always accepted).
 *
 * Memory: every pointer below is a device pointer unless stated otherwise,
 * contiguous, row-major, owned by the caller. The library allocates nothing
 * inside these calls and keeps no state between calls except per-device
 * kernel attributes set on first use. All calls are asynchronous on `stream`
 * (0 = legacy default stream) and never synchronise the host.
 *
 * Errors: argument errors return a status and launch nothing. Data errors in
 * a sequence (a NaN or +inf logit in a row the sequence uses, a row that is
 * -inf everywhere, a draft token outside [0, V), temperature < 0 or NaN,
 * top_p <= 0 or NaN, top_k < 0) are reported in band: out_n_accepted[b] = -1
 * and out_tokens[b, :] = -1. -inf logits are legal and mean probability 0.
 * A launch failure returns SV_ERR_CUDA.
 *
 * Limits: 1 <= B <= 65535, 1 <= K <= 16, 2 <= V <= 262144.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SV_BF16 = 0, SV_F32 = 1 } sv_dtype;

typedef enum {
  SV_OK = 0,
  SV_ERR_NULL = 1,       /* a required pointer is NULL */
  SV_ERR_SHAPE = 2,      /* B, K or V outside the limits */
  SV_ERR_DTYPE = 3,      /* unknown dtype */
  SV_ERR_WORKSPACE = 4,  /* workspace too small or misaligned */
  SV_ERR_CUDA = 5,       /* kernel launch or attribute call failed */
  SV_ERR_ALIGN = 6,      /* a pointer is not aligned to its element size */
  SV_ERR_SCRATCH = 7     /* (B, K) needs more than spec_verify_noalloc's fixed scratch */
} sv_status;

/* Bytes of device workspace spec_verify needs for (B, K). The workspace must
 * be 16-byte aligned and zero-filled before its first use (e.g. with
 * cudaMemsetAsync); every spec_verify call leaves it zero-filled again, so it
 * can be reused by later calls on the same stream. This includes a call in which
 * a bounded wait gave up (its sequences are reported as data errors, n = -1).
 * A call that returns SV_ERR_CUDA may have queued part of its kernels: zero the
 * workspace again (cudaMemsetAsync on the same stream) before reusing it. Two
 * calls that may run at the same time must not share a workspace. */
size_t spec_verify_workspace_bytes(int B, int K);

/* One verify-and-sample step for a batch.
 *   target_logits  [B, K+1, V] dtype: target rows for positions 0..K
 *   draft_logits   [B, K, V]   dtype: draft rows for positions 0..K-1; may be
 *                  NULL only if every temperature is 0 (greedy batch)
 *   draft_tokens   [B, K] int32: the drafted token ids
 *   temperature    [B] float: 0 selects greedy verification for that sequence
 *   top_k          [B] int32: 0 (or >= V) disables top-k
 *   top_p          [B] float: in (0, 1); >= 1 disables top-p
 *   philox_seed, philox_offset: host values (see above)
 *   out_tokens     [B, K+1] int32 (written): d_0..d_{n-1}, then the
 *                  replacement or bonus token, then -1
 *   out_n_accepted [B] int32 (written): n, or -1 on a data error
 *   workspace, workspace_bytes: see spec_verify_workspace_bytes()
 * Reads each logit row from HBM once. Returns SV_OK once the work is queued. */
sv_status spec_verify(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_tokens, const float* temperature,
                      const int32_t* top_k, const float* top_p, uint64_t philox_seed,
                      uint64_t philox_offset, int B, int K, int V, int32_t* out_tokens,
                      int32_t* out_n_accepted, void* workspace, size_t workspace_bytes,
                      void* stream /* cudaStream_t */);

/* One decode-loop step that keeps its state on the device, so that the step can
 * be captured once in a CUDA graph and replayed (the GPU-resident token handoff
 * of page "Optimizing on-device inference for Apple Silicon", decode section,
 * done the CUDA way). Same arguments and results as spec_verify, except:
 *   philox_offset [1] uint64 (device, 8-byte aligned): read as the Philox offset
 *                 of this step, then incremented by 1 once the step is done;
 *   next_token    [B] int32 (device, written; may be NULL): the last token the
 *                 step emitted for each sequence (out_tokens[b][n_b]), -1 on a
 *                 data error: the next step's input token;
 *   seq_len       [B] int32 (device, read-modify-write; may be NULL): increased
 *                 by n_b + 1, the tokens emitted (unchanged on a data error).
 * Nothing is read back to the host and nothing is allocated. The first call in
 * a process sets kernel attributes: make it before any stream capture. A
 * replayed graph reads the inputs from the same addresses each time: write the
 * next step's logits and drafts into them before replaying. Returns what
 * spec_verify returns, or SV_ERR_NULL / SV_ERR_ALIGN for the new pointers. */
sv_status spec_verify_step(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                           const int32_t* draft_tokens, const float* temperature,
                           const int32_t* top_k, const float* top_p, uint64_t philox_seed,
                           uint64_t* philox_offset, int B, int K, int V, int32_t* out_tokens,
                           int32_t* out_n_accepted, int32_t* next_token, int32_t* seq_len,
                           void* workspace, size_t workspace_bytes, void* stream /* cudaStream_t */);

/* spec_verify without a caller workspace. Same arguments, semantics and results as
 * spec_verify, minus the workspace: the workspace is a fixed array of
 * SV_NOALLOC_SCRATCH_BYTES bytes in the library's own device memory (a file-scope
 * __device__ array; one copy per device). The pages describe no such variant: it
 * exists for callers that cannot allocate device memory around the step, such as
 * plain C hosts without a device allocator, or runtimes that keep a fixed memory
 * budget and allow no allocation while a decode step runs.
 *   - Nothing is allocated: no cudaMalloc/cudaFree and no allocating library call.
 *   - Limit: spec_verify_workspace_bytes(B, K) must not exceed
 *     SV_NOALLOC_SCRATCH_BYTES (B <= 189 at K = 4, B <= 55 at K = 16); larger
 *     batches return SV_ERR_SCRATCH and launch nothing (use spec_verify with a
 *     workspace).
 *   - The scratch is zero when the library loads, and each call leaves it zero
 *     again; a call must run to completion before the next one starts. When
 *     spec_verify fails after queueing part of its work (SV_ERR_CUDA), this entry
 *     point queues a cudaMemsetAsync of the scratch on `stream` before returning the
 *     error, so the next call starts from zero (no allocation is involved).
 *   - The first call on a device looks up the scratch's device address with that
 *     device current (cudaGetSymbolAddress, which may load the module); make that
 *     first call outside any stream capture. Later calls reuse the cached address.
 *   - All calls on one device share the one scratch: two calls that may overlap
 *     (different streams, or host threads without ordering) race and corrupt each
 *     other's results. Order them on one stream or synchronise between them.
 * Returns the status spec_verify returns, or SV_ERR_SHAPE / SV_ERR_SCRATCH /
 * SV_ERR_CUDA (address lookup failed) before launching. */
#define SV_NOALLOC_SCRATCH_BYTES (1u << 20)
sv_status spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                              sv_dtype dtype, const int32_t* draft_tokens,
                              const float* temperature, const int32_t* top_k,
                              const float* top_p, uint64_t philox_seed, uint64_t philox_offset,
                              int B, int K, int V, int32_t* out_tokens, int32_t* out_n_accepted,
                              void* stream /* cudaStream_t */);

/* The truncated distribution of R independent rows, through the same device
 * code as spec_verify (a test and inspection hook): bf16 rows, 16-byte aligned,
 * R >= 16, through the key-histogram verify path's per-row code; otherwise, and
 * for the rows that code hands back, the cluster kernel.
 *   logits [R, V] dtype; temperature/top_k/top_p [R] (per row);
 *   out_probs [R, V] float (written): p(x) = weight(x) / kept mass for kept
 *   tokens, 0 elsewhere; for temperature == 0 rows, 1 at the argmax.
 * Limits: 1 <= R <= 2^20, V as above. Data errors write NaN to the row. */
sv_status spec_truncated_probs(const void* logits, sv_dtype dtype, int R, int V,
                               const float* temperature, const int32_t* top_k,
                               const float* top_p, float* out_probs, void* stream);

/* Draft-side sampler: draws d ~ q for a batch of draft rows, with the same
 * truncation and the same inverse-CDF rule as spec_verify, so that the
 * verifier's q is exactly the distribution the tokens came from.
 *   logits [B, K, V] dtype (row (b, i) = draft position i of sequence b);
 *   temperature/top_k/top_p [B] per sequence;
 *   uniform: sampling word of Philox at counter (i, b, offset) -- use an offset
 *   different from the one later passed to spec_verify;
 *   out_tokens [B, K] int32 (written), -1 on a data error in that row.
 * Limits: as spec_verify. */
sv_status spec_sample(const void* logits, sv_dtype dtype, int B, int K, int V,
                      const float* temperature, const int32_t* top_k, const float* top_p,
                      uint64_t philox_seed, uint64_t philox_offset, int32_t* out_tokens,
                      void* stream);

/* The Philox uniforms the library draws, as 24-bit grid indices (uniform =
 * index * 2^-24): out[(b * K1 + i) * 2 + 0] = acceptance index u_i of sequence
 * b, out[... + 1] = sampling index v_i, for b < B, i < K1. A test hook that
 * exposes the exact random stream of spec_verify and spec_sample.
 *   out [B * K1 * 2] uint32 (device, written). */
sv_status spec_philox_uniforms(uint64_t philox_seed, uint64_t philox_offset, int B, int K1,
                               uint32_t* out, void* stream);

/* Acceptance telemetry (page "Speculative decoding: draft models, VRAM economics,
 * 3x", acceptance rate and draft length; page "MTPLX", the tune command). Adds
 * the accepted-prefix lengths of one verify call to a caller-owned histogram:
 *   n_accepted [B] int32 (device): out_n_accepted of a spec_verify call
 *   hist       [K+2] uint64 (device, 8-byte aligned): hist[n] += #{b : n_b == n}
 *              for n in 0..K; hist[K+1] += data errors (n = -1) and any value
 *              outside [0, K]. The caller zeroes it to start a window; calls
 *              on one stream accumulate.
 * Limits: B >= 1, 1 <= K <= 16. Asynchronous on `stream`; allocates nothing.
 * Returns SV_ERR_SHAPE / SV_ERR_NULL / SV_ERR_ALIGN before launching, SV_ERR_CUDA
 * if the launch fails. */
sv_status spec_accept_histogram(const int32_t* n_accepted, int B, int K,
                                unsigned long long* hist, void* stream /* cudaStream_t */);

/* Human-readable name of a status code (static storage). */
const char* sv_status_string(sv_status status);

/* Library version as an integer: major * 10000 + minor * 100 + patch. */
int sv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
