/* spec_lm_head.h — LM-head logits on the tensor cores, and the verify step fed
 * from hidden states (the fused LM-head + verify row of this library).
 *
 * What the pages define. "Apple Silikon İçin Cihaz Üstü Çıkarımı Optimize Etme"
 * (perplexity.coolkeypoint.com), decode section: every decode step ends by
 * choosing the next token from the position's logit row, the output projection
 * z = h . W^T of its final hidden state h against the LM-head weight W. Its
 * section on the limits of further optimisation reports that fusing the output
 * projection with token selection was tried there. The verify step that consumes
 * the rows is spec_verify (include/spec_verify.h).
 *
 * The GEMM kernel runs on the 5th-generation tensor cores: tcgen05.mma with
 * TMA-staged operands (128-byte swizzle) and a TMEM accumulator. Its logits are
 * checked against the float64 oracle within the fp32 accumulation bound, and the
 * verify step fed from it against the oracle's verify on those logits. For a
 * greedy batch the projection and the token choice are fused: the GEMM's
 * epilogue keeps only each row's first maximum, so no logit row is written.
 */
#ifndef SPEC_LM_HEAD_H
#define SPEC_LM_HEAD_H

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* logits[M][N] = hidden[M][d] . weight[N][d]^T, accumulated in fp32.
 *   hidden  [M][d] bf16, row-major, device memory, 16-byte aligned
 *   weight  [N][d] bf16, row-major (row v = token v's LM-head vector), device,
 *           16-byte aligned
 *   logits  [M][N] fp32, row-major, device, caller-owned, 4-byte aligned
 *   flag    [1] int32, device, caller-owned: set to 1 when a pipeline wait of the
 *           kernel timed out (the logits are then undefined); never cleared here.
 *           The caller zeroes it before the call and checks it afterwards.
 * Limits: 1 <= M <= 2^31 - 129, 1 <= N <= 16,776,960 (65,535 column tiles of 256),
 * d a positive multiple of 64 and at most 65,536.
 * Every bf16 product is exact in fp32, so each logit lies within
 * gamma_(d-1) * sum_j |hidden_j * weight_vj| of the exact dot product
 * (gamma_n = n u / (1 - n u), u = 2^-23; the oracle's logit_error_bound).
 * Returns SV_ERR_NULL, SV_ERR_SHAPE or SV_ERR_ALIGN before launching; SV_ERR_CUDA
 * when the tensor-map encoder or the launch fails; SV_OK once the work is queued
 * on `stream` (a cudaStream_t). */
sv_status spec_lm_head_logits(const void* hidden, const void* weight, int M, int N, int d,
                              float* logits, int32_t* flag, void* stream);

/* spec_verify on logit rows computed from hidden states.
 *   hidden_target [B][K+1][d] bf16 and weight_target [V][d] bf16 give the K+1
 *                 target rows;
 *   hidden_draft  [B][K][d_draft] bf16 and weight_draft [V][d_draft] bf16 give the
 *                 K draft rows (an MTP head that shares the target's head passes
 *                 the same weight); both NULL when every temperature is 0;
 *   logits_scratch [B][2K+1][V] fp32, device, caller-owned, 16-byte aligned: the
 *                 target rows [B][K+1][V] first, then the draft rows [B][K][V];
 *                 they hold the computed logits when the call's work is done.
 *   flag          as in spec_lm_head_logits (set when either GEMM timed out). When
 *                 it is set, the verify step has run on undefined logits: its
 *                 out_tokens and out_n_accepted are not valid and must be dropped.
 * The two GEMMs run first (spec_lm_head_logits), then spec_verify with SV_F32 on
 * the scratch rows. All other arguments and results are those of spec_verify.
 * Every argument is checked before anything is launched: SV_ERR_NULL,
 * SV_ERR_SHAPE (B, K, V outside spec_verify's limits, or d / d_draft not a
 * positive multiple of 64 up to 65,536), SV_ERR_ALIGN, SV_ERR_WORKSPACE; then
 * SV_ERR_CUDA from a failed launch, else SV_OK. */
sv_status spec_verify_from_hidden(const void* hidden_target, const void* weight_target, int d,
                                  const void* hidden_draft, const void* weight_draft, int d_draft,
                                  const int32_t* draft_tokens, const float* temperature,
                                  const int32_t* top_k, const float* top_p, uint64_t philox_seed,
                                  uint64_t philox_offset, int B, int K, int V, float* logits_scratch,
                                  int32_t* flag, int32_t* out_tokens, int32_t* out_n_accepted,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* The greedy (temperature 0) verify step fused with the LM head: the target
 * logits are never written to memory.
 * What the pages define: the decode step chooses the token from the row z = h .
 * W^T ("Apple Silikon İçin Cihaz Üstü Çıkarımı Optimize Etme", decode section; its
 * section on the limits of further optimisation tried fusing this projection
 * with the token choice), and greedy verification compares each drafted token
 * with the target argmax ("after three fixes, Qwen3.5/3.6 MTP head reaches 1.4x
 * on Apple Silicon", deniz.in, section "Verification under sampling was wrong"):
 * the drafted tokens are kept while each equals its row's argmax, and the target
 * argmax is emitted at the first mismatch or after the K-th position.
 *   hidden_target [B][K+1][d] bf16, device, 16-byte aligned: the target's final
 *                 hidden states at positions 0..K
 *   weight        [V][d] bf16, device, 16-byte aligned: the LM-head weight
 *   draft_tokens  [B][K] int32, device: the drafted ids
 *   flag          [1] int32, device, caller-owned: set to 1 when a wait of the
 *                 GEMM timed out; the results are then not valid. The caller
 *                 zeroes it before the call.
 *   out_tokens [B][K+1], out_n_accepted [B]: as spec_verify with every temperature
 *                 0: n drafted tokens, then the target argmax, then -1; a row whose
 *                 maximum is NaN or +inf or whose logits are all -inf, or a drafted
 *                 id outside [0, V), gives n = -1 and K+1 tokens -1.
 *   workspace     spec_verify_workspace_bytes(B, K) bytes, 16-byte aligned and
 *                 zero-filled, left zero-filled (its first B(K+1) 64-bit words
 *                 hold the rows' keys during the call).
 * The argmax is that of the fp32-accumulated logits (lowest id among equal
 * maxima); it can differ from the exact dot products' only where two logits lie
 * within the fp32 accumulation bound of spec_lm_head_logits.
 * Limits: 1 <= B <= 65535, 1 <= K <= 16, 2 <= V <= 262144, d a positive multiple
 * of 64 and at most 65,536. Returns SV_ERR_NULL, SV_ERR_SHAPE, SV_ERR_ALIGN or
 * SV_ERR_WORKSPACE before launching anything; SV_ERR_CUDA when the tensor-map
 * encoder or a launch fails; SV_OK once the GEMM and the acceptance kernel are
 * queued on `stream`. */
sv_status spec_verify_greedy_from_hidden(const void* hidden_target, const void* weight, int d,
                                         const int32_t* draft_tokens, int B, int K, int V, int32_t* flag,
                                         int32_t* out_tokens, int32_t* out_n_accepted, void* workspace,
                                         size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_LM_HEAD_H */
