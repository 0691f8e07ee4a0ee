/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact IO-aware attention library.
 *
 * What the library computes (one attention head; every (b, h) is independent):
 *
 *   S = scale * Q K^T + bias          bias added after scaling
 *   P = row-softmax(S),  O = P V
 *   LSE_i = log(sum_j exp(S_ij))      natural log, one float per query row
 *
 * ("Understanding FlashAttention Pt 1", §0.2 Notation; "flash-attention"
 * Part IV, Stages 6-7 for the O + fp32 LSE contract.) The forward streams K and
 * V through on-chip tiles with the online-softmax recurrence ("Understanding
 * FlashAttention Pt 1", §2.3-2.4; "FlashAttention, Explained", §10 and §13), so
 * the Nq x Nk matrices S and P never reach device memory. The backward
 * recomputes P from the saved LSE ("Understanding FlashAttention Pt 1", §3.6;
 * "flash-attention", Part VII) and returns dQ, dK, dV.
 *
 * Layout. Every tensor is contiguous, row-major [B][H][N][d] with d innermost
 * (PyTorch SDPA order, not flash-attn's [B][N][H][d]); LSE is [B][H][Nq] fp32;
 * key_bias is [B][Nk] fp32, broadcast over heads and query rows.
 *
 * Masking.
 *   - causal != 0: key j is visible to query i iff j <= i + (Nk - Nq)
 *     (bottom-right alignment; the plain lower triangle when Nq == Nk);
 *   - key_bias[b][j] = -INFINITY masks key j of batch b;
 *   - a query row with no visible key gets O = 0 and LSE = -INFINITY
 *     ("flash-attention", Part VI: fully masked rows give zeros, not NaN).
 *
 * Pointers. q, k, v, o, lse, dO, dq, dk, dv, key_bias and the workspace are
 * DEVICE pointers owned by the caller; the library keeps none of them after a
 * call returns and allocates no device memory per call. q, k, v, o, dO, dq,
 * dk, dv must be 16-byte aligned; key_bias and lse 4-byte aligned.
 *
 * Streams and errors. Every call validates its arguments on the host before
 * any launch and returns a status without synchronising; the work is queued
 * on `stream` (a cudaStream_t; NULL = the legacy default stream). Launch
 * failures map to FA_ERR_CUDA. Device-side failures (a bounded wait inside a
 * kernel that timed out) are reported by fa_get_last_device_error; the error
 * is sticky: until that call clears it, later launches on the device stop at
 * their first slow wait, and their outputs are invalid too.
 * Calls on distinct streams may run concurrently.
 *
 * Supported: dtype FA_DTYPE_BF16 with d in {64, 128} (forward and backward);
 * dtype FA_DTYPE_FP32 with d in {64, 128} (forward only; fp32 arithmetic).
 * Nq, Nk >= 1, B, H >= 1, B * H < 2^31, Nq, Nk < 2^31 / d. Other values
 * return FA_ERR_UNSUPPORTED or FA_ERR_INVALID_ARG.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, bad workspace */
    FA_ERR_UNSUPPORTED = 2,   /* valid request outside what is implemented (d, dtype) */
    FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
    FA_ERR_DEVICE = 4         /* a kernel reported a device-side timeout */
} fa_status;

typedef enum {
    FA_DTYPE_BF16 = 0,
    FA_DTYPE_FP32 = 1
} fa_dtype;

/*
 * Forward. Writes o [B,H,Nq,d] (dtype) and lse [B,H,Nq] (fp32, natural log).
 * key_bias may be NULL (no bias). scale is applied to Q K^T before the bias
 * (1/sqrt(d) for standard attention). lse may be NULL for the fp32 path only
 * if the caller does not need it; the bf16 path always writes it.
 * Computes: tiling + online softmax ("FlashAttention, Explained", §13; the
 * query-tile-outer order of §20); causal tile skipping ("Understanding
 * FlashAttention Pt 1", §3.5).
 * Scheduling: with more query-tile pairs x heads than SMs (bf16, no bias),
 * one word of lse (row 0 of the last head) serves as the kernel's work
 * counter while the call runs: it is set with a memset on `stream` before the
 * kernel and holds that row's LSE when the kernel ends. lse must therefore
 * not be read or written by other work until the call has completed on
 * `stream`, as for any output.
 */
fa_status fa_fwd(const void *q, const void *k, const void *v, const float *key_bias,
                 void *o, float *lse,
                 int B, int H, int Nq, int Nk, int d, float scale, int causal,
                 fa_dtype dtype, void *stream);

/*
 * Grouped-query / multi-query attention ("Understanding FlashAttention Pt 1",
 * Part 4.1; "flash-attention", the MQA/GQA note): q, o (and dO, dq) are
 * [B,H,N,d]; k, v (and dk, dv) are [B,H_kv,Nk,d] with H a multiple of H_kv;
 * query head h attends key/value head h / (H / H_kv). H_kv == H is plain
 * multi-head attention (fa_fwd / fa_bwd are these calls with H_kv = H);
 * H_kv == 1 is multi-query attention. dk and dv of a shared head sum the
 * contributions of every query head of its group. Otherwise identical to
 * fa_fwd / fa_bwd (same workspace size, as a function of B, H, Nq, Nk, d).
 */
fa_status fa_fwd_gqa(const void *q, const void *k, const void *v, const float *key_bias,
                     void *o, float *lse,
                     int B, int H, int H_kv, int Nq, int Nk, int d, float scale, int causal,
                     fa_dtype dtype, void *stream);
fa_status fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o,
                     const float *lse, const void *dO,
                     void *dq, void *dk, void *dv, const float *key_bias,
                     int B, int H, int H_kv, int Nq, int Nk, int d, float scale, int causal,
                     fa_dtype dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Packed variable-length batches ("flash-attention", the varlen entry points
 * with cu_seqlens; padding replaced by packing): B sequences of different
 * lengths are stored back to back, per head:
 *   q, o: [H][total_q][d] bf16   k, v: [H_kv][total_k][d] bf16   lse: [H][total_q]
 * Sequence b occupies query rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key
 * rows [cu_seqlens_k[b], cu_seqlens_k[b+1]) (device int32 arrays of B+1
 * non-decreasing offsets, cu[0] = 0, cu[B] = total). Each sequence is an
 * independent problem: causal is bottom-right within the sequence, and no
 * query attends keys of another sequence. max_seqlen_q/k must be at least
 * the largest sequence length (they size the grid). A sequence whose offsets
 * or length break these rules is detected on the device and reported by
 * fa_get_last_device_error (its rows are then not written). No key bias.
 */
fa_status fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                        const int *cu_seqlens_q, const int *cu_seqlens_k,
                        int B, int H, int H_kv, int total_q, int total_k,
                        int max_seqlen_q, int max_seqlen_k, int d, float scale, int causal,
                        void *stream);

/*
 * Backward of fa_fwd_varlen (same packed layout; o and lse from that call;
 * dq [H][total_q][d], dk, dv [H_kv][total_k][d]). Workspace:
 * fa_bwd_varlen_workspace_size(B, H, total_q, max_seqlen_q, d) bytes,
 * 256-byte aligned.
 */
size_t fa_bwd_varlen_workspace_size(int B, int H, int total_q, int max_seqlen_q, int d);
fa_status fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                        const float *lse, const void *dO, void *dq, void *dk, void *dv,
                        const int *cu_seqlens_q, const int *cu_seqlens_k,
                        int B, int H, int H_kv, int total_q, int total_k,
                        int max_seqlen_q, int max_seqlen_k, int d, float scale, int causal,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Split-KV forward (Flash-Decoding) for problems with few query rows and many
 * keys, e.g. decoding: the keys of every (b, h) are cut into num_splits
 * contiguous ranges processed by separate CTAs, each producing a partial
 * normalised output O_s (fp32) and its log-sum-exp LSE_s in the workspace;
 * a second launch merges them with the log-sum-exp rule
 *   LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s
 * ("flash-attention", Part VI; "FlashAttention: Mathematical Foundations...",
 * Flash-Decoding). Same arguments, layout and results as fa_fwd_gqa (bf16 only),
 * plus num_splits >= 1 (1 = no split, no workspace use) and a device
 * workspace of fa_fwd_splitkv_workspace_size(...) bytes, 256-byte aligned.
 * fa_fwd_splitkv_default_splits gives a split count for the current device
 * (its SM count; no launch): the one whose grid, in waves of one CTA per SM,
 * leaves the least of its last wave idle, with at least 4 key tiles of 128
 * keys per split and at most 128 splits.
 */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits);
int fa_fwd_splitkv_default_splits(int B, int H, int Nq, int Nk, int d);
fa_status fa_fwd_splitkv(const void *q, const void *k, const void *v, const float *key_bias,
                         void *o, float *lse,
                         int B, int H, int H_kv, int Nq, int Nk, int d, float scale, int causal,
                         int num_splits, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace fa_bwd needs: -scale * D with D = rowsum(dO o O),
 * and -LSE rescaled to base 2, each fp32 [B*H][Nq rounded up to a multiple of 128],
 * an fp32 dQ accumulator [B,H,Nq,d] and a 256-byte work-item counter of the main
 * launch (reset by it), each starting on a 256-byte boundary.
 * Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int Nq, int Nk, int d);

/*
 * Backward. Given q, k, v, the o and lse written by fa_fwd with the same
 * arguments, and dO (dtype, [B,H,Nq,d]), writes dq, dk, dv (dtype). The result
 * is undefined if o/lse come from a different call. workspace must hold
 * fa_bwd_workspace_size(...) bytes and be 256-byte aligned; its contents on
 * entry do not matter. dQ is accumulated across key tiles with atomic adds,
 * so dq may differ in the last bits between runs; dk and dv are
 * deterministic.
 * Computes: D_i = rowsum(dO_i o O_i), then per key tile: recompute S and
 * P = exp(S - LSE), dV += P^T dO, dP = dO V^T, dS = P o (dP - D),
 * dQ += scale dS K, dK += scale dS^T Q ("Understanding FlashAttention Pt 1",
 * §3.6; "FlashAttention, Explained", §17; "flash-attention", Part VII).
 */
fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o,
                 const float *lse, const void *dO,
                 void *dq, void *dk, void *dv, const float *key_bias,
                 int B, int H, int Nq, int Nk, int d, float scale, int causal,
                 fa_dtype dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The three launches of fa_bwd, one per call, with fa_bwd's arguments and
 * validation; calling them in this order on one stream is equivalent to
 * fa_bwd ("flash-attention", Part VII: a preprocess launch, then the main
 * backward launch):
 *   fa_bwd_preprocess   -scale * rowsum(dO o O), -base-2 LSE, zeroed dQ accumulator
 *                       (reads o, lse, dO; writes the workspace);
 *   fa_bwd_main         recompute P per tile, dK and dV (written to dk, dv),
 *                       dQ reduced into the workspace accumulator;
 *   fa_bwd_postprocess  dq = bf16(dQ accumulator).
 * Useful to time or schedule the stages separately.
 */
fa_status fa_bwd_preprocess(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *dO,
                            void *dq, void *dk, void *dv, const float *key_bias,
                            int B, int H, int Nq, int Nk, int d, float scale, int causal,
                            fa_dtype dtype, void *workspace, size_t workspace_bytes,
                            void *stream);
fa_status fa_bwd_main(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dO,
                      void *dq, void *dk, void *dv, const float *key_bias,
                      int B, int H, int Nq, int Nk, int d, float scale, int causal,
                      fa_dtype dtype, void *workspace, size_t workspace_bytes, void *stream);
fa_status fa_bwd_postprocess(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dO,
                             void *dq, void *dk, void *dv, const float *key_bias,
                             int B, int H, int Nq, int Nk, int d, float scale, int causal,
                             fa_dtype dtype, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * FP8 forward ("FlashAttention, Explained", §21 and "FlashAttention:
 * Mathematical Foundations...", the FP8 forward of FA-3: e4m3 operands with
 * scaling factors, the matrix products at the fp8 tensor-core rate). Same
 * arguments and results as fa_fwd_gqa (bf16 q, k, v; bf16 o, fp32 lse;
 * d = 128 only, else FA_ERR_UNSUPPORTED), computed as:
 *   scale_x = max|x| / 448 per (batch, head) of each of q, k, v (1 if 0),
 *   x8 = e4m3(x / scale_x), round to nearest even;
 *   S = scale * scale_q * scale_k * (q8 k8^T) (fp32 accumulation),
 *   P = exp(S - m) rounded to e4m3, O = scale_v * (P v8) / rowsum(exp(S - m)),
 *   LSE from the fp32 S.
 * The result approximates attention on the dequantized inputs
 * scale_x * x8; P's rounding (relative 2^-4) bounds the difference.
 * workspace: fa_fwd_fp8_workspace_size(...) bytes, 256-byte aligned:
 *   [0]  fp32 max|q| [B*H], max|k| [B*H_kv], max|v| [B*H_kv]
 *   then, each on a 256-byte boundary: e4m3 q [B,H,Nq,d], e4m3 k
 *   [B,H_kv,Nk,d], e4m3 v transposed [B,H_kv,d,Nk16] (Nk16 = Nk rounded up to
 *   a multiple of 16, the padding 0).
 * fa_fwd_fp8_stage runs stage 1 (quantize into the workspace) or stage 2
 * (attention from the workspace) alone; 0 runs both (= fa_fwd_fp8).
 */
size_t fa_fwd_fp8_workspace_size(int B, int H, int H_kv, int Nq, int Nk, int d);
fa_status fa_fwd_fp8(const void *q, const void *k, const void *v, const float *key_bias,
                     void *o, float *lse,
                     int B, int H, int H_kv, int Nq, int Nk, int d, float scale, int causal,
                     void *workspace, size_t workspace_bytes, void *stream);
fa_status fa_fwd_fp8_stage(const void *q, const void *k, const void *v, const float *key_bias,
                           void *o, float *lse,
                           int B, int H, int H_kv, int Nq, int Nk, int d, float scale, int causal,
                           void *workspace, size_t workspace_bytes, void *stream, int stage);

/*
 * Deterministic backward ("flash-attention", Part VII: the backward's
 * deterministic option). fa_bwd accumulates dQ over key tiles with
 * reductions whose order depends on timing, so dq may differ in the last
 * bits between runs. Here dq is formed by a second, query-tile-outer kernel
 * that adds the key tiles' contributions in a fixed order inside one CTA, so
 * dq, dk and dv are bitwise identical from run to run for the same inputs
 * and device. Same arguments and results as fa_bwd_gqa (H_kv == H: plain
 * multi-head) and fa_bwd_varlen respectively. S and P are recomputed in both
 * kernels (seven tile products per (query tile, key tile) pair instead of
 * five); no dQ accumulator is needed, so the workspace is only D and the
 * base-2 LSE: fa_bwd_deterministic_workspace_size(B, H, Nq, d) bytes (for
 * the varlen call: Nq = max_seqlen_q), 256-byte aligned, contents on entry
 * irrelevant.
 * fa_bwd_deterministic_stage runs one of its three launches (stage 1:
 * preprocess; 2: dK and dV; 3: dQ); in that order on one stream they equal
 * fa_bwd_deterministic. Invalid stage numbers give FA_ERR_INVALID_ARG.
 */
size_t fa_bwd_deterministic_workspace_size(int B, int H, int Nq, int d);
fa_status fa_bwd_deterministic(const void *q, const void *k, const void *v, const void *o,
                               const float *lse, const void *dO,
                               void *dq, void *dk, void *dv, const float *key_bias,
                               int B, int H, int H_kv, int Nq, int Nk, int d, float scale,
                               int causal, fa_dtype dtype, void *workspace,
                               size_t workspace_bytes, void *stream);
fa_status fa_bwd_deterministic_stage(const void *q, const void *k, const void *v, const void *o,
                                     const float *lse, const void *dO,
                                     void *dq, void *dk, void *dv, const float *key_bias,
                                     int B, int H, int H_kv, int Nq, int Nk, int d, float scale,
                                     int causal, fa_dtype dtype, void *workspace,
                                     size_t workspace_bytes, void *stream, int stage);
fa_status fa_bwd_varlen_deterministic(const void *q, const void *k, const void *v, const void *o,
                                      const float *lse, const void *dO, void *dq, void *dk,
                                      void *dv, const int *cu_seqlens_q, const int *cu_seqlens_k,
                                      int B, int H, int H_kv, int total_q, int total_k,
                                      int max_seqlen_q, int max_seqlen_k, int d, float scale,
                                      int causal, void *workspace, size_t workspace_bytes,
                                      void *stream);

/*
 * Size in bytes of the device array fa_bwd_noalloc uses as its workspace.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * fa_bwd_noalloc -- fa_bwd without a caller-provided workspace. (The pages
 * have no counterpart: this is a convenience of this library.)
 *
 * For callers that cannot allocate device memory while attention runs (a
 * runtime that plans all device memory ahead and passes kernels only their
 * inputs and outputs, code running inside an allocator callback, a service
 * that may not call cudaMalloc on its request path). The workspace comes from
 * a fixed 32 MiB array in the library's device image, held by every GPU that
 * loads the library until the process exits; nothing is allocated per call.
 * Arguments, layout, results and error codes are those of fa_bwd, except:
 *   - FA_ERR_UNSUPPORTED if fa_bwd_workspace_size(B, H, Nq, Nk, d) exceeds
 *     FA_NOALLOC_SCRATCH_BYTES (checked before any launch);
 *   - all calls share the array: calls that overlap on the GPU race and must
 *     be serialised by the caller;
 *   - the first call on a device looks up the array's address on that device
 *     (the current one); make that first call before any stream capture.
 *     After cudaDeviceReset the device's next context holds the array at a
 *     new address: the library notices the new context and looks the address
 *     up again on the next call, which should likewise come before any
 *     capture.
 */
fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dO,
                         void *dq, void *dk, void *dv, const float *key_bias,
                         int B, int H, int Nq, int Nk, int d, float scale, int causal,
                         fa_dtype dtype, void *stream);

/* Static, human-readable name of a status code (never NULL). */
const char *fa_status_string(fa_status s);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word. Returns FA_ERR_DEVICE if any kernel since the last call gave up on a
 * bounded wait (its outputs are then invalid), FA_ERR_CUDA if the
 * synchronisation itself failed, FA_OK otherwise.
 */
fa_status fa_get_last_device_error(void *stream);

/*
 * Diagnostic of the device-side failure path: launches one thread that waits,
 * with the same bounded wait the kernels use, on a barrier nothing arrives at.
 * After about 2 seconds the wait gives up, records a timeout in the device
 * error word and the kernel returns, leaving the context usable; the next
 * fa_get_last_device_error returns FA_ERR_DEVICE (and clears the word).
 * Returns FA_ERR_CUDA if the launch fails.
 */
fa_status fa_selftest_device_timeout(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
