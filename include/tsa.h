/*
 * tsa.h -- C ABI of libtsa, the GB300 (sm_103a) hot path of trainable sparse
 * attention: indexer score -> deterministic exact top-k -> sparse attention
 * forward/backward, for the absorbed-MLA layout and for block Sparse-GQA.
 *
 * Sources (web pages, cited by title and section):
 *   [QSA]  Megatron-LM issue #7060 "Add trainable QSA sparse attention with a
 *          TileLang backend".
 *   [DSA]  Megatron-LM PR #3674 "Enable DSA CP/absorbed/THD paths with TileLang
 *          fused ops".
 *   [NOPE] Megatron-LM PR #7617 "Support NoPE shapes and unaligned top-k in
 *          TileLang sparse MLA".
 *
 * Conventions shared by every entry point
 *   - Pointers named *_dev are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them.  Host arrays are read during the
 *     call only.
 *   - bf16 tensors are passed as void* to raw, dense, row-major bf16 storage.
 *   - Sequences: cu_seqlens is a HOST int32 array of num_seqs+1 prefix offsets
 *     (cu_seqlens[0] = 0, non-decreasing, 1 <= num_seqs <= TSA_MAX_SEQS); the
 *     T = cu_seqlens[num_seqs] tokens are packed rows (THD).  BSHD batch B x S
 *     is cu_seqlens = {0, S, 2S, ..., B*S} [QSA "Describe the solution":
 *     BSHD and packed THD/variable-length paths].
 *   - Indices are key (or block) positions LOCAL to the query's sequence; -1 is
 *     the invalid sentinel [NOPE "What does this PR do?"].
 *   - stream is a cudaStream_t (NULL = legacy default stream).  Every call is
 *     asynchronous on it; host-side validation happens before any launch.
 *   - Return value: TSA_OK or a tsa_status error code; on error nothing was
 *     launched (argument errors) or the CUDA error is reported (TSA_ERR_CUDA).
 *     tsa_last_error() gives a one-line detail for the calling thread.  No
 *     unsupported shape is ever routed to a slower or CPU path: it is refused.
 *   - Index words outside their sequence never fault: the kernels treat them
 *     as -1 and raise TSA_FLAG_INDEX_RANGE, read with tsa_read_flags().
 */
#ifndef TSA_H_
#define TSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TSA_MAX_SEQS 1024

typedef enum {
  TSA_OK = 0,
  TSA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shapes   */
  TSA_ERR_UNSUPPORTED = 2,   /* valid but not built (e.g. an odd head count)  */
  TSA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required     */
  TSA_ERR_CUDA = 4,          /* a CUDA runtime call failed                     */
  TSA_ERR_INDEX_RANGE = 5,   /* reported by tsa_read_flags only                */
  TSA_ERR_TIMEOUT = 6        /* a bounded device wait gave up                  */
} tsa_status;

/* Device-side flags raised by kernels (never a trap). */
#define TSA_FLAG_INDEX_RANGE 0x1u  /* an index pointed outside its sequence */
#define TSA_FLAG_TIMEOUT     0x2u  /* a bounded spin-wait ran out           */

const char* tsa_status_string(int status);
const char* tsa_last_error(void);
int tsa_version(void);

/* Number of CUDA kernels this library has launched since it was loaded (all
 * devices, all threads).  Host-side counter; used to account for launches. */
unsigned long long tsa_kernel_launches(void);

/* Copy the device flags (bitwise OR of TSA_FLAG_*) to *flags after
 * synchronising `stream`; clear them when clear != 0. */
int tsa_read_flags(uint32_t* flags, int clear, void* stream);

/* Self-test of the failure path of the kernels' bounded waits, with no fault:
 * launches one CTA on `stream` that waits on a shared-memory barrier no thread
 * arrives on, using the same bounded wait as every pipeline of the library.
 * After the wait limit (2 s) the CTA raises TSA_FLAG_TIMEOUT and returns
 * normally; the CUDA context stays usable.  Asynchronous: read the flag with
 * tsa_read_flags.  Returns TSA_ERR_CUDA if the launch fails. */
int tsa_selftest_bounded_wait(void* stream);

/* ---------------------------------------------------------------------------
 * qsa_indexer_scores -- materialised indexer scores for a range of queries.
 * [QSA "Describe the solution": trainable indexer with ReLU scores, exact
 * block top-k over a [sequence, sequence/block_size] matrix; DSA "Changes":
 * fused indexer forward + logits cleaning.]
 *
 *   I_g[t,s] = score_scale * sum_{h in group g} w[t,h] * ReLU(q_I[t,h,:].k_I[s,:])
 *   for local keys s <= p(t) of t's sequence; group g owns heads
 *   [g*H_I/groups, (g+1)*H_I/groups).  block_size > 1 gives the block score
 *   max_{s in block b, s <= p(t)} I_g[t,s].  Non-candidates are -inf.
 *
 *   q_idx_dev  bf16 [T, H_I, d_I]     k_idx_dev bf16 [T, d_I]
 *   w_dev      fp32 [T, H_I]
 *   scores_dev fp32 [q_count, groups, width] for packed rows
 *              [q_begin, q_begin+q_count); width >= max sequence length
 *              (block_size == 1) or >= ceil(max length / block_size).
 * Supported: H_I in {2,4,...,128} (power of two), d_I in {64,128},
 * H_I/groups >= 2, block_size in {1, 16, 32, 64, 128}.
 * Fully deterministic.  Intended for parity checks and small problems; the
 * streaming qsa_topk never materialises the full score matrix.
 * ------------------------------------------------------------------------- */
int qsa_indexer_scores(const void* q_idx_dev, const void* k_idx_dev, const float* w_dev,
                       const int32_t* cu_seqlens, int num_seqs, int H_I, int d_I, int groups,
                       int block_size, float score_scale, int64_t q_begin, int64_t q_count,
                       float* scores_dev, int64_t width, void* stream);

/* ---------------------------------------------------------------------------
 * qsa_topk_from_scores -- deterministic exact top-k of fp32 score rows.
 * [QSA "Describe the solution": deterministic exact TopK with a lexicographic
 * (score, block_id) key, because ReLU scores tie at zero; "Additional
 * context": deterministic tie-breaking for recomputation and TP ranks.]
 *
 *   For every row r of scores_dev[rows][ld] (first `width` entries): the
 *   `topk` best finite entries under (score desc, index asc), -0.0 == +0.0,
 *   -inf entries are not candidates; indices_dev[r][0..topk) in that order,
 *   -1 after the last candidate.  Bit-identical across runs.
 * Supported: 1 <= topk <= 4096, width <= 2^31-1.
 * ------------------------------------------------------------------------- */
int qsa_topk_from_scores(const float* scores_dev, int64_t rows, int64_t width, int64_t ld,
                         int topk, int32_t* indices_dev, void* stream);

/* ---------------------------------------------------------------------------
 * qsa_topk -- streaming indexer + exact top-k, bounded memory.
 * [QSA "Describe the solution": streaming indexer runner with bounded memory;
 * "Describe alternatives": materialising all block scores is rejected.]
 *
 *   indices_dev int32 [T, groups, topk]: the row for (t, g) is
 *   qsa_topk_from_scores applied to qsa_indexer_scores(t, g).  Scores live
 *   only in the caller's workspace, two query chunks at a time
 *   (qsa_topk_workspace_size bytes: two score buffers of at most 512 MB each,
 *   independent of T beyond the longest sequence): the top-k of one chunk
 *   runs while the indexer scores the next into the other buffer.  The work
 *   goes to two library-owned streams of this device (created on the first
 *   call; the indexer's on the highest priority), forked from `stream` and
 *   joined back into it by events, so the call is ordered on `stream` like a
 *   single kernel.  Calls from several host threads are serialised while they
 *   enqueue.  The first call on a device creates those streams and events:
 *   make it before any stream capture (later calls may be captured; the fork
 *   and the join are ordinary event dependencies of the captured graph).
 * ------------------------------------------------------------------------- */
size_t qsa_topk_workspace_size(const int32_t* cu_seqlens, int num_seqs, int groups, int block_size);
int qsa_topk(const void* q_idx_dev, const void* k_idx_dev, const float* w_dev,
             const int32_t* cu_seqlens, int num_seqs, int H_I, int d_I, int groups, int block_size,
             float score_scale, int topk, int32_t* indices_dev, void* workspace_dev,
             size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * qsa_topk_no_alloc -- qsa_topk for callers that cannot provide scratch memory.
 * (The pages have no counterpart: this is an interface convenience.)
 *
 *   Same arguments and result as qsa_topk, minus the workspace.  It is for
 *   hosts that may not allocate device memory once running (fixed memory
 *   budgets, allocation-free serving loops, plugin interfaces that pass only
 *   input and output buffers).  The score scratch is a fixed 16 MiB device
 *   array inside the library, held by every GPU that loads it until exit; the
 *   library allocates nothing.  The first call on a device looks up that
 *   array's address with the device current -- make it before any stream
 *   capture.  All calls share the array: calls that overlap on the GPU race and
 *   must be serialised by the caller.  A problem needing more than 16 MiB for
 *   one query row of scores (groups * row width * 4 bytes) is refused with
 *   TSA_ERR_UNSUPPORTED.  Output is bit-identical to qsa_topk's.
 * ------------------------------------------------------------------------- */
int qsa_topk_no_alloc(const void* q_idx_dev, const void* k_idx_dev, const float* w_dev,
                      const int32_t* cu_seqlens, int num_seqs, int H_I, int d_I, int groups,
                      int block_size, float score_scale, int topk, int32_t* indices_dev,
                      void* stream);

/* ---------------------------------------------------------------------------
 * sparse_mla_fwd -- absorbed sparse MLA forward.
 * [DSA "Changes": sparse MLA forward over the absorbed latent; NOPE "What
 * does this PR do?": q [T,H,576], kv latent [T,576], value = kv[..., :512],
 * explicit softmax scale, -1 slots masked, NoPE 512-wide inputs.]
 *
 *   For each (t, h): logits_j = softmax_scale * q[t,h,:].kv[s0+idx[t,j], :]
 *   over valid slots j (idx >= 0; slots >= topk do not exist, so an unaligned
 *   topk behaves exactly like one padded with -1); out = softmax . kv[:, :512];
 *   lse = log(sum_j exp(logits_j)) (natural log).  No valid slot: out = 0,
 *   lse = -inf.  Indices are not re-masked for causality.
 *
 *   q_dev bf16 [T, H, d_qk], kv_dev bf16 [T, d_qk], indices_dev int32 [T, topk]
 *   out_dev bf16 [T, H, 512], lse_dev fp32 [T, H]
 * d_qk = 512 is the NoPE layout: identical to zero-padding q/kv to 576.
 * Supported: 1 <= H <= 128, d_qk in {512, 576}, 1 <= topk.
 * Deterministic (bit-identical across runs).
 * ------------------------------------------------------------------------- */
int sparse_mla_fwd(const void* q_dev, const void* kv_dev, const int32_t* indices_dev,
                   const int32_t* cu_seqlens, int num_seqs, int H, int d_qk, int topk,
                   float softmax_scale, void* out_dev, float* lse_dev, void* stream);

/* ---------------------------------------------------------------------------
 * sparse_mla_bwd -- absorbed sparse MLA backward.
 * [DSA "Changes": sparse MLA backward kernels; NOPE "Validation": the
 * backward accumulates dKV atomically and is tolerance-checked, not replayed.]
 *
 *   P = exp(scale*S - lse), dP = dO.V^T, Dlt = rowsum(dO*out),
 *   dS = P*(dP - Dlt); dq = scale*dS.K;
 *   dkv[idx] += scale*dS^T.q (+ P^T.dO on the first 512 channels).
 *   dq_dev bf16 [T, H, d_qk], dkv_dev bf16 [T, d_qk] (fully overwritten).
 *   teacher_dev: optional (NULL to skip) fp32 [T, topk], fully overwritten
 *   with the indexer's KL teacher [QSA "Describe the solution": sparse
 *   Stage-2 teacher]: the head mean (1/H) sum_h P[t,h,j] of the attention
 *   probabilities at every slot j (0 at -1 slots), from the P this backward
 *   recomputes anyway (bf16, as the dKV product uses it).  For H = 128 it is
 *   bit-identical across runs; for H < 128 the head blocks add their shares
 *   with fp32 atomics (order not fixed).
 *   workspace: sparse_mla_bwd_workspace_size(T, H, d_qk, topk) bytes: fp32
 *   dkv and Dlt, and for H = 128 a bf16 staging area for P and dS of one
 *   chunk of queries (at most 4 GiB; the chunk shrinks as topk grows).
 *   Returns 0 for T < 0, H < 1, d_qk < 1 or topk < 1.
 * Same support as sparse_mla_fwd.  dq is bit-identical across runs (no
 * atomics: every element accumulates its slots in a fixed order); the dkv
 * summation order is not fixed.
 * ------------------------------------------------------------------------- */
size_t sparse_mla_bwd_workspace_size(int64_t T, int H, int d_qk, int topk);
int sparse_mla_bwd(const void* q_dev, const void* kv_dev, const int32_t* indices_dev,
                   const void* out_dev, const float* lse_dev, const void* dout_dev,
                   const int32_t* cu_seqlens, int num_seqs, int H, int d_qk, int topk,
                   float softmax_scale, void* dq_dev, void* dkv_dev, float* teacher_dev,
                   void* workspace_dev, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * qsa_indexer_kl / qsa_indexer_bwd -- training the indexer on the selected
 * slots.  [QSA "Describe the problem": sparse KL supervision for training the
 * indexer; "Describe the solution you'd like": sparse Stage-2 teacher/KL loss
 * for indexer training; DSA "Changes": sparse-KL streaming for the indexer
 * loss, fused indexer backward kernel.]  The pages print no formula; the
 * reading (also the reference implementation's):
 *
 *   student I[t,j] = score_scale * sum_h w[t,h] * ReLU(q_I[t,h].k_I[s0+idx[t,j]])
 *   p[t,:] = softmax of I[t,:] over t's valid slots (idx in [0, length))
 *   loss[t] = KL(teacher[t,:] || p[t,:]) = sum_j a log(a/p) over valid slots
 *   with a > 0; dscore[t,j] = p - a on valid slots, 0 elsewhere.
 *
 * qsa_indexer_kl: indices_dev int32 [T, topk] (one group: the DSA token
 *   selection, e.g. qsa_topk's output), teacher_dev fp32 [T, topk] (e.g.
 *   sparse_mla_bwd's teacher_dev), loss_dev fp32 [T], dscore_dev fp32
 *   [T, topk] (fully overwritten).  A row without a valid slot gives 0, 0.
 * qsa_indexer_bwd: the gradient of sum_{t,j} dscore[t,j] * I[t,j] with
 *   respect to q_I, k_I and w (D = q_I[t,h].k_I[s]):
 *     dw[t,h]   = score_scale * sum_j dscore * ReLU(D)
 *     dq_I[t,h] = score_scale * sum_j dscore * w[t,h] * [D > 0] * k_I[s]
 *     dk_I[s]   = score_scale * sum_{t,j} dscore * sum_h w[t,h] [D > 0] q_I[t,h]
 *   dq_idx_dev bf16 [T, H_I, d_I], dk_idx_dev bf16 [T, d_I], dw_dev fp32
 *   [T, H_I] (all fully overwritten).  workspace:
 *   qsa_indexer_bwd_workspace_size(T, d_I) bytes (the fp32 dk accumulator;
 *   its summation order is not fixed; dq_idx and dw are bit-identical
 *   across runs).
 * Supported: d_I = 128, 1 <= H_I <= 128, 1 <= topk <= 4096.  Slots that are
 * -1 carry nothing; indices outside their sequence are treated as -1 and
 * raise TSA_FLAG_INDEX_RANGE.
 * ------------------------------------------------------------------------- */
int qsa_indexer_kl(const void* q_idx_dev, const void* k_idx_dev, const float* w_dev,
                   const int32_t* cu_seqlens, int num_seqs, int H_I, int d_I, float score_scale,
                   const int32_t* indices_dev, int topk, const float* teacher_dev, float* loss_dev,
                   float* dscore_dev, void* stream);
size_t qsa_indexer_bwd_workspace_size(int64_t T, int d_I);
int qsa_indexer_bwd(const void* q_idx_dev, const void* k_idx_dev, const float* w_dev,
                    const int32_t* cu_seqlens, int num_seqs, int H_I, int d_I, float score_scale,
                    const int32_t* indices_dev, int topk, const float* dscore_dev, void* dq_idx_dev,
                    void* dk_idx_dev, float* dw_dev, void* workspace_dev, size_t workspace_bytes,
                    void* stream);

/* ---------------------------------------------------------------------------
 * sparse_gqa_fwd / sparse_gqa_bwd -- block Sparse-GQA.
 * [QSA "Describe the solution": Sparse-GQA forward and backward over exact
 * block top-k selections, BSHD and packed THD.]
 *
 *   Query head h belongs to kv group g = h / (Hq/Hkv).  The keys of (t, h) are
 *   the local tokens s <= p(t) of every selected block b = block_indices[t,g,j]
 *   (b >= 0), i.e. s in [b*block_size, (b+1)*block_size).  Softmax of
 *   softmax_scale * q.k over them, times v; lse natural log; empty: 0 / -inf.
 *
 *   q_dev bf16 [T, Hq, d], k_dev/v_dev bf16 [T, Hkv, d],
 *   block_indices_dev int32 [T, Hkv, nsel], out_dev bf16 [T, Hq, d],
 *   lse_dev fp32 [T, Hq].  Forward workspace:
 *   sparse_gqa_fwd_workspace_size(T, Hq, Hkv, d, nsel) bytes: the selections
 *   inverted per (block, kv group), and per selection slot the normalised
 *   partial output of its block (bf16, Hq/Hkv x d: a convex combination of
 *   value rows) with its log-sum-exp (fp32); the slots are merged in slot
 *   order.  Backward: dq [T,Hq,d], dk/dv [T,Hkv,d]
 *   bf16 (overwritten), workspace sparse_gqa_bwd_workspace_size(T, Hq, Hkv,
 *   d, nsel) bytes: fp32 dq/dk/dv accumulators, rowsum(dO * O) and the
 *   selections inverted per (block, kv group), so that the backward visits
 *   each selected block once per chunk of the queries that chose it.
 * Supported: Hq/Hkv in {1..16}, d in {64, 128}, block_size in {32, 64},
 * T * Hkv * nsel < 2^31, T * Hq < 2^31.  Block ids at or past the end of their sequence are
 * dropped and raise TSA_FLAG_INDEX_RANGE.
 * Forward deterministic (bit-identical across runs); backward dq/dk/dv
 * summation order not fixed.
 * ------------------------------------------------------------------------- */
size_t sparse_gqa_fwd_workspace_size(int64_t T, int Hq, int Hkv, int d, int nsel);
int sparse_gqa_fwd(const void* q_dev, const void* k_dev, const void* v_dev,
                   const int32_t* block_indices_dev, const int32_t* cu_seqlens, int num_seqs,
                   int Hq, int Hkv, int d, int block_size, int nsel, float softmax_scale,
                   void* out_dev, float* lse_dev, void* workspace_dev, size_t workspace_bytes,
                   void* stream);

size_t sparse_gqa_bwd_workspace_size(int64_t T, int Hq, int Hkv, int d, int nsel);
int sparse_gqa_bwd(const void* q_dev, const void* k_dev, const void* v_dev,
                   const int32_t* block_indices_dev, const void* out_dev, const float* lse_dev,
                   const void* dout_dev, const int32_t* cu_seqlens, int num_seqs, int Hq, int Hkv,
                   int d, int block_size, int nsel, float softmax_scale, void* dq_dev,
                   void* dk_dev, void* dv_dev, void* workspace_dev, size_t workspace_bytes,
                   void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TSA_H_ */
