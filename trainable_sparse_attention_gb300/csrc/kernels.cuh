// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include "common.cuh"

namespace tsa {

struct TopkRows {
  const float* scores;  // row r starts at scores + r * ld
  int64_t ld;
  int64_t width;        // entries per row (upper bound on candidates)
  int mode;             // 0: n = width; 1: causal tokens; 2: causal blocks
  int groups;           // rows are (query, group) pairs in causal modes
  int bs;               // block size (mode 2)
  int64_t p0;           // local position of the query of row 0 (causal modes)
  int32_t* out;         // row r writes out + r * out_ld
  int64_t out_ld;
  int k;
};

struct IndexerArgs {
  const __nv_bfloat16* q;  // [T, H_I, d_I]
  const __nv_bfloat16* k;  // [T, d_I]
  const float* w;          // [T, H_I]
  int H_I, d_I, groups, bs;
  float score_scale;
  int seq_start;   // packed row of the sequence's first token
  int p_begin;     // local position of the launch's first query
  int nq;          // queries in this launch
  float* out;      // query q, group g -> out + (q*groups + g) * width
  int64_t width;
  int T_total = 0;                 // packed rows of q_I / k_I (bounds of the TMA maps)
  unsigned int* flags = nullptr;   // device error flags
};

struct MlaFwdArgs {
  const __nv_bfloat16* q;   // [T, H, D]
  const __nv_bfloat16* kv;  // [T, D]
  const int32_t* idx;       // [T, topk]
  int T, H, topk;
  float scale_log2;         // softmax_scale * log2(e)
  __nv_bfloat16* out;       // [T, H, 512]
  float* lse;               // [T, H]
  unsigned int* flags;      // device error flags
  SeqTable st;
};

struct MlaBwdArgs {
  const __nv_bfloat16* q;    // [T, H, D]
  const __nv_bfloat16* kv;   // [T, D]
  const int32_t* idx;        // [T, topk]
  const float* lse;          // [T, H] natural log
  const float* dlt;          // [T, H]
  const __nv_bfloat16* dout; // [T, H, 512]
  int T, H, topk;
  float scale;               // softmax scale
  float scale_log2;          // softmax scale * log2(e)
  __nv_bfloat16* dq;         // [T, H, D]
  float* dkv_acc;            // [T, D] fp32, zeroed by the caller
  SeqTable st;
  // 128-head tcgen05 path: queries q0 .. q0+nq of one chunk, P and dS (bf16)
  // staged in p_out / ds_out as [query - q0][head][kp].
  int q0 = 0;
  int kp = 0;
  __nv_bfloat16* p_out = nullptr;
  __nv_bfloat16* ds_out = nullptr;
  unsigned int* flags = nullptr;  // device error flags
  // optional indexer teacher [T, topk]: head mean of P at each slot (zeroed by the
  // caller for the H < 128 kernel, which adds each head block's share)
  float* teacher = nullptr;
};

// Inputs of the tcgen05 dKV GEMM: P and dS of queries q0 .. q0+nq in bf16,
// [query - q0][128 heads][kp slots], kp = topk rounded up to 128 (zero padded).
struct MlaBwdTcArgs {
  const __nv_bfloat16* q;     // [T, 128, D]
  const __nv_bfloat16* dout;  // [T, 128, 512]
  const __nv_bfloat16* ds;    // [nq, 128, kp]  scale * P * (dP - Dlt)
  const __nv_bfloat16* p;     // [nq, 128, kp]
  const int32_t* idx;         // [T, topk]
  int T, D, topk, kp, q0;
  float* dkv_acc;             // [T, D] fp32
  unsigned int* flags;        // device error flags
  SeqTable st;
  // optional indexer teacher [T, topk] (D = 576 only): the head mean of P, from
  // the rope block's spare accumulator lane
  float* teacher = nullptr;
};

// Key-centric Sparse-GQA on tcgen05 (gqa_tc.cu): selections inverted into
// per-(block, group) lists of entries t * nsel + j; the forward writes per-slot
// partials that a combine pass merges in slot order.  All buffers are the
// caller's workspace.
struct GqaTcArgs {
  const __nv_bfloat16* q;     // [T, Hq, d]
  const __nv_bfloat16* k;     // [T, Hkv, d]
  const __nv_bfloat16* v;     // [T, Hkv, d]
  const __nv_bfloat16* dout;  // backward: [T, Hq, d]
  const int32_t* blk;         // [T, Hkv, nsel] local block ids, -1 = none
  const float* lse_in;        // backward: [T, Hq] natural log
  const float* dlt;           // backward: [T, Hq] rowsum(dO * O)
  int T, Hq, Hkv, G, nsel, bs, d;
  float scale, scale_log2;
  int nblk;                   // blocks over all sequences
  int qseg, nseg;             // lists per query segment of qseg tokens (segment-major), nseg segments
  int* cnt;                   // [nseg * nblk * Hkv] entries per (segment, block, group)
  int* off;                   // [nseg * nblk * Hkv + 1] list offsets
  int* cur;                   // [nseg * nblk * Hkv] fill cursors
  int* choff;                 // [nseg * nblk * Hkv + 1] chunk offsets
  int* list;                  // [T * Hkv * nsel] per list: flat selection indices (t * Hkv + g) * nsel + j
  __nv_bfloat16* part_o;      // forward: [T * Hkv * nsel, G, d] normalised partial outputs (bf16)
  float* part_l;              // forward: [T * Hkv * nsel, G] their log2-sum-exp
  __nv_bfloat16* out;         // forward: [T, Hq, d]
  float* lse;                 // forward: [T, Hq]
  float* dq_acc;              // backward: [T, Hq, d] fp32
  float* dk_acc;              // backward: [T, Hkv, d] fp32
  float* dv_acc;              // backward: [T, Hkv, d] fp32
  unsigned int* flags;
  SeqTable st;
  int blk_base[TSA_MAX_SEQS + 1];  // first global block of each sequence
};
cudaError_t launch_gqa_fwd_tc(const GqaTcArgs& a, cudaStream_t stream);
cudaError_t launch_gqa_bwd_tc(const GqaTcArgs& a, cudaStream_t stream);

// Indexer training on the selected slots (indexer_kl.cu): the sparse KL of the
// student scores against the attention teacher, and the indexer backward.
struct IndexerSelArgs {
  const float* w;             // [T, H_I]
  const int32_t* idx;         // [T, topk] local positions, -1 = none
  const float* teacher;       // KL: [T, topk]
  const float* dscore;        // backward: [T, topk]
  float* loss;                // KL: [T]
  float* dscore_out;          // KL: [T, topk]
  __nv_bfloat16* dq;          // backward: [T, H_I, 128]
  float* dw;                  // backward: [T, H_I]
  float* dk_acc;              // backward: [T, 128] fp32, zeroed by the caller
  int T, H_I, topk;
  float score_scale;
  unsigned int* flags;
  SeqTable st;
};
bool indexer_sel_supported(int H_I, int d_I);
cudaError_t launch_indexer_sel(const IndexerSelArgs& a, const void* q, const void* k, bool bwd, cudaStream_t stream);
// Head mean of the staged bf16 P of one 128-head backward chunk -> teacher rows q0 .. q0+nq.
cudaError_t launch_mla_teacher_from_p(const __nv_bfloat16* P, int nq, int H, int kp, int topk, int q0,
                                      float* teacher, cudaStream_t stream);

cudaError_t launch_topk_rows(const TopkRows& a, int64_t rows, cudaStream_t stream);
cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t stream);
// tcgen05 indexer (token-level scores); launch_indexer routes to it when it applies.
bool indexer_tc_supported(int H_I, int d_I, int groups, int bs);
cudaError_t launch_indexer_tc(const IndexerArgs& a, cudaStream_t stream);
// Account for one kernel launch of this library (the count tsa_kernel_launches reports);
// every launch site calls it right after its <<<...>>> statement.
void note_launch();

// Host helpers of the C-ABI layer (api.cu), shared by every entry-point file.
// note_error records the detail message tsa_last_error() returns and passes the
// status through; device_flags is the current device's flag word (null if it
// cannot be looked up); make_seq_table validates cu_seqlens and fills the
// kernel-side table; check_indexer_shape refuses indexer shapes that are not
// built; score_width is the score-row width for the longest sequence.
int note_error(int code, const char* msg);
unsigned int* device_flags();
int make_seq_table(const int32_t* cu, int num_seqs, SeqTable* st, int64_t* T_out);
int check_indexer_shape(int H_I, int d_I, int groups, int block_size);
int64_t score_width(int max_len, int block_size);
cudaError_t launch_fill(float* p, int64_t n, float v, cudaStream_t stream);
cudaError_t launch_bounded_wait_selftest(unsigned int* flags, cudaStream_t stream);
cudaError_t launch_mla_fwd(const MlaFwdArgs& a, int D, cudaStream_t stream);
cudaError_t launch_mla_fwd_tc(const MlaFwdArgs& a, int D, cudaStream_t stream);
cudaError_t launch_mla_bwd(const MlaBwdArgs& a, int D, cudaStream_t stream);
cudaError_t launch_mla_bwd_dkv_tc(const MlaBwdTcArgs& a, int nq, cudaStream_t stream);
// tcgen05 recompute of P and dS (to a.p_out / a.ds_out) and dQ = dS K for queries a.q0 .. a.q0+nq.
cudaError_t launch_mla_bwd_pds_tc(const MlaBwdArgs& a, int D, int nq, cudaStream_t stream);
cudaError_t launch_mla_bwd_dq_tc(const MlaBwdArgs& a, int D, int nq, cudaStream_t stream);
cudaError_t launch_bwd_delta(const __nv_bfloat16* o, const __nv_bfloat16* dout, float* dlt, int64_t rows, int dv,
                             cudaStream_t stream);
cudaError_t launch_f32_to_bf16(const float* src, __nv_bfloat16* dst, int64_t n, cudaStream_t stream);

constexpr int kMlaFwdTcMinHeads = 32;  // the forward runs on tcgen05 (heads padded to 128) above this
constexpr int kIndexerKTile = 128;  // keys per indexer tile (block sizes must divide it)
constexpr int kTopkMaxK = 4096;

}  // namespace tsa
