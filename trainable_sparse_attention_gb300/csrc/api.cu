// C-ABI entry points of libtsa: argument validation, workspace carving and
// kernel launches.  No entry point allocates device memory or falls back to a
// different implementation: unsupported shapes are refused with a status code.
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "kernels.cuh"

using namespace tsa;

namespace {

// Error flag word raised by kernels (never a trap); read by tsa_read_flags.
__device__ unsigned int g_flags = 0;

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return TSA_OK;
  return fail(TSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define TSA_CHECK_CUDA(expr, where)            \
  do {                                         \
    cudaError_t _e = (expr);                   \
    if (_e != cudaSuccess) return cuda_status(_e, where); \
  } while (0)

// Kernels launched by this library since load (counted at every launch site).
std::atomic<unsigned long long> g_launches{0};

// A launcher call; its kernels count themselves (note_launch at each launch site).
#define TSA_LAUNCH(expr, where)                \
  do {                                         \
    cudaError_t _e = (expr);                   \
    if (_e != cudaSuccess) return cuda_status(_e, where); \
  } while (0)

// Score scratch of one query chunk of the streaming indexer + top-k.  Large
// enough that a chunk's top-k launch has thousands of rows (one CTA each) in
// flight; far below the T x T scores it replaces.
static constexpr int64_t kScoreChunkBytes = int64_t(512) << 20;

// Query rows per streamed chunk: the chunk's scores stay within kScoreChunkBytes.
int64_t chunk_rows(int max_len, int groups, int block_size) {
  int64_t w = score_width(max_len, block_size);
  if (w < 1) w = 1;
  int64_t c = kScoreChunkBytes / (4 * w * groups);
  c = (c / 128) * 128;
  if (c < 128) c = 128;
  if (c > max_len) c = max_len;
  if (c < 1) c = 1;
  return c;
}

}  // namespace

namespace tsa {
// Record a detail message for tsa_last_error() (entry points of other
// translation units), and account for a kernel launch (every launch site).
int note_error(int code, const char* msg) {
  g_last_error = msg;
  return code;
}
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

unsigned int* device_flags() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_flags) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<unsigned int*>(p);
}

// Validate cu_seqlens and fill the kernel-side table.
int make_seq_table(const int32_t* cu, int num_seqs, SeqTable* st, int64_t* T_out) {
  if (cu == nullptr) return fail(TSA_ERR_INVALID_ARG, "cu_seqlens is null");
  if (num_seqs < 1 || num_seqs > TSA_MAX_SEQS)
    return fail(TSA_ERR_INVALID_ARG, "num_seqs=%d outside [1, %d]", num_seqs, TSA_MAX_SEQS);
  if (cu[0] != 0) return fail(TSA_ERR_INVALID_ARG, "cu_seqlens[0]=%d, expected 0", cu[0]);
  st->num_seqs = num_seqs;
  st->max_len = 0;
  st->cu[0] = 0;
  for (int i = 1; i <= num_seqs; ++i) {
    if (cu[i] < cu[i - 1]) return fail(TSA_ERR_INVALID_ARG, "cu_seqlens not non-decreasing at %d", i);
    st->cu[i] = cu[i];
    int len = cu[i] - cu[i - 1];
    if (len > st->max_len) st->max_len = len;
  }
  *T_out = cu[num_seqs];
  return TSA_OK;
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int check_indexer_shape(int H_I, int d_I, int groups, int block_size) {
  if (!is_pow2(H_I) || H_I < 2 || H_I > 128)
    return fail(TSA_ERR_UNSUPPORTED, "H_I=%d: need a power of two in [2, 128]", H_I);
  if (d_I != 64 && d_I != 128) return fail(TSA_ERR_UNSUPPORTED, "d_I=%d: need 64 or 128", d_I);
  if (groups < 1 || H_I % groups != 0 || H_I / groups < 2)
    return fail(TSA_ERR_UNSUPPORTED, "groups=%d: need H_I/groups >= 2 and integral", groups);
  if (block_size != 1 && block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128)
    return fail(TSA_ERR_UNSUPPORTED, "block_size=%d: need 1, 16, 32, 64 or 128", block_size);
  return TSA_OK;
}

int64_t score_width(int max_len, int block_size) {
  return block_size == 1 ? max_len : (max_len + block_size - 1) / block_size;
}

}  // namespace tsa

extern "C" {

const char* tsa_status_string(int status) {
  switch (status) {
    case TSA_OK: return "TSA_OK";
    case TSA_ERR_INVALID_ARG: return "TSA_ERR_INVALID_ARG: invalid argument";
    case TSA_ERR_UNSUPPORTED: return "TSA_ERR_UNSUPPORTED: shape or option not built";
    case TSA_ERR_WORKSPACE: return "TSA_ERR_WORKSPACE: workspace missing or too small";
    case TSA_ERR_CUDA: return "TSA_ERR_CUDA: CUDA runtime error";
    case TSA_ERR_INDEX_RANGE: return "TSA_ERR_INDEX_RANGE: index outside its sequence";
    case TSA_ERR_TIMEOUT: return "TSA_ERR_TIMEOUT: bounded device wait expired";
    default: return "unknown tsa status";
  }
}

const char* tsa_last_error(void) { return g_last_error.c_str(); }

int tsa_version(void) { return 1; }

unsigned long long tsa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int tsa_read_flags(uint32_t* flags, int clear, void* stream) {
  if (flags == nullptr) return fail(TSA_ERR_INVALID_ARG, "flags is null");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  TSA_CHECK_CUDA(cudaMemcpyFromSymbolAsync(&v, g_flags, sizeof(v), 0, cudaMemcpyDeviceToHost, s), "read flags");
  TSA_CHECK_CUDA(cudaStreamSynchronize(s), "read flags sync");
  if (clear) {
    unsigned int z = 0;
    TSA_CHECK_CUDA(cudaMemcpyToSymbolAsync(g_flags, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s), "clear flags");
    TSA_CHECK_CUDA(cudaStreamSynchronize(s), "clear flags sync");
  }
  *flags = v;
  return TSA_OK;
}

int tsa_selftest_bounded_wait(void* stream) {
  unsigned int* f = device_flags();
  if (f == nullptr) return fail(TSA_ERR_CUDA, "device flag word unavailable");
  TSA_LAUNCH(launch_bounded_wait_selftest(f, static_cast<cudaStream_t>(stream)), "self-test launch");
  return TSA_OK;
}

// ---------------------------------------------------------------- indexer

int qsa_indexer_scores(const void* q_idx, const void* k_idx, const float* w, const int32_t* cu_seqlens,
                       int num_seqs, int H_I, int d_I, int groups, int block_size, float score_scale,
                       int64_t q_begin, int64_t q_count, float* scores, int64_t width, void* stream) {
  SeqTable st;
  int64_t T;
  int rc = make_seq_table(cu_seqlens, num_seqs, &st, &T);
  if (rc) return rc;
  if ((rc = check_indexer_shape(H_I, d_I, groups, block_size))) return rc;
  if (q_begin < 0 || q_count < 0 || q_begin + q_count > T)
    return fail(TSA_ERR_INVALID_ARG, "query range [%lld, %lld) outside [0, %lld)", (long long)q_begin,
                (long long)(q_begin + q_count), (long long)T);
  if (width < score_width(st.max_len, block_size))
    return fail(TSA_ERR_INVALID_ARG, "width=%lld < %lld", (long long)width,
                (long long)score_width(st.max_len, block_size));
  if (q_count == 0) return TSA_OK;
  if (!q_idx || !k_idx || !w || !scores) return fail(TSA_ERR_INVALID_ARG, "null tensor pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  TSA_LAUNCH(launch_fill(scores, q_count * groups * width, -INFINITY, s), "fill");
  for (int b = 0; b < num_seqs; ++b) {
    int64_t lo = std::max<int64_t>(q_begin, st.cu[b]);
    int64_t hi = std::min<int64_t>(q_begin + q_count, st.cu[b + 1]);
    if (lo >= hi) continue;
    IndexerArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q_idx);
    a.k = static_cast<const __nv_bfloat16*>(k_idx);
    a.w = w;
    a.H_I = H_I; a.d_I = d_I; a.groups = groups; a.bs = block_size;
    a.score_scale = score_scale;
    a.seq_start = st.cu[b];
    a.p_begin = static_cast<int>(lo - st.cu[b]);
    a.nq = static_cast<int>(hi - lo);
    a.out = scores + (lo - q_begin) * groups * width;
    a.width = width;
      a.T_total = static_cast<int>(T);
      a.flags = device_flags();
    TSA_LAUNCH(launch_indexer(a, s), "indexer launch");
  }
  return TSA_OK;
}

// ---------------------------------------------------------------- top-k

int qsa_topk_from_scores(const float* scores, int64_t rows, int64_t width, int64_t ld, int topk,
                         int32_t* indices, void* stream) {
  if (rows < 0 || width < 0 || ld < width) return fail(TSA_ERR_INVALID_ARG, "bad rows/width/ld");
  if (width > 0x7fffffffLL) return fail(TSA_ERR_UNSUPPORTED, "width beyond 2^31-1");
  if (rows > 0x7fffffffLL) return fail(TSA_ERR_UNSUPPORTED, "rows beyond 2^31-1");
  if (topk < 1 || topk > kTopkMaxK) return fail(TSA_ERR_UNSUPPORTED, "topk=%d outside [1, %d]", topk, kTopkMaxK);
  if (rows == 0) return TSA_OK;
  if (!scores || !indices) return fail(TSA_ERR_INVALID_ARG, "null tensor pointer");
  TopkRows a;
  a.scores = scores; a.ld = ld; a.width = width; a.mode = 0; a.groups = 1; a.bs = 1; a.p0 = 0;
  a.out = indices; a.out_ld = topk; a.k = topk;
  TSA_LAUNCH(launch_topk_rows(a, rows, static_cast<cudaStream_t>(stream)), "topk launch");
  return TSA_OK;
}

size_t qsa_topk_workspace_size(const int32_t* cu_seqlens, int num_seqs, int groups, int block_size) {
  SeqTable st;
  int64_t T;
  if (make_seq_table(cu_seqlens, num_seqs, &st, &T) || groups < 1 || block_size < 1) return 0;
  int64_t C = chunk_rows(st.max_len, groups, block_size);
  // two score buffers: the top-k of one chunk runs while the indexer fills the other
  return 2 * static_cast<size_t>(C * groups * score_width(st.max_len, block_size) * sizeof(float));
}

namespace {

// The two internal streams of the streamed indexer (per device, created on
// first use): the indexer's on the highest stream priority, so that its
// persistent CTAs take an SM as soon as one frees up, and the top-k's on the
// lowest, whose CTAs fill the room the indexer leaves.  Both fork from the
// caller's stream and join back into it with events, so the caller sees one
// ordered operation on its own stream.
struct TopkPipe {
  cudaStream_t idx = nullptr, sel = nullptr;
  cudaEvent_t start = nullptr, filled[2] = {nullptr, nullptr}, drained[2] = {nullptr, nullptr};
  cudaEvent_t joined[2] = {nullptr, nullptr};  // the ends of the two streams, waited by the caller's
};
constexpr int kMaxPipeDevices = 64;
TopkPipe g_pipes[kMaxPipeDevices];
std::mutex g_pipe_mu;

int topk_pipe(TopkPipe** out) {
  int dev = 0;
  TSA_CHECK_CUDA(cudaGetDevice(&dev), "current device");
  if (dev < 0 || dev >= kMaxPipeDevices) return fail(TSA_ERR_UNSUPPORTED, "device %d beyond the stream table", dev);
  TopkPipe& p = g_pipes[dev];
  if (p.idx == nullptr) {
    int least = 0, greatest = 0;
    TSA_CHECK_CUDA(cudaDeviceGetStreamPriorityRange(&least, &greatest), "stream priorities");
    TopkPipe q;
    TSA_CHECK_CUDA(cudaStreamCreateWithPriority(&q.idx, cudaStreamNonBlocking, greatest), "indexer stream");
    TSA_CHECK_CUDA(cudaStreamCreateWithPriority(&q.sel, cudaStreamNonBlocking, least), "top-k stream");
    TSA_CHECK_CUDA(cudaEventCreateWithFlags(&q.start, cudaEventDisableTiming), "event");
    for (int i = 0; i < 2; ++i) {
      TSA_CHECK_CUDA(cudaEventCreateWithFlags(&q.filled[i], cudaEventDisableTiming), "event");
      TSA_CHECK_CUDA(cudaEventCreateWithFlags(&q.drained[i], cudaEventDisableTiming), "event");
      TSA_CHECK_CUDA(cudaEventCreateWithFlags(&q.joined[i], cudaEventDisableTiming), "event");
    }
    p = q;
  }
  *out = &p;
  return TSA_OK;
}

}  // namespace

int qsa_topk(const void* q_idx, const void* k_idx, const float* w, const int32_t* cu_seqlens, int num_seqs,
             int H_I, int d_I, int groups, int block_size, float score_scale, int topk, int32_t* indices,
             void* workspace, size_t workspace_bytes, void* stream) {
  SeqTable st;
  int64_t T;
  int rc = make_seq_table(cu_seqlens, num_seqs, &st, &T);
  if (rc) return rc;
  if ((rc = check_indexer_shape(H_I, d_I, groups, block_size))) return rc;
  if (topk < 1 || topk > kTopkMaxK) return fail(TSA_ERR_UNSUPPORTED, "topk=%d outside [1, %d]", topk, kTopkMaxK);
  if (T == 0) return TSA_OK;
  if (!q_idx || !k_idx || !w || !indices) return fail(TSA_ERR_INVALID_ARG, "null tensor pointer");
  size_t need = qsa_topk_workspace_size(cu_seqlens, num_seqs, groups, block_size);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < %zu", workspace_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t C = chunk_rows(st.max_len, groups, block_size);
  const int64_t width = score_width(st.max_len, block_size);
  // Chunk i: the indexer writes score buffer i % 2 on the indexer stream, and
  // the top-k reads it on the top-k stream, which the indexer of chunk i + 2
  // waits for before it overwrites the buffer.
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  TopkPipe* pp = nullptr;
  if ((rc = topk_pipe(&pp))) return rc;
  cudaError_t fe = cudaEventRecord(pp->start, s);
  if (fe == cudaErrorInvalidResourceHandle || fe == cudaErrorContextIsDestroyed) {
    // the context that owned the streams and events is gone (the application
    // reset the device): make a new set for the current context
    cudaGetLastError();
    *pp = TopkPipe();
    if ((rc = topk_pipe(&pp))) return rc;
    fe = cudaEventRecord(pp->start, s);
  }
  TSA_CHECK_CUDA(fe, "fork");
  TSA_CHECK_CUDA(cudaStreamWaitEvent(pp->idx, pp->start, 0), "fork");
  TSA_CHECK_CUDA(cudaStreamWaitEvent(pp->sel, pp->start, 0), "fork");
  const size_t buf_floats = static_cast<size_t>(C) * groups * width;
  auto enqueue = [&]() -> int {
  int64_t chunk = 0;
  for (int b = 0; b < num_seqs; ++b) {
    const int len = st.cu[b + 1] - st.cu[b];
    for (int64_t p0 = 0; p0 < len; p0 += C, ++chunk) {
      const int nq = static_cast<int>(std::min<int64_t>(C, len - p0));
      const int nb = static_cast<int>(chunk & 1);
      float* scratch = static_cast<float*>(workspace) + nb * buf_floats;
      if (chunk >= 2) TSA_CHECK_CUDA(cudaStreamWaitEvent(pp->idx, pp->drained[nb], 0), "buffer reuse");
      IndexerArgs a;
      a.q = static_cast<const __nv_bfloat16*>(q_idx);
      a.k = static_cast<const __nv_bfloat16*>(k_idx);
      a.w = w;
      a.H_I = H_I; a.d_I = d_I; a.groups = groups; a.bs = block_size;
      a.score_scale = score_scale;
      a.seq_start = st.cu[b];
      a.p_begin = static_cast<int>(p0);
      a.nq = nq;
      a.out = scratch;
      a.width = width;
      a.T_total = static_cast<int>(T);
      a.flags = device_flags();
      TSA_LAUNCH(launch_indexer(a, pp->idx), "indexer launch");
      TSA_CHECK_CUDA(cudaEventRecord(pp->filled[nb], pp->idx), "chunk scored");
      TSA_CHECK_CUDA(cudaStreamWaitEvent(pp->sel, pp->filled[nb], 0), "chunk scored");
      TopkRows r;
      r.scores = scratch; r.ld = width; r.width = width;
      r.mode = block_size == 1 ? 1 : 2;
      r.groups = groups; r.bs = block_size; r.p0 = p0;
      r.out = indices + (st.cu[b] + p0) * groups * topk;
      r.out_ld = topk;
      r.k = topk;
      TSA_LAUNCH(launch_topk_rows(r, (int64_t)nq * groups, pp->sel), "topk launch");
      TSA_CHECK_CUDA(cudaEventRecord(pp->drained[nb], pp->sel), "chunk selected");
    }
  }
  return TSA_OK;
  };
  const int erc = enqueue();
  // join both streams into the caller's, also after a failed launch, so that
  // everything enqueued so far is ordered before the caller's next use of the
  // workspace and the indices
  cudaError_t je = cudaEventRecord(pp->joined[0], pp->idx);
  if (je == cudaSuccess) je = cudaEventRecord(pp->joined[1], pp->sel);
  if (je == cudaSuccess) je = cudaStreamWaitEvent(s, pp->joined[0], 0);
  if (je == cudaSuccess) je = cudaStreamWaitEvent(s, pp->joined[1], 0);
  if (erc) return erc;
  TSA_CHECK_CUDA(je, "join");
  return TSA_OK;
}

// ---------------------------------------------------------------- sparse MLA

static int check_mla(int64_t T, int H, int d_qk, int topk) {
  if (H < 1 || H > 128) return fail(TSA_ERR_UNSUPPORTED, "H=%d outside [1, 128]", H);
  if (d_qk != 512 && d_qk != 576) return fail(TSA_ERR_UNSUPPORTED, "d_qk=%d: need 512 or 576", d_qk);
  if (topk < 1) return fail(TSA_ERR_INVALID_ARG, "topk=%d < 1", topk);
  if (T > 0x7fffffffLL) return fail(TSA_ERR_UNSUPPORTED, "T beyond 2^31-1");
  return TSA_OK;
}

int sparse_mla_fwd(const void* q, const void* kv, const int32_t* indices, const int32_t* cu_seqlens, int num_seqs,
                   int H, int d_qk, int topk, float softmax_scale, void* out, float* lse, void* stream) {
  MlaFwdArgs a;
  int64_t T;
  int rc = make_seq_table(cu_seqlens, num_seqs, &a.st, &T);
  if (rc) return rc;
  if ((rc = check_mla(T, H, d_qk, topk))) return rc;
  if (T == 0) return TSA_OK;
  if (!q || !kv || !indices || !out || !lse) return fail(TSA_ERR_INVALID_ARG, "null tensor pointer");
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.kv = static_cast<const __nv_bfloat16*>(kv);
  a.idx = indices;
  a.T = static_cast<int>(T); a.H = H; a.topk = topk;
  a.scale_log2 = softmax_scale * kLog2e;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.flags = device_flags();
  TSA_LAUNCH(launch_mla_fwd(a, d_qk, static_cast<cudaStream_t>(stream)), "mla fwd launch");
  return TSA_OK;
}

// The 128-head backward stages P and dS of one chunk of queries in bf16
// ([query][head][slot], slots rounded up to 128) for the dKV GEMM; the chunk
// is sized so that the staging stays within kMlaStageBytes.
static constexpr int64_t kMlaStageBytes = int64_t(4) << 30;

static int64_t mla_kp(int topk) { return (static_cast<int64_t>(topk) + 127) / 128 * 128; }

static int64_t mla_bwd_chunk(int64_t T, int H, int topk) {
  if (H != 128) return 0;
  const int64_t per_query = static_cast<int64_t>(H) * mla_kp(topk) * 2 * sizeof(__nv_bfloat16);
  return std::max<int64_t>(1, std::min<int64_t>(T, kMlaStageBytes / per_query));
}

static size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

size_t sparse_mla_bwd_workspace_size(int64_t T, int H, int d_qk, int topk) {
  if (T < 0 || H < 1 || d_qk < 1 || topk < 1) return 0;
  size_t a = align256(static_cast<size_t>(T) * d_qk * sizeof(float));
  a += align256(static_cast<size_t>(T) * H * sizeof(float));
  const int64_t chunk = mla_bwd_chunk(T, H, topk);
  return a + static_cast<size_t>(chunk) * H * mla_kp(topk) * 2 * sizeof(__nv_bfloat16);
}

int sparse_mla_bwd(const void* q, const void* kv, const int32_t* indices, const void* out, const float* lse,
                   const void* dout, const int32_t* cu_seqlens, int num_seqs, int H, int d_qk, int topk,
                   float softmax_scale, void* dq, void* dkv, float* teacher, void* workspace,
                   size_t workspace_bytes, void* stream) {
  MlaBwdArgs a;
  int64_t T;
  int rc = make_seq_table(cu_seqlens, num_seqs, &a.st, &T);
  if (rc) return rc;
  if ((rc = check_mla(T, H, d_qk, topk))) return rc;
  if (T == 0) return TSA_OK;
  if (!q || !kv || !indices || !out || !lse || !dout || !dq || !dkv)
    return fail(TSA_ERR_INVALID_ARG, "null tensor pointer");
  size_t need = sparse_mla_bwd_workspace_size(T, H, d_qk, topk);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < %zu", workspace_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t dkv_bytes = align256(static_cast<size_t>(T) * d_qk * sizeof(float));
  const size_t dlt_bytes = align256(static_cast<size_t>(T) * H * sizeof(float));
  float* dkv_acc = static_cast<float*>(workspace);
  float* dlt = reinterpret_cast<float*>(static_cast<char*>(workspace) + dkv_bytes);
  TSA_CHECK_CUDA(cudaMemsetAsync(dkv_acc, 0, static_cast<size_t>(T) * d_qk * sizeof(float), s), "memset");
  TSA_LAUNCH(launch_bwd_delta(static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout),
                                  dlt, T * H, 512, s), "delta launch");
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.kv = static_cast<const __nv_bfloat16*>(kv);
  a.idx = indices;
  a.lse = lse;
  a.dlt = dlt;
  a.dout = static_cast<const __nv_bfloat16*>(dout);
  a.T = static_cast<int>(T); a.H = H; a.topk = topk;
  a.scale = softmax_scale;
  a.scale_log2 = softmax_scale * kLog2e;
  a.dq = static_cast<__nv_bfloat16*>(dq);
  a.dkv_acc = dkv_acc;
  if (H == 128) {
    // chunks of queries: P and dS (plus dQ) from the recompute kernel, then the dKV GEMM
    const int64_t chunk = mla_bwd_chunk(T, H, topk);
    const int64_t kp = mla_kp(topk);
    auto* stage = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(workspace) + dkv_bytes + dlt_bytes);
    a.kp = static_cast<int>(kp);
    a.flags = device_flags();
    a.p_out = stage;
    a.ds_out = stage + chunk * H * kp;
    MlaBwdTcArgs b;
    b.q = a.q;
    b.dout = a.dout;
    b.ds = a.ds_out;
    b.p = a.p_out;
    b.idx = indices;
    b.T = a.T; b.D = d_qk; b.topk = topk; b.kp = a.kp;
    b.dkv_acc = dkv_acc;
    b.flags = device_flags();
    b.st = a.st;
    b.teacher = d_qk == 576 ? teacher : nullptr;
    for (int64_t q0 = 0; q0 < T; q0 += chunk) {
      const int nq = static_cast<int>(std::min(chunk, T - q0));
      a.q0 = b.q0 = static_cast<int>(q0);
      TSA_LAUNCH(launch_mla_bwd_pds_tc(a, d_qk, nq, s), "mla bwd recompute launch");
      // the teacher comes out of the dKV GEMM's rope block for d_qk = 576, and
      // from a pass over the staged P otherwise
      if (teacher != nullptr && d_qk != 576)
        TSA_LAUNCH(launch_mla_teacher_from_p(a.p_out, nq, H, a.kp, topk, a.q0, teacher, s), "teacher launch");
      TSA_LAUNCH(launch_mla_bwd_dq_tc(a, d_qk, nq, s), "mla bwd dq launch");
      TSA_LAUNCH(launch_mla_bwd_dkv_tc(b, nq, s), "mla bwd dkv launch");
    }
  } else {
    if (teacher != nullptr) {
      TSA_CHECK_CUDA(cudaMemsetAsync(teacher, 0, static_cast<size_t>(T) * topk * sizeof(float), s), "memset");
      a.teacher = teacher;
    }
    TSA_LAUNCH(launch_mla_bwd(a, d_qk, s), "mla bwd launch");
  }
  TSA_LAUNCH(launch_f32_to_bf16(dkv_acc, static_cast<__nv_bfloat16*>(dkv), T * d_qk, s), "convert launch");
  return TSA_OK;
}

// ---------------------------------------------------------------- indexer training

static int check_indexer_sel(int64_t T, int H_I, int d_I, int topk) {
  if (!indexer_sel_supported(H_I, d_I))
    return fail(TSA_ERR_UNSUPPORTED, "H_I=%d d_I=%d: need d_I = 128 and 1 <= H_I <= 128", H_I, d_I);
  if (topk < 1 || topk > kTopkMaxK) return fail(TSA_ERR_UNSUPPORTED, "topk=%d outside [1, %d]", topk, kTopkMaxK);
  if (T > 0x7fffffffLL / 128) return fail(TSA_ERR_UNSUPPORTED, "T too large");
  return TSA_OK;
}

int qsa_indexer_kl(const void* q_idx, const void* k_idx, const float* w, const int32_t* cu_seqlens, int num_seqs,
                   int H_I, int d_I, float score_scale, const int32_t* indices, int topk, const float* teacher,
                   float* loss, float* dscore, void* stream) {
  IndexerSelArgs a;
  memset(static_cast<void*>(&a), 0, sizeof(a) - sizeof(SeqTable));
  int64_t T;
  int rc = make_seq_table(cu_seqlens, num_seqs, &a.st, &T);
  if (rc) return rc;
  if ((rc = check_indexer_sel(T, H_I, d_I, topk))) return rc;
  if (T == 0) return TSA_OK;
  if (!q_idx || !k_idx || !w || !indices || !teacher || !loss || !dscore)
    return fail(TSA_ERR_INVALID_ARG, "null tensor pointer");
  a.w = w;
  a.idx = indices;
  a.teacher = teacher;
  a.loss = loss;
  a.dscore_out = dscore;
  a.T = static_cast<int>(T); a.H_I = H_I; a.topk = topk;
  a.score_scale = score_scale;
  a.flags = device_flags();
  TSA_LAUNCH(launch_indexer_sel(a, q_idx, k_idx, false, static_cast<cudaStream_t>(stream)), "indexer kl launch");
  return TSA_OK;
}

size_t qsa_indexer_bwd_workspace_size(int64_t T, int d_I) {
  if (T < 0 || d_I < 1) return 0;
  return align256(static_cast<size_t>(T) * d_I * sizeof(float));
}

int qsa_indexer_bwd(const void* q_idx, const void* k_idx, const float* w, const int32_t* cu_seqlens, int num_seqs,
                    int H_I, int d_I, float score_scale, const int32_t* indices, int topk, const float* dscore,
                    void* dq_idx, void* dk_idx, float* dw, void* workspace, size_t workspace_bytes, void* stream) {
  IndexerSelArgs a;
  memset(static_cast<void*>(&a), 0, sizeof(a) - sizeof(SeqTable));
  int64_t T;
  int rc = make_seq_table(cu_seqlens, num_seqs, &a.st, &T);
  if (rc) return rc;
  if ((rc = check_indexer_sel(T, H_I, d_I, topk))) return rc;
  if (T == 0) return TSA_OK;
  if (!q_idx || !k_idx || !w || !indices || !dscore || !dq_idx || !dk_idx || !dw)
    return fail(TSA_ERR_INVALID_ARG, "null tensor pointer");
  const size_t need = qsa_indexer_bwd_workspace_size(T, d_I);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < %zu", workspace_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* dk_acc = static_cast<float*>(workspace);
  TSA_CHECK_CUDA(cudaMemsetAsync(dk_acc, 0, static_cast<size_t>(T) * d_I * sizeof(float), s), "memset");
  a.w = w;
  a.idx = indices;
  a.dscore = dscore;
  a.dq = static_cast<__nv_bfloat16*>(dq_idx);
  a.dw = dw;
  a.dk_acc = dk_acc;
  a.T = static_cast<int>(T); a.H_I = H_I; a.topk = topk;
  a.score_scale = score_scale;
  a.flags = device_flags();
  TSA_LAUNCH(launch_indexer_sel(a, q_idx, k_idx, true, s), "indexer bwd launch");
  TSA_LAUNCH(launch_f32_to_bf16(dk_acc, static_cast<__nv_bfloat16*>(dk_idx), T * d_I, s), "convert launch");
  return TSA_OK;
}

// ---------------------------------------------------------------- sparse GQA

static int check_gqa(int64_t T, int Hq, int Hkv, int d, int block_size, int nsel) {
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || Hq / Hkv > 16)
    return fail(TSA_ERR_UNSUPPORTED, "Hq=%d Hkv=%d: need Hq = G*Hkv with 1 <= G <= 16", Hq, Hkv);
  if (d != 64 && d != 128) return fail(TSA_ERR_UNSUPPORTED, "d=%d: need 64 or 128", d);
  if (block_size != 32 && block_size != 64) return fail(TSA_ERR_UNSUPPORTED, "block_size=%d: need 32 or 64", block_size);
  if (nsel < 1) return fail(TSA_ERR_INVALID_ARG, "nsel=%d < 1", nsel);
  if (T > 0x7fffffffLL) return fail(TSA_ERR_UNSUPPORTED, "T beyond 2^31-1");
  return TSA_OK;
}

// Workspace of the tcgen05 forward: the inverted selections and, per selection
// slot (t, g, j), the normalised partial output of its block (bf16, G x d) and
// its log2-sum-exp (fp32).
static size_t gqa_ws_align(size_t x) { return (x + 255) & ~size_t(255); }

static size_t gqa_inv_bytes(size_t t, int Hkv, int nsel) {
  const size_t nb = t * Hkv + 1;
  return gqa_ws_align(t * Hkv * nsel * sizeof(int)) + 4 * gqa_ws_align((nb + 1) * sizeof(int));
}

size_t sparse_gqa_fwd_workspace_size(int64_t T, int Hq, int Hkv, int d, int nsel) {
  if (T < 0 || Hq < 1 || Hkv < 1 || d < 1 || nsel < 1) return 0;
  const size_t t = static_cast<size_t>(T);
  return gqa_inv_bytes(t, Hkv, nsel) + gqa_ws_align(t * Hq * nsel * d * sizeof(__nv_bfloat16)) +
         gqa_ws_align(t * Hq * nsel * sizeof(float));
}

// Per-sequence first global block, and the total.
static int gqa_block_bases(const SeqTable& st, int block_size, int* base) {
  int nblk = 0;
  for (int i = 0; i < st.num_seqs; ++i) {
    base[i] = nblk;
    nblk += (st.cu[i + 1] - st.cu[i] + block_size - 1) / block_size;
  }
  base[st.num_seqs] = nblk;
  return nblk;
}

int sparse_gqa_fwd(const void* q, const void* k, const void* v, const int32_t* block_indices,
                   const int32_t* cu_seqlens, int num_seqs, int Hq, int Hkv, int d, int block_size, int nsel,
                   float softmax_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                   void* stream) {
  GqaTcArgs a;
  memset(static_cast<void*>(&a), 0, sizeof(a));
  int64_t T;
  int rc = make_seq_table(cu_seqlens, num_seqs, &a.st, &T);
  if (rc) return rc;
  if ((rc = check_gqa(T, Hq, Hkv, d, block_size, nsel))) return rc;
  if (T * Hkv * nsel > 0x7fffffffLL || T * Hq > 0x7fffffffLL)
    return fail(TSA_ERR_UNSUPPORTED, "T * Hkv * nsel or T * Hq beyond 2^31-1");
  if (T == 0) return TSA_OK;
  if (!q || !k || !v || !block_indices || !out || !lse) return fail(TSA_ERR_INVALID_ARG, "null tensor pointer");
  const size_t need = sparse_gqa_fwd_workspace_size(T, Hq, Hkv, d, nsel);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < %zu", workspace_bytes, need);
  a.nblk = gqa_block_bases(a.st, block_size, a.blk_base);
  const size_t t = static_cast<size_t>(T);
  a.nseg = 1;  // the forward writes partials, no reductions: one query segment
  a.qseg = static_cast<int>(T);
  const size_t nb = t * Hkv + 1;
  char* w = static_cast<char*>(workspace);
  auto take = [&](size_t bytes) { char* p = w; w += gqa_ws_align(bytes); return p; };
  a.list = reinterpret_cast<int*>(take(t * Hkv * nsel * sizeof(int)));
  a.cnt = reinterpret_cast<int*>(take((nb + 1) * sizeof(int)));
  a.off = reinterpret_cast<int*>(take((nb + 1) * sizeof(int)));
  a.cur = reinterpret_cast<int*>(take((nb + 1) * sizeof(int)));
  a.choff = reinterpret_cast<int*>(take((nb + 1) * sizeof(int)));
  a.part_o = reinterpret_cast<__nv_bfloat16*>(take(t * Hq * nsel * d * sizeof(__nv_bfloat16)));
  a.part_l = reinterpret_cast<float*>(take(t * Hq * nsel * sizeof(float)));
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.blk = block_indices;
  a.T = static_cast<int>(T); a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.nsel = nsel; a.bs = block_size; a.d = d;
  a.scale = softmax_scale;
  a.scale_log2 = softmax_scale * kLog2e;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.flags = device_flags();
  TSA_LAUNCH(launch_gqa_fwd_tc(a, static_cast<cudaStream_t>(stream)), "gqa fwd launch");
  return TSA_OK;
}

// Workspace of the key-centric backward: fp32 dQ, dK, dV accumulators, Delta,
// the inverted selections and their offsets.  At most one block per token, so
// T * Hkv bounds the number of (block, group) lists of one query segment.
//
// The backward's lists are split by query segment (up to 8) so that the CTAs
// running together reduce into one segment's slice of the fp32 dQ accumulator,
// about 48 MB or less: at the THD 32768 workload (537 MB of dQ) the reductions
// otherwise missed L2 and went to DRAM as read-modify-writes.
static int gqa_bwd_segments(int64_t T, int Hq, int d) {
  const int64_t dq_bytes = T * Hq * d * static_cast<int64_t>(sizeof(float));
  const int64_t want = (dq_bytes + (int64_t(48) << 20) - 1) / (int64_t(48) << 20);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(8, want)));
}

size_t sparse_gqa_bwd_workspace_size(int64_t T, int Hq, int Hkv, int d, int nsel) {
  if (T < 0 || Hq < 1 || Hkv < 1 || d < 1 || nsel < 1) return 0;
  const size_t t = static_cast<size_t>(T);
  const size_t nl = static_cast<size_t>(gqa_bwd_segments(T, Hq, d)) * (t * Hkv + 1);
  return gqa_ws_align(t * Hq * d * sizeof(float)) + 2 * gqa_ws_align(t * Hkv * d * sizeof(float)) +
         gqa_ws_align(t * Hq * sizeof(float)) + gqa_ws_align(t * Hkv * nsel * sizeof(int)) +
         4 * gqa_ws_align((nl + 1) * sizeof(int));
}

int sparse_gqa_bwd(const void* q, const void* k, const void* v, const int32_t* block_indices, const void* out,
                   const float* lse, const void* dout, const int32_t* cu_seqlens, int num_seqs, int Hq, int Hkv,
                   int d, int block_size, int nsel, float softmax_scale, void* dq, void* dk, void* dv,
                   void* workspace, size_t workspace_bytes, void* stream) {
  GqaTcArgs a;
  memset(static_cast<void*>(&a), 0, sizeof(a));
  int64_t T;
  int rc = make_seq_table(cu_seqlens, num_seqs, &a.st, &T);
  if (rc) return rc;
  if ((rc = check_gqa(T, Hq, Hkv, d, block_size, nsel))) return rc;
  if (T * Hkv * nsel > 0x7fffffffLL || T * Hq > 0x7fffffffLL)
    return fail(TSA_ERR_UNSUPPORTED, "T * Hkv * nsel or T * Hq beyond 2^31-1");
  if (T == 0) return TSA_OK;
  if (!q || !k || !v || !block_indices || !out || !lse || !dout || !dq || !dk || !dv)
    return fail(TSA_ERR_INVALID_ARG, "null tensor pointer");
  size_t need = sparse_gqa_bwd_workspace_size(T, Hq, Hkv, d, nsel);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < %zu", workspace_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  a.nblk = gqa_block_bases(a.st, block_size, a.blk_base);
  const size_t t = static_cast<size_t>(T);
  a.nseg = gqa_bwd_segments(T, Hq, d);
  while (a.nseg > 1 && static_cast<int64_t>(a.nseg) * a.nblk * Hkv >= 0x7fffffffLL) --a.nseg;  // int list indices
  a.qseg = static_cast<int>((T + a.nseg - 1) / a.nseg);
  const size_t nb = static_cast<size_t>(a.nseg) * (t * Hkv + 1);
  char* w = static_cast<char*>(workspace);
  auto take = [&](size_t bytes) { char* p = w; w += gqa_ws_align(bytes); return p; };
  float* dq_acc = reinterpret_cast<float*>(take(t * Hq * d * sizeof(float)));
  float* dk_acc = reinterpret_cast<float*>(take(t * Hkv * d * sizeof(float)));
  float* dv_acc = reinterpret_cast<float*>(take(t * Hkv * d * sizeof(float)));
  float* dlt = reinterpret_cast<float*>(take(t * Hq * sizeof(float)));
  a.list = reinterpret_cast<int*>(take(t * Hkv * nsel * sizeof(int)));
  a.cnt = reinterpret_cast<int*>(take((nb + 1) * sizeof(int)));
  a.off = reinterpret_cast<int*>(take((nb + 1) * sizeof(int)));
  a.cur = reinterpret_cast<int*>(take((nb + 1) * sizeof(int)));
  a.choff = reinterpret_cast<int*>(take((nb + 1) * sizeof(int)));
  TSA_CHECK_CUDA(cudaMemsetAsync(dq_acc, 0, t * Hq * d * sizeof(float), s), "memset");
  TSA_CHECK_CUDA(cudaMemsetAsync(dk_acc, 0, t * Hkv * d * sizeof(float), s), "memset");
  TSA_CHECK_CUDA(cudaMemsetAsync(dv_acc, 0, t * Hkv * d * sizeof(float), s), "memset");
  TSA_LAUNCH(launch_bwd_delta(static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout),
                              dlt, T * Hq, d, s), "delta launch");
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.dout = static_cast<const __nv_bfloat16*>(dout);
  a.blk = block_indices;
  a.lse_in = lse;
  a.dlt = dlt;
  a.T = static_cast<int>(T); a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.nsel = nsel; a.bs = block_size; a.d = d;
  a.scale = softmax_scale;
  a.scale_log2 = softmax_scale * kLog2e;
  a.dq_acc = dq_acc;
  a.dk_acc = dk_acc;
  a.dv_acc = dv_acc;
  a.flags = device_flags();
  TSA_LAUNCH(launch_gqa_bwd_tc(a, s), "gqa bwd launch");
  TSA_LAUNCH(launch_f32_to_bf16(dq_acc, static_cast<__nv_bfloat16*>(dq), (int64_t)(t * Hq * d), s), "convert");
  TSA_LAUNCH(launch_f32_to_bf16(dk_acc, static_cast<__nv_bfloat16*>(dk), (int64_t)(t * Hkv * d), s), "convert");
  TSA_LAUNCH(launch_f32_to_bf16(dv_acc, static_cast<__nv_bfloat16*>(dv), (int64_t)(t * Hkv * d), s), "convert");
  return TSA_OK;
}

}  // extern "C"
