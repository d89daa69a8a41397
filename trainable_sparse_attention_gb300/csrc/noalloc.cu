// qsa_topk_no_alloc: the streaming indexer + exact top-k with no workspace
// argument and no device allocation.
//
// Some callers cannot give this library device memory for scratch: hosts that
// forbid allocation once they are running (a fixed memory budget decided at
// start-up, an allocation-free serving loop, a plugin interface that hands the
// library only its input and output buffers).  For them this entry point keeps
// its score scratch in a file-scope device array of fixed size, so a call needs
// nothing beyond the inputs and the output indices.
//
// Properties a caller must know:
//  * the array (kNoAllocScratchBytes = 16 MiB) is part of the library image:
//    every GPU that loads the library holds it until the process exits;
//  * the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current and caches it; make that
//    first call before any stream capture;
//  * all calls share the one array: two calls whose kernels overlap on the GPU
//    (different streams, or different host threads on one device) race on it
//    and produce garbage -- serialise them;
//  * each call writes every scratch entry it later reads, so nothing needs
//    clearing and leftovers of an earlier call are never read;
//  * a problem whose single query row of scores (groups * row width * 4 bytes)
//    does not fit the array is refused with TSA_ERR_UNSUPPORTED; otherwise the
//    rows are processed in chunks that fit, and the indices are bit-identical
//    to qsa_topk's.
// No cudaMalloc, cudaFree or allocating library routine is called here.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "kernels.cuh"

using namespace tsa;

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

// The shared scratch.  In host code this name is only a stand-in for the
// device object; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return note_error(TSA_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return note_error(TSA_ERR_UNSUPPORTED, "device ordinal beyond 63");
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      return note_error(TSA_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e) : "null scratch address");
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TSA_OK;
}

}  // namespace

extern "C" int qsa_topk_no_alloc(const void* q_idx, const void* k_idx, const float* w, const int32_t* cu_seqlens,
                                 int num_seqs, int H_I, int d_I, int groups, int block_size, float score_scale,
                                 int topk, int32_t* indices, void* stream) {
  // ---- host-side validation (nothing is launched or looked up on failure):
  // the same checks, in the same helpers, as qsa_topk
  SeqTable st;
  int64_t T = 0;
  int rc = make_seq_table(cu_seqlens, num_seqs, &st, &T);
  if (rc != TSA_OK) return rc;
  if ((rc = check_indexer_shape(H_I, d_I, groups, block_size)) != TSA_OK) return rc;
  if (topk < 1 || topk > kTopkMaxK) return note_error(TSA_ERR_UNSUPPORTED, "topk must be 1..4096");
  const int max_len = st.max_len;
  const int64_t width = score_width(max_len, block_size);
  const int64_t row_bytes = int64_t(4) * groups * (width > 0 ? width : 1);
  if (row_bytes > static_cast<int64_t>(kNoAllocScratchBytes)) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "one query row of scores needs %lld bytes; the fixed scratch holds %zu (use qsa_topk with a workspace)",
             (long long)row_bytes, kNoAllocScratchBytes);
    return note_error(TSA_ERR_UNSUPPORTED, msg);
  }
  if (T == 0) return TSA_OK;
  if (!q_idx || !k_idx || !w || !indices) return note_error(TSA_ERR_INVALID_ARG, "null tensor pointer");

  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != TSA_OK) return rc;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t C = std::min<int64_t>(std::max<int64_t>(static_cast<int64_t>(kNoAllocScratchBytes) / row_bytes, 1),
                                      std::max(max_len, 1));
  for (int b = 0; b < num_seqs; ++b) {
    const int len = cu_seqlens[b + 1] - cu_seqlens[b];
    for (int64_t p0 = 0; p0 < len; p0 += C) {
      const int nq = static_cast<int>(std::min<int64_t>(C, len - p0));
      IndexerArgs a;
      a.q = static_cast<const __nv_bfloat16*>(q_idx);
      a.k = static_cast<const __nv_bfloat16*>(k_idx);
      a.w = w;
      a.H_I = H_I; a.d_I = d_I; a.groups = groups; a.bs = block_size;
      a.score_scale = score_scale;
      a.seq_start = cu_seqlens[b];
      a.p_begin = static_cast<int>(p0);
      a.nq = nq;
      a.out = static_cast<float*>(scratch);
      a.width = width;
      a.T_total = static_cast<int>(T);
      a.flags = device_flags();  // a bounded wait that gives up raises TSA_FLAG_TIMEOUT, as in qsa_topk
      cudaError_t e = launch_indexer(a, s);
      if (e != cudaSuccess) return note_error(TSA_ERR_CUDA, cudaGetErrorString(e));
      TopkRows r;
      r.scores = static_cast<const float*>(scratch); r.ld = width; r.width = width;
      r.mode = block_size == 1 ? 1 : 2;
      r.groups = groups; r.bs = block_size; r.p0 = p0;
      r.out = indices + (static_cast<int64_t>(cu_seqlens[b]) + p0) * groups * topk;
      r.out_ld = topk;
      r.k = topk;
      e = launch_topk_rows(r, static_cast<int64_t>(nq) * groups, s);
      if (e != cudaSuccess) return note_error(TSA_ERR_CUDA, cudaGetErrorString(e));
    }
  }
  return TSA_OK;
}
