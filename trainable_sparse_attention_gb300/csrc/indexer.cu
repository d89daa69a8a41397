// Indexer score kernel: I_g[t,s] = scale * sum_{h in g} w[t,h] * ReLU(q_I[t,h].k_I[s]),
// causal s <= t, optionally reduced to block maxima.
//
// Megatron-LM issue #7060 "Add trainable QSA sparse attention with a TileLang
// backend" ("Describe the solution you'd like": trainable indexer, ReLU scores,
// exact block top-k, streaming bounded-memory runner) and Megatron-LM PR #3674
// "Enable DSA CP/absorbed/THD paths with TileLang fused ops" (fused indexer
// forward + logits cleaning kernel).
//
// Both score kinds run on the tcgen05 kernel in indexer_tc.cu (token scores,
// and block maxima from the same MMAs with a cross-lane epilogue); this file
// routes the launch and holds the -inf fill of materialised score buffers.
#include "kernels.cuh"

namespace tsa {

// Scores for queries at local positions [p_begin, p_begin + nq) of one sequence:
// token scores, or block maxima when a.bs > 1.
cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t stream) {
  if (a.nq <= 0) return cudaSuccess;
  if (a.T_total <= 0 || !indexer_tc_supported(a.H_I, a.d_I, a.groups, a.bs)) return cudaErrorInvalidValue;
  return launch_indexer_tc(a, stream);
}

__global__ void fill_kernel(float* p, int64_t n, float v) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = v;
}

cudaError_t launch_fill(float* p, int64_t n, float v, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  fill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, n, v);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tsa
