// Indexer score kernel: I_g[t,s] = scale * sum_{h in g} w[t,h] * ReLU(q_I[t,h].k_I[s]),
// causal s <= t, optionally reduced to block maxima.
//
// Megatron-LM issue #7060 "Add trainable QSA sparse attention with a TileLang
// backend" ("Describe the solution you'd like": trainable indexer, ReLU scores,
// exact block top-k, streaming bounded-memory runner) and Megatron-LM PR #3674
// "Enable DSA CP/absorbed/THD paths with TileLang fused ops" (fused indexer
// forward + logits cleaning kernel).
//
// This is the warp-level tensor-core (mma.sync m16n8k16) variant:
//  * keys sit on the MMA's M side (16 per warp, 128 per CTA tile) and the
//    CTA's (query, head) pairs on N (128 columns), K = d_I;
//  * the epilogue applies ReLU and the head weight and reduces each group's
//    heads inside a thread quad, so a (query, group, key) score never leaves
//    registers before it is final; masked ("cleaned") logits are never written;
//  * the q_I block stays in shared memory while key tiles stream through a
//    double-buffered cp.async pipeline.
#include "kernels.cuh"

namespace tsa {

constexpr int IX_THREADS = 256;   // 8 warps x 16 keys
constexpr int IX_KTILE = 128;     // keys per tile
constexpr int IX_NCOL = 128;      // (query, head) columns per CTA
constexpr int IX_KT_PER_CTA = 8;  // key tiles streamed per CTA


__global__ void __launch_bounds__(IX_THREADS) indexer_mma_kernel(IndexerArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int d = a.d_I;
  const int RS = d + 8;  // padded row stride (elements) -> conflict-free ldmatrix
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* Ks = Qs + IX_NCOL * RS;                       // [2][128][RS]
  float* Ws = reinterpret_cast<float*>(Ks + 2 * IX_KTILE * RS);  // [128]
  float* Sc = Ws + IX_NCOL;                                    // [segments][128]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int QB = IX_NCOL / a.H_I;
  const int hg = a.H_I / a.groups;
  const int nseg = IX_NCOL / hg;
  const int q0 = blockIdx.y * QB;
  const int qn = min(QB, a.nq - q0);
  const int p_last = a.p_begin + q0 + qn - 1;
  const int p_first = a.p_begin + q0;
  const int kt0 = blockIdx.x * IX_KT_PER_CTA;
  if (kt0 * IX_KTILE > p_last) return;
  const int kt_end = min(kt0 + IX_KT_PER_CTA, p_last / IX_KTILE + 1);

  // q_I block + head weights
  const int cpr = d / 8;  // 16-byte chunks per row
  for (int i = tid; i < IX_NCOL * cpr; i += IX_THREADS) {
    int c = i / cpr, ch = i % cpr;
    int qq = c / a.H_I, h = c % a.H_I;
    bool ok = qq < qn;
    int64_t t = a.seq_start + a.p_begin + q0 + (ok ? qq : 0);
    const __nv_bfloat16* src = a.q + (t * a.H_I + h) * d + ch * 8;
    cp_async16(smem_u32(Qs + c * RS + ch * 8), src, ok ? 16u : 0u);
  }
  for (int c = tid; c < IX_NCOL; c += IX_THREADS) {
    int qq = c / a.H_I, h = c % a.H_I;
    Ws[c] = (qq < qn) ? a.w[(int64_t)(a.seq_start + a.p_begin + q0 + qq) * a.H_I + h] : 0.f;
  }
  auto load_tile = [&](int kt, int buf) {
    __nv_bfloat16* dst = Ks + buf * IX_KTILE * RS;
    for (int i = tid; i < IX_KTILE * cpr; i += IX_THREADS) {
      int r = i / cpr, ch = i % cpr;
      int s = kt * IX_KTILE + r;
      bool ok = s <= p_last;
      const __nv_bfloat16* src = a.k + (int64_t)(a.seq_start + (ok ? s : 0)) * d + ch * 8;
      cp_async16(smem_u32(dst + r * RS + ch * 8), src, ok ? 16u : 0u);
    }
  };
  load_tile(kt0, 0);
  cp_async_commit();

  const int g = lane >> 2, c4 = lane & 3;
  const float NEG_INF = __int_as_float(0xff800000);
  for (int kt = kt0; kt < kt_end; ++kt) {
    const int buf = (kt - kt0) & 1;
    if (kt + 1 < kt_end) { load_tile(kt + 1, buf ^ 1); cp_async_commit(); cp_async_wait<1>(); }
    else { cp_async_wait<0>(); }
    __syncthreads();

    float acc[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    const __nv_bfloat16* Kb = Ks + buf * IX_KTILE * RS + warp * 16 * RS;
    for (int ks = 0; ks < d / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(smem_u32(Kb + (lane & 15) * RS + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
#pragma unroll
      for (int np = 0; np < 8; ++np) {  // pairs of n-tiles (16 columns)
        uint32_t b0, b1, b2, b3;
        // matrices: cols np*16+0..7 (k lo, k hi), cols np*16+8..15 (k lo, k hi)
        int col = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        int kof = ks * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4(smem_u32(Qs + col * RS + kof), b0, b1, b2, b3);
        mma_bf16(acc[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }

    // epilogue: per (segment, key) sums of w * ReLU(dot)
    const int key_r0 = warp * 16 + g, key_r1 = key_r0 + 8;
    float seg0 = 0.f, seg1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      int c0 = nt * 8 + 2 * c4;
      float w0 = Ws[c0], w1 = Ws[c0 + 1];
      float v0 = w0 * fmaxf(acc[nt][0], 0.f) + w1 * fmaxf(acc[nt][1], 0.f);
      float v1 = w0 * fmaxf(acc[nt][2], 0.f) + w1 * fmaxf(acc[nt][3], 0.f);
      if (hg == 2) {
        int sg = c0 >> 1;
        Sc[sg * IX_KTILE + key_r0] = v0 * a.score_scale + 0.f;
        Sc[sg * IX_KTILE + key_r1] = v1 * a.score_scale + 0.f;
      } else if (hg == 4) {
        v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        if ((c4 & 1) == 0) {
          int sg = c0 >> 2;
          Sc[sg * IX_KTILE + key_r0] = v0 * a.score_scale + 0.f;
          Sc[sg * IX_KTILE + key_r1] = v1 * a.score_scale + 0.f;
        }
      } else {
        seg0 += v0;
        seg1 += v1;
        int per = hg >> 3;  // n-tiles per segment
        if ((nt % per) == per - 1) {
          seg0 += __shfl_xor_sync(0xffffffffu, seg0, 1);
          seg0 += __shfl_xor_sync(0xffffffffu, seg0, 2);
          seg1 += __shfl_xor_sync(0xffffffffu, seg1, 1);
          seg1 += __shfl_xor_sync(0xffffffffu, seg1, 2);
          if (c4 == 0) {
            int sg = nt / per;
            Sc[sg * IX_KTILE + key_r0] = seg0 * a.score_scale + 0.f;
            Sc[sg * IX_KTILE + key_r1] = seg1 * a.score_scale + 0.f;
          }
          seg0 = seg1 = 0.f;
        }
      }
    }
    __syncthreads();

    // output: causal part only
    const int sbase = kt * IX_KTILE;
    if (a.bs == 1) {
      for (int i = tid; i < nseg * IX_KTILE; i += IX_THREADS) {
        int sg = i / IX_KTILE, j = i % IX_KTILE;
        int qq = sg / a.groups, gg = sg % a.groups;
        int s = sbase + j;
        if (qq < qn && s <= a.p_begin + q0 + qq)
          a.out[((int64_t)(q0 + qq) * a.groups + gg) * a.width + s] = Sc[i];
      }
    } else {
      const int nbt = IX_KTILE / a.bs;
      for (int i = tid; i < nseg * nbt; i += IX_THREADS) {
        int sg = i / nbt, bl = i % nbt;
        int qq = sg / a.groups, gg = sg % a.groups;
        if (qq >= qn) continue;
        int p = a.p_begin + q0 + qq;
        int s_lo = sbase + bl * a.bs;
        if (s_lo > p) continue;
        float m = NEG_INF;
        int jmax = min(a.bs, p - s_lo + 1);
        for (int j = 0; j < jmax; ++j) m = fmaxf(m, Sc[sg * IX_KTILE + bl * a.bs + j]);
        a.out[((int64_t)(q0 + qq) * a.groups + gg) * a.width + s_lo / a.bs] = m;
      }
    }
    __syncthreads();
  }
  (void)p_first;
}

size_t indexer_smem_bytes(int d_I, int H_I, int groups) {
  int RS = d_I + 8;
  int hg = H_I / groups;
  return sizeof(__nv_bfloat16) * (size_t)(IX_NCOL * RS + 2 * IX_KTILE * RS) +
         sizeof(float) * (IX_NCOL + (size_t)(IX_NCOL / hg) * IX_KTILE);
}

// Scores for queries at local positions [p_begin, p_begin + nq) of one sequence.
// Token-level scores run on the tcgen05 kernel (indexer_tc.cu); block scores
// (max over a block's causal tokens) run here.
cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t stream) {
  if (a.nq <= 0) return cudaSuccess;
  if (a.T_total > 0 && indexer_tc_supported(a.H_I, a.d_I, a.groups, a.bs)) return launch_indexer_tc(a, stream);
  size_t smem = indexer_smem_bytes(a.d_I, a.H_I, a.groups);
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(indexer_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr_set = true;
  }
  int QB = IX_NCOL / a.H_I;
  int p_last = a.p_begin + a.nq - 1;
  int ktiles = p_last / IX_KTILE + 1;
  dim3 grid((ktiles + IX_KT_PER_CTA - 1) / IX_KT_PER_CTA, (a.nq + QB - 1) / QB);
  indexer_mma_kernel<<<grid, IX_THREADS, smem, stream>>>(a);
  note_launch();
  return cudaGetLastError();
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
