// Block Sparse-GQA forward and backward.
//
// Megatron-LM issue #7060 "Add trainable QSA sparse attention with a TileLang
// backend" ("Describe the solution you'd like": Sparse-GQA forward and
// backward kernels over exact block top-k selections, BSHD and packed THD).
//
// Forward.  One CTA per (query t, kv group g) holds the group's Hq/Hkv query
// heads in a 16-row MMA tile; each selected block (block_size tokens of the
// group's k and v, causal inside the query's own block) streams through a
// double-buffered cp.async pipeline; online softmax, natural-log LSE.  The
// backward is key-centric (gqa_bwd_kv.cu).
#include "kernels.cuh"

namespace tsa {


// BS tokens per block, DH head dim.  4 warps.
template <int BS, int DH>
struct GqaSmem {
  static constexpr int RS = DH + 8;
  static constexpr int PRS = BS + 8;
};

// NST-stage cp.async ring of selected blocks (K and V tiles).
template <int BS, int DH, int NST>
__global__ void __launch_bounds__(128) gqa_fwd_mma_kernel(const __grid_constant__ GqaArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int RS = DH + 8, PRS = BS + 8;
  constexpr int KPW = BS / 4;        // keys per warp in S
  constexpr int NKT = KPW / 8;       // n-tiles per warp in S
  constexpr int CPW = DH / 4;        // channels per warp in PV
  constexpr int NTV = CPW / 8;
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [16][RS]
  __nv_bfloat16* Ks = Qs + 16 * RS;                                 // [NST][BS][RS]
  __nv_bfloat16* Vs = Ks + NST * BS * RS;                           // [NST][BS][RS]
  __nv_bfloat16* Ps = Vs + NST * BS * RS;                           // [16][PRS]
  float* red_max = reinterpret_cast<float*>(Ps + 16 * PRS);         // [4][16]
  float* red_sum = red_max + 64;
  int* s_blk = reinterpret_cast<int*>(red_sum + 64);                // [NST]

  const int t = blockIdx.x, gk = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, c4 = lane & 3;
  const int sq = seq_of(a.st, t);
  const int s0 = a.st.cu[sq];
  const int n = a.st.cu[sq + 1] - s0;
  const int p = t - s0;
  const int h0 = gk * a.G;
  const int* blk_row = a.blk + ((int64_t)t * a.Hkv + gk) * a.nsel;
  constexpr int CPR = DH / 8;

  for (int i = tid; i < 16 * CPR; i += 128) {
    int r = i / CPR, ch = i % CPR;
    bool ok = r < a.G;
    const __nv_bfloat16* src = a.q + ((int64_t)t * a.Hq + h0 + (ok ? r : 0)) * DH + ch * 8;
    cp_async16(smem_u32(Qs + r * RS + ch * 8), src, ok ? 16u : 0u);
  }
  auto gather = [&](int j, int buf) {
    int b = __ldg(blk_row + j);
    bool bok = b >= 0 && b * BS < n;
    if (b >= 0 && b * BS >= n && tid == 0) raise_flag(a.flags, TSA_FLAG_INDEX_RANGE);
    for (int i = tid; i < BS * CPR; i += 128) {
      int r = i / CPR, ch = i % CPR;
      int pos = b * BS + r;
      bool ok = bok && pos <= p;
      int64_t row = ((int64_t)(s0 + (ok ? pos : 0)) * a.Hkv + gk) * DH + ch * 8;
      cp_async16(smem_u32(Ks + (buf * BS + r) * RS + ch * 8), a.k + row, ok ? 16u : 0u);
      cp_async16(smem_u32(Vs + (buf * BS + r) * RS + ch * 8), a.v + row, ok ? 16u : 0u);
    }
    if (tid == 0) s_blk[buf] = bok ? b : -1;
  };
  // the q rows and the first NST - 1 blocks; one cp.async group per block
  // (empty groups past the last block keep the group count uniform)
#pragma unroll
  for (int j = 0; j < NST - 1; ++j) {
    if (j < a.nsel) gather(j, j);
    cp_async_commit();
  }

  const float NEG_INF = __int_as_float(0xff800000);
  float m_r[2] = {NEG_INF, NEG_INF}, l_r[2] = {0.f, 0.f};
  float o[NTV][4];
#pragma unroll
  for (int i = 0; i < NTV; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int j = 0; j < a.nsel; ++j) {
    const int buf = j % NST;
    // buffer (j + NST - 1) % NST was consumed in iteration j - 1 (closing barrier)
    if (j + NST - 1 < a.nsel) gather(j + NST - 1, (j + NST - 1) % NST);
    cp_async_commit();
    cp_async_wait<NST - 1>();  // block j has landed
    __syncthreads();
    const int b = s_blk[buf];
    const __nv_bfloat16* Kb = Ks + buf * BS * RS;
    const __nv_bfloat16* Vb = Vs + buf * BS * RS;
    float s[NKT][4];
#pragma unroll
    for (int i = 0; i < NKT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < DH / 16; ks += 2) {
      uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
      ldsm_x4(smem_u32(Qs + (lane & 15) * RS + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
      ldsm_x4(smem_u32(Qs + (lane & 15) * RS + (ks + 1) * 16 + (lane >> 4) * 8), a4, a5, a6, a7);
#pragma unroll
      for (int nk = 0; nk < NKT; ++nk) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(Kb + (warp * KPW + nk * 8 + (lane & 7)) * RS + ks * 16 + (lane >> 3) * 8), b0, b1, b2, b3);
        mma_bf16(s[nk], a0, a1, a2, a3, b0, b1);
        mma_bf16(s[nk], a4, a5, a6, a7, b2, b3);
      }
    }
    float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
    for (int nk = 0; nk < NKT; ++nk) {
      int key = warp * KPW + nk * 8 + 2 * c4;
      bool v0 = b >= 0 && b * BS + key <= p, v1 = b >= 0 && b * BS + key + 1 <= p;
      s[nk][0] = v0 ? s[nk][0] * a.scale_log2 : NEG_INF;
      s[nk][1] = v1 ? s[nk][1] * a.scale_log2 : NEG_INF;
      s[nk][2] = v0 ? s[nk][2] * a.scale_log2 : NEG_INF;
      s[nk][3] = v1 ? s[nk][3] * a.scale_log2 : NEG_INF;
      mx0 = fmaxf(mx0, fmaxf(s[nk][0], s[nk][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nk][2], s[nk][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    if (c4 == 0) { red_max[warp * 16 + gq] = mx0; red_max[warp * 16 + gq + 8] = mx1; }
    __syncthreads();
    float mnew[2], muse[2], alpha[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      int row = gq + rr * 8;
      float tm = fmaxf(fmaxf(red_max[row], red_max[16 + row]), fmaxf(red_max[32 + row], red_max[48 + row]));
      mnew[rr] = fmaxf(m_r[rr], tm);
      muse[rr] = mnew[rr] == NEG_INF ? 0.f : mnew[rr];
      alpha[rr] = exp2f(m_r[rr] - muse[rr]);
    }
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nk = 0; nk < NKT; ++nk) {
      float p0 = exp2f(s[nk][0] - muse[0]), p1 = exp2f(s[nk][1] - muse[0]);
      float p2 = exp2f(s[nk][2] - muse[1]), p3 = exp2f(s[nk][3] - muse[1]);
      ps0 += p0 + p1;
      ps1 += p2 + p3;
      int key = warp * KPW + nk * 8 + 2 * c4;
      *reinterpret_cast<uint32_t*>(Ps + gq * PRS + key) = pack_bf16(p0, p1);
      *reinterpret_cast<uint32_t*>(Ps + (gq + 8) * PRS + key) = pack_bf16(p2, p3);
    }
    ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
    ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
    ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
    ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
    if (c4 == 0) { red_sum[warp * 16 + gq] = ps0; red_sum[warp * 16 + gq + 8] = ps1; }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      int row = gq + rr * 8;
      float ts = (red_sum[row] + red_sum[16 + row]) + (red_sum[32 + row] + red_sum[48 + row]);
      l_r[rr] = l_r[rr] * alpha[rr] + ts;
      m_r[rr] = mnew[rr];
    }
#pragma unroll
    for (int nt = 0; nt < NTV; ++nt) {
      o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
    }
#pragma unroll
    for (int ks = 0; ks < BS / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(smem_u32(Ps + (lane & 15) * PRS + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NTV; nt += 2) {
        uint32_t b0, b1, b2, b3;
        int key = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        int ch = warp * CPW + nt * 8 + (lane >> 4) * 8;
        ldsm_x4_t(smem_u32(Vb + key * RS + ch), b0, b1, b2, b3);
        mma_bf16(o[nt], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[nt + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    int r = gq + rr * 8;
    if (r < a.G) {
      float inv = l_r[rr] > 0.f ? 1.f / l_r[rr] : 0.f;
      __nv_bfloat16* orow = a.out + ((int64_t)t * a.Hq + h0 + r) * DH + warp * CPW + 2 * c4;
#pragma unroll
      for (int nt = 0; nt < NTV; ++nt)
        *reinterpret_cast<uint32_t*>(orow + nt * 8) = pack_bf16(o[nt][2 * rr] * inv, o[nt][2 * rr + 1] * inv);
      if (warp == 0 && c4 == 0)
        a.lse[(int64_t)t * a.Hq + h0 + r] = l_r[rr] > 0.f ? (m_r[rr] + log2f(l_r[rr])) * kLn2 : NEG_INF;
    }
  }
}

template <int BS, int DH>
static cudaError_t launch_gqa_t(const GqaArgs& a, cudaStream_t stream) {
  constexpr int RS = DH + 8, PRS = BS + 8;
  constexpr int NST = 3;  // two blocks in flight per CTA, two CTAs per SM at BS = 64, DH = 128
  dim3 grid(a.T, a.Hkv);
  size_t smem = sizeof(__nv_bfloat16) * (16 * RS + 2 * NST * BS * RS + 16 * PRS) + sizeof(float) * 128 + 4 * NST;
  cudaError_t e = cudaFuncSetAttribute(gqa_fwd_mma_kernel<BS, DH, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  gqa_fwd_mma_kernel<BS, DH, NST><<<grid, 128, smem, stream>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_gqa(const GqaArgs& a, int bs, int d, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  if (bs == 64 && d == 128) return launch_gqa_t<64, 128>(a, stream);
  if (bs == 64 && d == 64) return launch_gqa_t<64, 64>(a, stream);
  if (bs == 32 && d == 128) return launch_gqa_t<32, 128>(a, stream);
  return launch_gqa_t<32, 64>(a, stream);
}

}  // namespace tsa
