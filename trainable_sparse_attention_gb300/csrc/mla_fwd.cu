// Sparse MLA forward over a query's selected latent rows.
//
// Megatron-LM PR #3674 "Enable DSA CP/absorbed/THD paths with TileLang fused
// ops" (sparse MLA forward over the absorbed latent) and Megatron-LM PR #7617
// "Support NoPE shapes and unaligned top-k in TileLang sparse MLA" ("What does
// this PR do?": q [T,H,576], kv latent, value = kv[..., :512], -1 slots,
// explicit scale, NoPE 512-wide inputs).
//
// Warp-level tensor-core variant (mma.sync m16n8k16), one CTA per (query, 16
// heads): the selected kv rows stream through a double-buffered cp.async
// gather (32 rows per tile), S = Q K^T and O += P V use the same staged rows
// (values are the first 512 channels), the softmax is online in the log2
// domain and the LSE is returned in natural log.  Slots >= topk and -1 slots
// are masked, so an unaligned topk needs no padding; d_qk = 512 simply runs a
// shorter K loop (identical to zero-padding the RoPE channels).
#include "kernels.cuh"

namespace tsa {

constexpr int MF_THREADS = 128;
constexpr int MF_KT = 32;   // keys per tile
constexpr int MF_HB = 16;   // heads per CTA
constexpr int MF_DV = 512;


template <int D>
__global__ void __launch_bounds__(MF_THREADS) mla_fwd_mma_kernel(const __grid_constant__ MlaFwdArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int RS = D + 8;
  constexpr int PRS = MF_KT + 8;
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [16][RS]
  __nv_bfloat16* KVs = Qs + MF_HB * RS;                             // [2][32][RS]
  __nv_bfloat16* Ps = KVs + 2 * MF_KT * RS;                         // [16][PRS]
  float* red_max = reinterpret_cast<float*>(Ps + MF_HB * PRS);      // [4][16]
  float* red_sum = red_max + 4 * MF_HB;                             // [4][16]

  const int t = blockIdx.x;
  const int h0 = blockIdx.y * MF_HB;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  const int sq = seq_of(a.st, t);
  const int s0 = a.st.cu[sq];
  const int n = a.st.cu[sq + 1] - s0;
  const int* idx_row = a.idx + (int64_t)t * a.topk;
  constexpr int CPR = D / 8;

  for (int i = tid; i < MF_HB * CPR; i += MF_THREADS) {
    int r = i / CPR, ch = i % CPR;
    bool ok = h0 + r < a.H;
    const __nv_bfloat16* src = a.q + ((int64_t)t * a.H + (ok ? h0 + r : 0)) * D + ch * 8;
    cp_async16(smem_u32(Qs + r * RS + ch * 8), src, ok ? 16u : 0u);
  }
  auto gather = [&](int jt, int buf) {
    __nv_bfloat16* dst = KVs + buf * MF_KT * RS;
    for (int i = tid; i < MF_KT * CPR; i += MF_THREADS) {
      int r = i / CPR, ch = i % CPR;
      int slot = jt * MF_KT + r;
      int id = slot < a.topk ? __ldg(idx_row + slot) : -1;
      bool ok = id >= 0 && id < n;
      const __nv_bfloat16* src = a.kv + (int64_t)(s0 + (ok ? id : 0)) * D + ch * 8;
      cp_async16(smem_u32(dst + r * RS + ch * 8), src, ok ? 16u : 0u);
    }
  };
  const int ntile = (a.topk + MF_KT - 1) / MF_KT;
  if (tid < MF_KT) {  // range check of every index word (flag only; the slot is masked)
    for (int s = tid; s < a.topk; s += MF_KT) {
      int id = __ldg(idx_row + s);
      if (id >= n) raise_flag(a.flags, TSA_FLAG_INDEX_RANGE);
    }
  }
  gather(0, 0);
  cp_async_commit();

  const float NEG_INF = __int_as_float(0xff800000);
  float m_r[2] = {NEG_INF, NEG_INF}, l_r[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int jt = 0; jt < ntile; ++jt) {
    const int buf = jt & 1;
    if (jt + 1 < ntile) { gather(jt + 1, buf ^ 1); cp_async_commit(); cp_async_wait<1>(); }
    else { cp_async_wait<0>(); }
    __syncthreads();
    const __nv_bfloat16* KVb = KVs + buf * MF_KT * RS;

    // S = Q K^T for keys 8*warp .. 8*warp+7
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int ks = 0; ks < D / 16; ks += 2) {
      uint32_t a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3;
      ldsm_x4(smem_u32(Qs + (lane & 15) * RS + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
      ldsm_x4(smem_u32(Qs + (lane & 15) * RS + (ks + 1) * 16 + (lane >> 4) * 8), a4, a5, a6, a7);
      ldsm_x4(smem_u32(KVb + (warp * 8 + (lane & 7)) * RS + ks * 16 + (lane >> 3) * 8), b0, b1, b2, b3);
      mma_bf16(s, a0, a1, a2, a3, b0, b1);
      mma_bf16(s, a4, a5, a6, a7, b2, b3);
    }
    const int slot0 = jt * MF_KT + warp * 8 + 2 * c4;
    bool v0 = false, v1 = false;
    if (slot0 < a.topk) { int id = __ldg(idx_row + slot0); v0 = id >= 0 && id < n; }
    if (slot0 + 1 < a.topk) { int id = __ldg(idx_row + slot0 + 1); v1 = id >= 0 && id < n; }
    float x[4];
    x[0] = v0 ? s[0] * a.scale_log2 : NEG_INF;
    x[1] = v1 ? s[1] * a.scale_log2 : NEG_INF;
    x[2] = v0 ? s[2] * a.scale_log2 : NEG_INF;
    x[3] = v1 ? s[3] * a.scale_log2 : NEG_INF;
    float mx0 = fmaxf(x[0], x[1]), mx1 = fmaxf(x[2], x[3]);
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    if (c4 == 0) { red_max[warp * MF_HB + g] = mx0; red_max[warp * MF_HB + g + 8] = mx1; }
    __syncthreads();
    float mnew[2], alpha[2], muse[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      int row = g + rr * 8;
      float tm = fmaxf(fmaxf(red_max[row], red_max[MF_HB + row]), fmaxf(red_max[2 * MF_HB + row], red_max[3 * MF_HB + row]));
      mnew[rr] = fmaxf(m_r[rr], tm);
      muse[rr] = (mnew[rr] == NEG_INF) ? 0.f : mnew[rr];
      alpha[rr] = exp2f(m_r[rr] - muse[rr]);
    }
    float p[4];
    p[0] = exp2f(x[0] - muse[0]);
    p[1] = exp2f(x[1] - muse[0]);
    p[2] = exp2f(x[2] - muse[1]);
    p[3] = exp2f(x[3] - muse[1]);
    float ps0 = p[0] + p[1], ps1 = p[2] + p[3];
    ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
    ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
    ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
    ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
    if (c4 == 0) { red_sum[warp * MF_HB + g] = ps0; red_sum[warp * MF_HB + g + 8] = ps1; }
    *reinterpret_cast<uint32_t*>(Ps + g * PRS + warp * 8 + 2 * c4) = pack_bf16(p[0], p[1]);
    *reinterpret_cast<uint32_t*>(Ps + (g + 8) * PRS + warp * 8 + 2 * c4) = pack_bf16(p[2], p[3]);
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      int row = g + rr * 8;
      float ts = (red_sum[row] + red_sum[MF_HB + row]) + (red_sum[2 * MF_HB + row] + red_sum[3 * MF_HB + row]);
      l_r[rr] = l_r[rr] * alpha[rr] + ts;
      m_r[rr] = mnew[rr];
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
    }
    // O[:, 128*warp .. +128) += P V
#pragma unroll
    for (int ks = 0; ks < MF_KT / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(smem_u32(Ps + (lane & 15) * PRS + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < 16; nt += 2) {
        uint32_t b0, b1, b2, b3;
        int key = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        int ch = warp * 128 + nt * 8 + (lane >> 4) * 8;
        ldsm_x4_t(smem_u32(KVb + key * RS + ch), b0, b1, b2, b3);
        mma_bf16(o[nt], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[nt + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    int h = h0 + g + rr * 8;
    float inv = l_r[rr] > 0.f ? 1.f / l_r[rr] : 0.f;
    if (h < a.H) {
      __nv_bfloat16* orow = a.out + ((int64_t)t * a.H + h) * MF_DV + warp * 128 + 2 * c4;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
        *reinterpret_cast<uint32_t*>(orow + nt * 8) = pack_bf16(o[nt][2 * rr] * inv, o[nt][2 * rr + 1] * inv);
      if (warp == 0 && c4 == 0)
        a.lse[(int64_t)t * a.H + h] = l_r[rr] > 0.f ? (m_r[rr] + log2f(l_r[rr])) * kLn2 : NEG_INF;
    }
  }
}

template <int D>
static size_t mla_fwd_smem() {
  return sizeof(__nv_bfloat16) * ((size_t)MF_HB * (D + 8) + 2 * MF_KT * (D + 8) + MF_HB * (MF_KT + 8)) +
         sizeof(float) * 8 * MF_HB;
}

// H > 32 runs on the tcgen05 cluster kernel (mla_fwd_tc.cu), heads padded to
// its 128 MMA rows; fewer heads, which would leave most of a 128-row MMA empty,
// run here (one CTA per query and 16 heads).
cudaError_t launch_mla_fwd(const MlaFwdArgs& a, int D, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  if (a.H > kMlaFwdTcMinHeads) return launch_mla_fwd_tc(a, D, stream);
  dim3 grid(a.T, (a.H + MF_HB - 1) / MF_HB);
  if (D == 576) {
    size_t smem = mla_fwd_smem<576>();
    cudaError_t e = cudaFuncSetAttribute(mla_fwd_mma_kernel<576>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mla_fwd_mma_kernel<576><<<grid, MF_THREADS, smem, stream>>>(a);
    note_launch();
  } else {
    size_t smem = mla_fwd_smem<512>();
    cudaError_t e = cudaFuncSetAttribute(mla_fwd_mma_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mla_fwd_mma_kernel<512><<<grid, MF_THREADS, smem, stream>>>(a);
    note_launch();
  }
  return cudaGetLastError();
}

}  // namespace tsa
