// Sparse MLA backward.
//
// Megatron-LM PR #3674 "Enable DSA CP/absorbed/THD paths with TileLang fused
// ops" (sparse MLA backward kernels) and Megatron-LM PR #7617 "Support NoPE
// shapes and unaligned top-k in TileLang sparse MLA" ("Validation": the
// backward accumulates atomically, so it is checked numerically rather than
// replayed bit for bit).
//
//   P = exp(scale*S - lse), dP = dO V^T, Dlt = rowsum(dO * O),
//   dS = P (dP - Dlt), dQ = scale dS K, dKV[idx] += scale dS^T Q + [P^T dO | 0].
//
// Three launches: (1) Dlt per (t, h); (2) one CTA per (query, head block)
// recomputes S/P from the stored LSE, keeps dQ in registers and scatters its
// dKV tile contribution with 16-byte vector reductions into an fp32
// workspace; (3) fp32 -> bf16 conversion of dKV.  Warp-level tensor-core
// (mma.sync) kernel for H < 128; 128 heads take the tcgen05 kernels
// (mla_bwd_pds_tc.cu, mla_bwd_tc.cu) between the same first and last launch.
#include "kernels.cuh"

namespace tsa {

constexpr int MB_KT = 32;  // keys per tile
constexpr int MB_DV = 512;


// Dlt[t,h] = sum_c dO[t,h,c] * O[t,h,c]; one warp per (t, h) row of `dv` channels.
__global__ void bwd_delta_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                                 float* __restrict__ dlt, int64_t rows, int dv) {
  int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const __nv_bfloat16* a = o + row * dv;
  const __nv_bfloat16* b = dout + row * dv;
  float acc = 0.f;
  for (int c = lane * 8; c < dv; c += 256) {
    uint4 va = *reinterpret_cast<const uint4*>(a + c);
    uint4 vb = *reinterpret_cast<const uint4*>(b + c);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&va);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&vb);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 fa = __bfloat1622float2(pa[j]), fb = __bfloat1622float2(pb[j]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) dlt[row] = acc;
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, int64_t n) {
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < n; i += (int64_t)gridDim.x * blockDim.x * 4) {
    if (i + 3 < n) {
      float4 v = *reinterpret_cast<const float4*>(src + i);
      uint2 pk;
      pk.x = pack_bf16(v.x, v.y);
      pk.y = pack_bf16(v.z, v.w);
      *reinterpret_cast<uint2*>(dst + i) = pk;
    } else {
      for (int64_t j = i; j < n; ++j) dst[j] = __float2bfloat16_rn(src[j]);
    }
  }
}

// MW m-tiles of 16 heads per CTA (HB = 16*MW heads), 4*MW warps.
template <int D, int MW>
__global__ void __launch_bounds__(128 * MW) mla_bwd_mma_kernel(const __grid_constant__ MlaBwdArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int HB = 16 * MW;
  constexpr int NW = 4 * MW;
  constexpr int NTHR = 128 * MW;
  constexpr int RS = D + 8;
  constexpr int ORS = MB_DV + 8;
  constexpr int PRS = MB_KT + 8;
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [HB][RS]
  __nv_bfloat16* dOs = Qs + HB * RS;                                // [HB][ORS]
  __nv_bfloat16* KVs = dOs + HB * ORS;                              // [2][32][RS]
  __nv_bfloat16* Ps = KVs + 2 * MB_KT * RS;                         // [HB][PRS]
  __nv_bfloat16* dSs = Ps + HB * PRS;                               // [HB][PRS]
  int* s_rows = reinterpret_cast<int*>(dSs + HB * PRS);             // [2][32] kv row or -1

  const int t = blockIdx.x;
  const int h0 = blockIdx.y * HB;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  const int sq = seq_of(a.st, t);
  const int s0 = a.st.cu[sq];
  const int n = a.st.cu[sq + 1] - s0;
  const int* idx_row = a.idx + (int64_t)t * a.topk;
  constexpr int CPR = D / 8;
  constexpr int OCPR = MB_DV / 8;

  for (int i = tid; i < HB * CPR; i += NTHR) {
    int r = i / CPR, ch = i % CPR;
    bool ok = h0 + r < a.H;
    const __nv_bfloat16* src = a.q + ((int64_t)t * a.H + (ok ? h0 + r : 0)) * D + ch * 8;
    cp_async16(smem_u32(Qs + r * RS + ch * 8), src, ok ? 16u : 0u);
  }
  for (int i = tid; i < HB * OCPR; i += NTHR) {
    int r = i / OCPR, ch = i % OCPR;
    bool ok = h0 + r < a.H;
    const __nv_bfloat16* src = a.dout + ((int64_t)t * a.H + (ok ? h0 + r : 0)) * MB_DV + ch * 8;
    cp_async16(smem_u32(dOs + r * ORS + ch * 8), src, ok ? 16u : 0u);
  }
  auto gather = [&](int jt, int buf) {
    __nv_bfloat16* dst = KVs + buf * MB_KT * RS;
    for (int i = tid; i < MB_KT * CPR; i += NTHR) {
      int r = i / CPR, ch = i % CPR;
      int slot = jt * MB_KT + r;
      int id = slot < a.topk ? __ldg(idx_row + slot) : -1;
      bool ok = id >= 0 && id < n;
      const __nv_bfloat16* src = a.kv + (int64_t)(s0 + (ok ? id : 0)) * D + ch * 8;
      cp_async16(smem_u32(dst + r * RS + ch * 8), src, ok ? 16u : 0u);
    }
    if (tid < MB_KT) {
      int slot = jt * MB_KT + tid;
      int id = slot < a.topk ? __ldg(idx_row + slot) : -1;
      s_rows[buf * MB_KT + tid] = (id >= 0 && id < n) ? s0 + id : -1;
    }
  };
  gather(0, 0);
  cp_async_commit();

  // per-thread row constants for the S/dP phase: m-tile mt, rows g / g+8
  const int mt = warp / 4, kq = warp % 4;
  float lse2[2], dl[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    int h = h0 + mt * 16 + g + rr * 8;
    float L = (h < a.H) ? a.lse[(int64_t)t * a.H + h] : __int_as_float(0xff800000);
    lse2[rr] = L * kLog2e;
    dl[rr] = (h < a.H) ? a.dlt[(int64_t)t * a.H + h] : 0.f;
  }
  constexpr int NTQ = D / 32;  // dQ n-tiles per warp (quarter of D)
  float dq[NTQ][4];
#pragma unroll
  for (int i = 0; i < NTQ; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;

  const int ntile = (a.topk + MB_KT - 1) / MB_KT;
  for (int jt = 0; jt < ntile; ++jt) {
    const int buf = jt & 1;
    if (jt + 1 < ntile) { gather(jt + 1, buf ^ 1); cp_async_commit(); cp_async_wait<1>(); }
    else { cp_async_wait<0>(); }
    __syncthreads();
    const __nv_bfloat16* KVb = KVs + buf * MB_KT * RS;
    const int* rows_b = s_rows + buf * MB_KT;

    // S and dP for rows mt*16.., keys 8*kq..
    float s[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
    const __nv_bfloat16* Qm = Qs + mt * 16 * RS;
    const __nv_bfloat16* dOm = dOs + mt * 16 * ORS;
#pragma unroll 4
    for (int ks = 0; ks < D / 16; ks += 2) {
      uint32_t a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3;
      ldsm_x4(smem_u32(Qm + (lane & 15) * RS + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
      ldsm_x4(smem_u32(Qm + (lane & 15) * RS + (ks + 1) * 16 + (lane >> 4) * 8), a4, a5, a6, a7);
      ldsm_x4(smem_u32(KVb + (kq * 8 + (lane & 7)) * RS + ks * 16 + (lane >> 3) * 8), b0, b1, b2, b3);
      mma_bf16(s, a0, a1, a2, a3, b0, b1);
      mma_bf16(s, a4, a5, a6, a7, b2, b3);
    }
#pragma unroll 4
    for (int ks = 0; ks < MB_DV / 16; ks += 2) {
      uint32_t a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3;
      ldsm_x4(smem_u32(dOm + (lane & 15) * ORS + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
      ldsm_x4(smem_u32(dOm + (lane & 15) * ORS + (ks + 1) * 16 + (lane >> 4) * 8), a4, a5, a6, a7);
      ldsm_x4(smem_u32(KVb + (kq * 8 + (lane & 7)) * RS + ks * 16 + (lane >> 3) * 8), b0, b1, b2, b3);
      mma_bf16(dp, a0, a1, a2, a3, b0, b1);
      mma_bf16(dp, a4, a5, a6, a7, b2, b3);
    }
    const int key0 = kq * 8 + 2 * c4;
    const bool v0 = rows_b[key0] >= 0, v1 = rows_b[key0 + 1] >= 0;
    float P[4], dS[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int rr = i >> 1;
      bool v = (i & 1) ? v1 : v0;
      P[i] = (v && lse2[rr] != __int_as_float(0xff800000)) ? exp2f(s[i] * a.scale_log2 - lse2[rr]) : 0.f;
      dS[i] = a.scale * P[i] * (dp[i] - dl[rr]);
    }
    const int prow = mt * 16 + g;
    *reinterpret_cast<uint32_t*>(Ps + prow * PRS + key0) = pack_bf16(P[0], P[1]);
    *reinterpret_cast<uint32_t*>(Ps + (prow + 8) * PRS + key0) = pack_bf16(P[2], P[3]);
    *reinterpret_cast<uint32_t*>(dSs + prow * PRS + key0) = pack_bf16(dS[0], dS[1]);
    *reinterpret_cast<uint32_t*>(dSs + (prow + 8) * PRS + key0) = pack_bf16(dS[2], dS[3]);
    __syncthreads();
    if (a.teacher != nullptr && tid < MB_KT) {
      // indexer teacher: this head block's share of the head mean of P at the tile's slots
      const int slot = jt * MB_KT + tid;
      if (slot < a.topk) {
        float sp = 0.f;
        for (int h = 0; h < HB; ++h) sp += __bfloat162float(Ps[h * PRS + tid]);
        if (sp != 0.f) atomicAdd(a.teacher + (int64_t)t * a.topk + slot, sp / static_cast<float>(a.H));
      }
    }

    // dQ[mt rows, quarter kq of D] += (scale dS) K
    {
      const __nv_bfloat16* dSm = dSs + mt * 16 * PRS;
#pragma unroll
      for (int ks = 0; ks < MB_KT / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(smem_u32(dSm + (lane & 15) * PRS + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NTQ; nt += 2) {
          uint32_t b0, b1, b2, b3;
          int key = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          int ch = kq * (D / 4) + nt * 8 + (lane >> 4) * 8;
          ldsm_x4_t(smem_u32(KVb + key * RS + ch), b0, b1, b2, b3);
          mma_bf16(dq[nt], a0, a1, a2, a3, b0, b1);
          mma_bf16(dq[nt + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    // dKV tile [32 keys x D] = (scale dS)^T Q + P^T dO, channels split across warps
    {
      constexpr int CPW = D / NW;     // channels per warp
      constexpr int NTK = CPW / 8;    // n-tiles per warp
#pragma unroll 1
      for (int nt = 0; nt < NTK; ++nt) {
        const int ch0 = warp * CPW + nt * 8;
        float acc[2][4];
#pragma unroll
        for (int m2 = 0; m2 < 2; ++m2) acc[m2][0] = acc[m2][1] = acc[m2][2] = acc[m2][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < MW; ++ks) {  // 16 heads per k-step
          uint32_t b0, b1, c0, c1;
          // B = Q[heads ks*16.., ch0..ch0+8) (k = heads, n = channels), stored [head][ch] -> trans
          ldsm_x2_t(smem_u32(Qs + (ks * 16 + (lane & 15)) * RS + ch0), b0, b1);
          const bool has_v = ch0 < MB_DV;
          if (has_v) ldsm_x2_t(smem_u32(dOs + (ks * 16 + (lane & 15)) * ORS + ch0), c0, c1);
#pragma unroll
          for (int m2 = 0; m2 < 2; ++m2) {
            uint32_t a0, a1, a2, a3;
            // A = dS^T[keys m2*16.., heads ks*16..]: stored [head][key] -> trans
            int hrow = ks * 16 + (lane & 7) + (lane >> 4) * 8;
            int kcol = m2 * 16 + ((lane >> 3) & 1) * 8;
            ldsm_x4_t(smem_u32(dSs + hrow * PRS + kcol), a0, a1, a2, a3);
            mma_bf16(acc[m2], a0, a1, a2, a3, b0, b1);
            if (has_v) {
              ldsm_x4_t(smem_u32(Ps + hrow * PRS + kcol), a0, a1, a2, a3);
              mma_bf16(acc[m2], a0, a1, a2, a3, c0, c1);
            }
          }
        }
#pragma unroll
        for (int m2 = 0; m2 < 2; ++m2) {
          const int r0 = rows_b[m2 * 16 + g], r1 = rows_b[m2 * 16 + g + 8];
          red_frag_v4(r0 >= 0 ? a.dkv_acc + (int64_t)r0 * D + ch0 : nullptr,
                      r1 >= 0 ? a.dkv_acc + (int64_t)r1 * D + ch0 : nullptr, acc[m2], c4);
        }
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    int h = h0 + mt * 16 + g + rr * 8;
    if (h < a.H) {
      __nv_bfloat16* drow = a.dq + ((int64_t)t * a.H + h) * D + kq * (D / 4) + 2 * c4;
#pragma unroll
      for (int nt = 0; nt < NTQ; ++nt)
        *reinterpret_cast<uint32_t*>(drow + nt * 8) = pack_bf16(dq[nt][2 * rr], dq[nt][2 * rr + 1]);
    }
  }
}

template <int D, int MW>
static size_t mla_bwd_smem() {
  constexpr int HB = 16 * MW;
  return sizeof(__nv_bfloat16) * ((size_t)HB * (D + 8) + HB * (MB_DV + 8) + 2 * MB_KT * (D + 8) +
                                  2 * HB * (MB_KT + 8)) +
         sizeof(int) * 2 * MB_KT;
}

template <int D, int MW>
static cudaError_t launch_bwd_main(const MlaBwdArgs& a, cudaStream_t stream) {
  size_t smem = mla_bwd_smem<D, MW>();
  cudaError_t e = cudaFuncSetAttribute(mla_bwd_mma_kernel<D, MW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.T, (a.H + 16 * MW - 1) / (16 * MW));
  mla_bwd_mma_kernel<D, MW><<<grid, 128 * MW, smem, stream>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_bwd_delta(const __nv_bfloat16* o, const __nv_bfloat16* dout, float* dlt, int64_t rows, int dv,
                             cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  int64_t blocks = (rows + 7) / 8;
  bwd_delta_kernel<<<(unsigned)blocks, 256, 0, stream>>>(o, dout, dlt, rows, dv);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* src, __nv_bfloat16* dst, int64_t n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n / 4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  f32_to_bf16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, dst, n);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_mla_bwd(const MlaBwdArgs& a, int D, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const bool wide = a.H > 16;
  if (D == 576) return wide ? launch_bwd_main<576, 2>(a, stream) : launch_bwd_main<576, 1>(a, stream);
  return wide ? launch_bwd_main<512, 2>(a, stream) : launch_bwd_main<512, 1>(a, stream);
}

}  // namespace tsa
