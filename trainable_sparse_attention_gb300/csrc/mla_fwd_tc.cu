// Sparse MLA forward for H = 128 heads on tcgen05 (TMEM accumulators, TMA
// gather4, 2-CTA cluster).
//
// Megatron-LM PR #3674 "Enable DSA CP/absorbed/THD paths with TileLang fused
// ops" (sparse MLA forward over the absorbed latent) and Megatron-LM PR #7617
// "Support NoPE shapes and unaligned top-k in TileLang sparse MLA" (q
// [T,H,576], value = kv[..., :512], -1 slots, explicit scale, NoPE inputs).
//
// Why a cluster: one query's fp32 output accumulator, 128 heads x 512 value
// channels, is exactly the 512 TMEM columns of an SM, leaving no room for the
// logits.  So a CTA pair shares one query and splits the value channels
// (CTA r owns O[:, 256r, 256r+256)).  Each CTA also owns the matching slice of
// the 576 q/kv channels (CTA 0: [0,256), CTA 1: [256, D)), gathers only that
// slice of the selected rows (TMA tile::gather4, 4 rows per instruction), and
// computes the partial logits Q_r K_r^T over it.  The two 128 x 32 partials
// are swapped through distributed shared memory and added; fp32 addition is
// commutative, so both CTAs hold bit-identical logits and take identical
// softmax decisions.  No MMA is repeated and every selected row is read once.
//
// Per CTA: TMEM columns [0,256) = O slice, [256,320) = two 32-key S buffers.
// Warps 0-3: softmax (thread h = head h = TMEM lane h), warp 4: TMA producer
// (q slice once, then a 4-stage ring of 32-key tiles), warp 5: TMEM owner and
// single-thread MMA issuer (QK^T of tile j+1 is issued before PV of tile j).
// The running max is rescaled lazily (only when it grows by more than 2^8), so
// the O slice in TMEM is rarely touched.  Every wait is bounded; a timeout
// raises TSA_FLAG_TIMEOUT and both CTAs wind down.
#include "kernels.cuh"
#include "tc.cuh"

namespace tsa {

namespace {

constexpr int MT_H = 128;        // heads = MMA M
constexpr int MT_N = 32;         // keys per tile
constexpr int MT_STAGES = 4;
constexpr int MT_THREADS = 192;  // warps 0-3 softmax, 4 producer, 5 MMA
constexpr int MT_DV = 512;
constexpr int MT_OCOLS = 256;    // value channels per CTA
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct MtLayout {
  static constexpr int KB0 = 4;                      // CTA 0: channels [0, 256)
  static constexpr int KB1 = (D - 256) / 64;         // CTA 1: channels [256, D)
  static constexpr int KBMAX = KB1 > KB0 ? KB1 : KB0;
  static constexpr int Q_BYTES = KBMAX * MT_H * 128;
  static constexpr int KV_BLOCK = MT_N * 128;        // one 64-channel column block of a tile
  static constexpr int KV_STAGE = KBMAX * KV_BLOCK;
  static constexpr int P_BYTES = MT_H * 128;
  static constexpr int X_BYTES = MT_H * MT_N * 4;
  static constexpr int OFF_KV = Q_BYTES;
  static constexpr int OFF_P = OFF_KV + MT_STAGES * KV_STAGE;
  static constexpr int OFF_X = OFF_P + P_BYTES;
  static constexpr int OFF_BAR = OFF_X + X_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 512;
};

}  // namespace

template <int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MT_THREADS, 1)
    mla_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                      const __grid_constant__ MlaFwdArgs a) {
  using L = MtLayout<D>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base, sKV = base + L::OFF_KV, sP = base + L::OFF_P;
  float* X = reinterpret_cast<float*>(gbase + L::OFF_X);  // [128][32] partial logits written by the peer
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + L::OFF_BAR);
  uint64_t* qfull = bars;
  uint64_t* kv_full = bars + 1;                       // [STAGES]
  uint64_t* kv_empty = bars + 1 + MT_STAGES;          // [STAGES]
  uint64_t* s_full = bars + 1 + 2 * MT_STAGES;        // [2]
  uint64_t* s_empty = s_full + 2;                     // [2]
  uint64_t* p_full = s_empty + 2;
  uint64_t* p_empty = p_full + 1;
  uint64_t* xfull = p_empty + 1;                      // peer wrote my X
  uint64_t* xfree = xfull + 1;                        // peer consumed what I wrote into its X
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xfree + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t rank = tc::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int t = blockIdx.x >> 1;
  const int sq = seq_of(a.st, t);
  const int s0 = a.st.cu[sq];
  const int n = a.st.cu[sq + 1] - s0;
  const int* idx_row = a.idx + (int64_t)t * a.topk;
  const int ntiles = (a.topk + MT_N - 1) / MT_N;
  const int kb = rank == 0 ? L::KB0 : L::KB1;
  const int ch0 = static_cast<int>(rank) * 256;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float NEG_INF = __int_as_float(0xff800000);

  if (tid == 0) {
    tc::mbar_init(qfull, 1);
    for (int i = 0; i < MT_STAGES; ++i) { tc::mbar_init(&kv_full[i], 1); tc::mbar_init(&kv_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { tc::mbar_init(&s_full[i], 1); tc::mbar_init(&s_empty[i], MT_H); }
    tc::mbar_init(p_full, MT_H);
    tc::mbar_init(p_empty, 1);
    tc::mbar_init(xfull, MT_H);
    tc::mbar_init(xfree, MT_H);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 5) tc::tmem_alloc(tmem_slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  __syncwarp();
  tc::cluster_sync();  // the peer's barriers exist before any remote arrival
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_kv);
      tc::mbar_arrive_expect_tx(qfull, kb * MT_H * 128);
      for (int c = 0; c < kb; ++c) tc::tma_load_2d(sQ + c * (MT_H * 128), &tm_q, qfull, ch0 + c * 64, t * MT_H);
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % MT_STAGES;
        if (!tc::mbar_wait(&kv_empty[st], ((j / MT_STAGES) & 1) ^ 1u, abort_flag)) { *abort_flag = 1; break; }
        int rows[MT_N];
#pragma unroll
        for (int i = 0; i < MT_N; ++i) {
          const int slot = j * MT_N + i;
          const int id = slot < a.topk ? __ldg(idx_row + slot) : -1;
          if (id >= n) raise_flag(a.flags, TSA_FLAG_INDEX_RANGE);
          rows[i] = (id >= 0 && id < n) ? s0 + id : 0;  // invalid slots read a real row and are masked
        }
        tc::mbar_arrive_expect_tx(&kv_full[st], kb * L::KV_BLOCK);
        const uint32_t dst = sKV + st * L::KV_STAGE;
        for (int c = 0; c < kb; ++c) {
#pragma unroll
          for (int g = 0; g < MT_N / 4; ++g)
            tc::tma_gather4(dst + c * L::KV_BLOCK + g * 512, &tm_kv, &kv_full[st], ch0 + c * 64, rows[4 * g],
                            rows[4 * g + 1], rows[4 * g + 2], rows[4 * g + 3]);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(MT_H, MT_N);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32_bmn(MT_H, MT_OCOLS);
      bool ok = tc::mbar_wait(qfull, 0, abort_flag);
      auto issue_qk = [&](int j) -> bool {
        const int st = j % MT_STAGES, b = j & 1;
        if (!tc::mbar_wait(&kv_full[st], (j / MT_STAGES) & 1, abort_flag)) return false;
        if (!tc::mbar_wait(&s_empty[b], ((j >> 1) & 1) ^ 1u, abort_flag)) return false;
        tc::fence_after_sync();
        const uint32_t d = tmem + MT_OCOLS + b * MT_N;
        for (int c = 0; c < kb; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = tc::desc_sw128(sQ + c * (MT_H * 128) + kk * 32);
            const uint64_t bd = tc::desc_sw128(sKV + st * L::KV_STAGE + c * L::KV_BLOCK + kk * 32);
            tc::mma_bf16_ss(d, ad, bd, idesc_qk, (c | kk) != 0 ? 1u : 0u);
          }
        }
        tc::mma_commit(&s_full[b]);
        return true;
      };
      if (ok && ntiles > 0) ok = issue_qk(0);
      for (int j = 0; ok && j < ntiles; ++j) {
        if (j + 1 < ntiles && !issue_qk(j + 1)) { ok = false; break; }
        if (!tc::mbar_wait(p_full, j & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        const int st = j % MT_STAGES;
#pragma unroll
        for (int ks = 0; ks < MT_N / 16; ++ks) {
          const uint64_t ad = tc::desc_sw128(sP + ks * 32);
          const uint64_t bd = tc::desc_sw128_mn(sKV + st * L::KV_STAGE + ks * 2048, L::KV_BLOCK);
          tc::mma_bf16_ss(tmem, ad, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc::mma_commit(&kv_empty[st]);
        tc::mma_commit(p_empty);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int h = tid;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t x_peer_row = tc::mapa(smem_u32(X + h * MT_N), peer);
    const uint32_t peer_xfull = tc::mapa(smem_u32(xfull), peer);
    const uint32_t peer_xfree = tc::mapa(smem_u32(xfree), peer);
    float m_use = NEG_INF, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&s_full[b], (j >> 1) & 1, abort_flag))) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t r[32];
      __syncwarp();
      tc::tmem_ld32(tmem + lane_base + MT_OCOLS + b * MT_N, r);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      tc::mbar_arrive(&s_empty[b]);
      // swap partial logits with the peer CTA
      if (!__all_sync(0xffffffffu, tc::mbar_wait_cluster(xfree, (j & 1) ^ 1u, abort_flag))) { ok = false; break; }
#pragma unroll
      for (int q = 0; q < 8; ++q)
        tc::st_cluster_v4(x_peer_row + q * 16, __uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                          __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
      tc::mbar_arrive_remote(peer_xfull);
      if (!__all_sync(0xffffffffu, tc::mbar_wait_cluster(xfull, j & 1, abort_flag))) { ok = false; break; }
      float x2[32];
      const float4* xr = reinterpret_cast<const float4*>(X + h * MT_N);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 v = xr[q];
        x2[4 * q] = __uint_as_float(r[4 * q]) + v.x;
        x2[4 * q + 1] = __uint_as_float(r[4 * q + 1]) + v.y;
        x2[4 * q + 2] = __uint_as_float(r[4 * q + 2]) + v.z;
        x2[4 * q + 3] = __uint_as_float(r[4 * q + 3]) + v.w;
      }
      tc::mbar_arrive_remote(peer_xfree);
      // mask, scale, lazy running max
      float tmax = NEG_INF;
#pragma unroll
      for (int i = 0; i < MT_N; ++i) {
        const int slot = j * MT_N + i;
        const int id = slot < a.topk ? __ldg(idx_row + slot) : -1;
        x2[i] = (id >= 0 && id < n) ? x2[i] * a.scale_log2 : NEG_INF;
        tmax = fmaxf(tmax, x2[i]);
      }
      float alpha = 1.f;
      const bool resc = tmax > m_use + kRescaleLog2;
      if (resc) {
        alpha = (m_use == NEG_INF) ? 0.f : exp2f(m_use - tmax);
        m_use = tmax;
        l *= alpha;
      }
      const float mu = (m_use == NEG_INF) ? 0.f : m_use;
      uint32_t pk[MT_N / 2];
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < MT_N; i += 2) {
        const float p0 = exp2f(x2[i] - mu), p1 = exp2f(x2[i + 1] - mu);
        psum += p0 + p1;
        pk[i / 2] = pack_bf16(p0, p1);
      }
      l += psum;
      // P and the O slice are free once PV of the previous tile has completed
      if (j > 0) {
        if (!__all_sync(0xffffffffu, tc::mbar_wait(p_empty, (j - 1) & 1, abort_flag))) { ok = false; break; }
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, resc)) {
          for (int cb = 0; cb < MT_OCOLS / 32; ++cb) {
            uint32_t o[32];
            tc::tmem_ld32(tmem + lane_base + cb * 32, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tc::tmem_st32(tmem + lane_base + cb * 32, o);
          }
          tc::tmem_st_wait();
        }
      }
      // P row h: 32 bf16 = 4 x 16 B chunks in a 128-byte-swizzled K-major row
      unsigned char* prow = gbase + L::OFF_P + h * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (h & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(p_full);
    }
    if (!ok) *abort_flag = 1;
    // epilogue: O slice / l -> bf16, lse
    const bool last_ok = ok && __all_sync(0xffffffffu, tc::mbar_wait(p_empty, (ntiles - 1) & 1, abort_flag));
    if (last_ok) {
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = a.out + ((int64_t)t * MT_H + h) * MT_DV + ch0;
      for (int cb = 0; cb < MT_OCOLS / 32; ++cb) {
        uint32_t o[32];
        __syncwarp();
        tc::tmem_ld32(tmem + lane_base + cb * 32, o);
        tc::tmem_ld_wait();
        uint4* dst = reinterpret_cast<uint4*>(orow + cb * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(pack_bf16(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                              pack_bf16(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                              pack_bf16(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                              pack_bf16(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
      }
      if (rank == 0) a.lse[(int64_t)t * MT_H + h] = l > 0.f ? (m_use + log2f(l)) * kLn2 : NEG_INF;
    } else {
      // nothing selected (or wound down): zero output slice, -inf lse
      __nv_bfloat16* orow = a.out + ((int64_t)t * MT_H + h) * MT_DV + ch0;
      for (int c = 0; c < MT_OCOLS; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
      if (rank == 0) a.lse[(int64_t)t * MT_H + h] = NEG_INF;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && tid == 0) raise_flag(a.flags, TSA_FLAG_TIMEOUT);
  __syncwarp();
  tc::cluster_sync();  // the peer no longer writes into this CTA's shared memory
  if (warp == 5) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

cudaError_t make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                              uint32_t box_cols);

template <int D>
static cudaError_t launch_tc_t(const MlaFwdArgs& a, cudaStream_t stream) {
  CUtensorMap tq, tkv;
  cudaError_t e = make_tmap_bf16_2d(&tq, a.q, (uint64_t)a.T * MT_H, D, MT_H, 64);
  if (e != cudaSuccess) return e;
  e = make_tmap_bf16_2d(&tkv, a.kv, (uint64_t)a.T, D, 1, 64);
  if (e != cudaSuccess) return e;
  constexpr int smem = MtLayout<D>::SMEM;
  e = cudaFuncSetAttribute(mla_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mla_fwd_tc_kernel<D><<<dim3(2 * a.T), MT_THREADS, smem, stream>>>(tq, tkv, a);
  return cudaGetLastError();
}

cudaError_t launch_mla_fwd_tc(const MlaFwdArgs& a, int D, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  return D == 576 ? launch_tc_t<576>(a, stream) : launch_tc_t<512>(a, stream);
}

}  // namespace tsa
