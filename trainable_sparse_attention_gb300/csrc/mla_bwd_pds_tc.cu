// Sparse MLA backward for 128 heads on tcgen05: the recompute of P and dS, and dQ.
//
// Megatron-LM PR #3674 "Enable DSA CP/absorbed/THD paths with TileLang fused
// ops" (sparse MLA backward) and Megatron-LM PR #7617 "Support NoPE shapes and
// unaligned top-k in TileLang sparse MLA" (value = kv[..., :512], -1 slots,
// explicit softmax scale, NoPE inputs).
//
// With the forward's log-sum-exp L and Dlt = rowsum(dO * O) per (t, h):
//   S = q K^T, P = exp(scale S - L), dP = dO V^T, dS = scale P (dP - Dlt),
//   dQ = dS K.
//
// mla_bwd_pds_tc_kernel: one CTA per query.  The query's q rows (128 heads x
// D) live in TMEM and are the A operand of S = q K^T, so shared memory holds
// only dO (the A operand of dP = dO V^T, loaded once by TMA) and a two-stage
// ring of gathered 32-key tiles of kv.  S and dP of a tile land in TMEM
// (double-buffered); warps 0-3 (thread = head = TMEM lane) turn them into P
// and dS and write both in bf16 to the staging area, [query][head][slot],
// slots padded to kp with zeros.  No softmax state is carried between tiles:
// L is known, so every tile is final when it is computed.
//
// mla_bwd_dq_tc_kernel: dQ = dS K over the gathered rows.  The 128 x D fp32
// accumulator does not fit one SM's 512 TMEM columns for D = 576, so two CTAs
// share a query, split by channel (CTA 0: [0, 256), CTA 1: [256, D)); each
// gathers only its slice of the selected rows as the MN-major B operand and
// streams the dS tiles (A, K-major) by TMA.
#include "kernels.cuh"
#include "tc.cuh"

namespace tsa {

cudaError_t make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                              uint32_t box_cols);

namespace {

constexpr int PB_H = 128;        // heads = MMA M
constexpr int PB_N = 32;         // keys per tile
constexpr int PB_STAGES = 2;
constexpr int PB_THREADS = 288;  // warps 0-3 P/dS, warp 4 MMA + TMA, warps 5-8 gather producers
constexpr int PB_QC = 288;       // TMEM columns reserved for q (D / 2 packed bf16 pairs)

template <int D>
struct PbLayout {
  static constexpr int KB = D / 64;                  // 64-channel blocks of a kv row
  static constexpr int DO_BYTES = 8 * PB_H * 128;    // dO, 8 boxes of 64 channels x 128 rows
  static constexpr int KV_BLOCK = PB_N * 128;        // one 64-channel block of a 32-key tile
  static constexpr int KV_STAGE = KB * KV_BLOCK;
  static constexpr int OFF_KV = DO_BYTES;
  static constexpr int OFF_BAR = OFF_KV + PB_STAGES * KV_STAGE;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
};

constexpr int DQ_N = 64;          // slots per tile (MMA K per tile)
constexpr int DQ_STAGES = 3;
constexpr int DQ_THREADS = 288;   // warps 0-3 and 5-8 gather (thread 0 also loads the dS tiles, 0-3 drain dQ), warp 4 MMA
constexpr int DQ_A = PB_H * 128;  // dS tile: 128 rows x 64 slots bf16 = 16 KB
constexpr int DQ_BBLK = DQ_N * 128;  // 64 channels x 64 slots = 8 KB
constexpr int DQ_B = 5 * DQ_BBLK;    // up to 320 channels
constexpr int DQ_STAGE = DQ_A + DQ_B;
constexpr int DQ_OFF_BAR = DQ_STAGES * DQ_STAGE;
constexpr int DQ_SMEM = 1024 + DQ_OFF_BAR + 256;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(PB_THREADS, 1)
    mla_bwd_pds_tc_kernel(const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ MlaBwdArgs a) {
  using L = PbLayout<D>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t sDO = base, sKV = base + L::OFF_KV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + L::OFF_BAR);
  uint64_t* dofull = bars;                      // [1] dO landed (TMA)
  uint64_t* qready = bars + 1;                  // [1] q stored into TMEM (4 warps)
  uint64_t* kv_full = bars + 2;                 // [STAGES] 128 asynchronous producer arrivals
  uint64_t* kv_empty = kv_full + PB_STAGES;     // [STAGES]
  uint64_t* sd_full = kv_empty + PB_STAGES;     // [2] S and dP of a tile in TMEM
  uint64_t* sd_empty = sd_full + 2;             // [2] (4 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sd_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int lq = blockIdx.x;
  const int t = a.q0 + lq;
  const int sq = seq_of(a.st, t);
  const int s0 = a.st.cu[sq];
  const int n = a.st.cu[sq + 1] - s0;
  const int* idx_row = a.idx + (int64_t)t * a.topk;
  const int ntiles = (a.topk + PB_N - 1) / PB_N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tc::mbar_init(dofull, 1);
    tc::mbar_init(qready, 4);
    for (int i = 0; i < PB_STAGES; ++i) {
      tc::mbar_init(&kv_full[i], 128);
      tc::mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sd_full[i], 1);
      tc::mbar_init(&sd_empty[i], 4);
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 4) tc::tmem_alloc(tmem_slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 5) {
    // ------------------------------------------------------------ gather producers (128 threads)
    // 32 rows x 4 parts; each thread copies KB*2 16-byte chunks of one selected
    // row into the 128-byte-swizzled K-major tile, arriving asynchronously on
    // the stage's barrier when they land.
    const int pt = tid - 160;
    const int row = pt >> 2, part = pt & 3;
    constexpr int per = L::KB * 2;
    const char* kvb = reinterpret_cast<const char*>(a.kv);
    bool ok = true;
    int id_next = row < a.topk ? __ldg(idx_row + row) : -1;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % PB_STAGES;
      const int id = id_next;
      const int slot_next = (j + 1) * PB_N + row;
      id_next = slot_next < a.topk ? __ldg(idx_row + slot_next) : -1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&kv_empty[st], ((j / PB_STAGES) & 1) ^ 1u, abort_flag))) {
        ok = false;
        break;
      }
      const bool valid = id >= 0 && id < n;
      if (part == 0 && id >= n) raise_flag(a.flags, TSA_FLAG_INDEX_RANGE);
      const char* src_row = kvb + (int64_t)(valid ? s0 + id : 0) * D * 2;
      const uint32_t dst = sKV + st * L::KV_STAGE + row * 128;
#pragma unroll
      for (int q = 0; q < per; ++q) {
        const int c16 = part * per + q;
        const int cb = c16 >> 3, jj = c16 & 7;
        cp_async16(dst + cb * L::KV_BLOCK + ((jj ^ (row & 7)) << 4), src_row + c16 * 16, valid ? 16u : 0u);
      }
      cp_async_commit();
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&kv_full[st]))
                   : "memory");
    }
    cp_async_wait<0>();
    if (!ok) *abort_flag = 1;
  } else if (warp == 4) {
    // ------------------------------------------------------------ dO (TMA) + MMA issuer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_do);
      tc::mbar_arrive_expect_tx(dofull, L::DO_BYTES);
      for (int c = 0; c < 8; ++c) tc::tma_load_2d(sDO + c * (PB_H * 128), &tm_do, dofull, c * 64, t * PB_H);
      constexpr uint32_t idesc = tc::idesc_bf16_f32(PB_H, PB_N);
      bool ok = tc::mbar_wait(dofull, 0, abort_flag) && tc::mbar_wait(qready, 0, abort_flag);
      tc::fence_after_sync();
      for (int j = 0; ok && j < ntiles; ++j) {
        const int st = j % PB_STAGES, b = j & 1;
        if (!tc::mbar_wait(&kv_full[st], (j / PB_STAGES) & 1, abort_flag) ||
            !tc::mbar_wait(&sd_empty[b], ((j >> 1) & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_proxy_async_smem();  // the gathered tile was written through the generic proxy
        tc::fence_after_sync();
        const uint32_t dS_ = tmem + PB_QC + b * PB_N;
        const uint32_t dP_ = tmem + PB_QC + 2 * PB_N + b * PB_N;
        const uint32_t kv = sKV + st * L::KV_STAGE;
        // S = q K^T: A = q from TMEM (8 columns per 16 channels)
        for (int c = 0; c < L::KB; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_ts(dS_, tmem + (c * 4 + kk) * 8, tc::desc_sw128(kv + c * L::KV_BLOCK + kk * 32), idesc,
                            (c | kk) != 0 ? 1u : 0u);
        }
        // dP = dO V^T over the 512 value channels
        for (int c = 0; c < 8; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_ss(dP_, tc::desc_sw128(sDO + c * (PB_H * 128) + kk * 32),
                            tc::desc_sw128(kv + c * L::KV_BLOCK + kk * 32), idesc, (c | kk) != 0 ? 1u : 0u);
        }
        tc::mma_commit(&kv_empty[st]);
        tc::mma_commit(&sd_full[b]);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ P / dS (warps 0-3, thread = head)
    const int h = tid;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float NEG_INF = __int_as_float(0xff800000);
    const float Lh = a.lse[(int64_t)t * PB_H + h];
    const float lse2 = Lh * kLog2e;
    const bool live = Lh != NEG_INF;  // a row without valid slots has P = dS = 0
    const float dl = a.dlt[(int64_t)t * PB_H + h];
    // q row h -> TMEM columns [0, D/2): 32 columns (64 channels) per store
    {
      const uint4* qrow = reinterpret_cast<const uint4*>(a.q + ((int64_t)t * PB_H + h) * D);
      for (int c = 0; c < D / 64; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = __ldg(qrow + c * 8 + i);
          r[4 * i] = v.x;
          r[4 * i + 1] = v.y;
          r[4 * i + 2] = v.z;
          r[4 * i + 3] = v.w;
        }
        __syncwarp();
        tc::tmem_st32(tmem + lane_base + c * 32, r);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(qready);
    }
    __nv_bfloat16* prow = a.p_out + ((int64_t)lq * PB_H + h) * a.kp;
    __nv_bfloat16* dsrow = a.ds_out + ((int64_t)lq * PB_H + h) * a.kp;
    bool ok = true;
    int idn = lane < a.topk ? __ldg(idx_row + lane) : -1;
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1;
      const uint32_t mask = __ballot_sync(0xffffffffu, idn >= 0 && idn < n);
      const int slot_next = (j + 1) * PB_N + lane;
      idn = slot_next < a.topk ? __ldg(idx_row + slot_next) : -1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&sd_full[b], (j >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      uint32_t s[32], dp[32];
      tc::tmem_ld32(tmem + lane_base + PB_QC + b * PB_N, s);
      tc::tmem_ld32(tmem + lane_base + PB_QC + 2 * PB_N + b * PB_N, dp);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sd_empty[b]);
      uint32_t pk[16], dk[16];
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float p0 = 0.f, p1 = 0.f;
        if (live && ((mask >> i) & 1u)) p0 = ex2(fmaf(__uint_as_float(s[i]), a.scale_log2, -lse2));
        if (live && ((mask >> (i + 1)) & 1u)) p1 = ex2(fmaf(__uint_as_float(s[i + 1]), a.scale_log2, -lse2));
        const float d0 = a.scale * p0 * (__uint_as_float(dp[i]) - dl);
        const float d1 = a.scale * p1 * (__uint_as_float(dp[i + 1]) - dl);
        pk[i / 2] = pack_bf16(p0, p1);
        dk[i / 2] = pack_bf16(d0, d1);
      }
      uint4* pd = reinterpret_cast<uint4*>(prow + j * PB_N);
      uint4* dd = reinterpret_cast<uint4*>(dsrow + j * PB_N);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        pd[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        dd[c] = make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
      }
    }
    if (!ok) *abort_flag = 1;
    // zero the padding slots [ntiles * 32, kp)
    for (int c = ntiles * PB_N; c < a.kp; c += 8) {
      *reinterpret_cast<uint4*>(prow + c) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(dsrow + c) = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && tid == 0) raise_flag(a.flags, TSA_FLAG_TIMEOUT);
  if (warp == 4) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// grid.x = 2 * nq: query q0 + blockIdx.x / 2, channel half blockIdx.x % 2.
template <int D>
__global__ void __launch_bounds__(DQ_THREADS, 1)
    mla_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_ds, const __grid_constant__ MlaBwdArgs a) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + DQ_OFF_BAR);
  uint64_t* afull = bars;                     // [STAGES] dS tile (TMA)
  uint64_t* bfull = afull + DQ_STAGES;        // [STAGES] 256 asynchronous gather arrivals
  uint64_t* sempty = bfull + DQ_STAGES;       // [STAGES]
  uint64_t* dfull = sempty + DQ_STAGES;       // [1] all MMAs done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int lq = blockIdx.x >> 1;
  const int t = a.q0 + lq;
  const int half = blockIdx.x & 1;
  const int ch0 = half * 256;
  const int nch = half == 0 ? 256 : D - 256;  // 256, or 320 for D = 576
  const int nblk = nch / 64;
  const int sq = seq_of(a.st, t);
  const int s0 = a.st.cu[sq];
  const int n = a.st.cu[sq + 1] - s0;
  const int* idx_row = a.idx + (int64_t)t * a.topk;
  const int ntiles = a.kp / DQ_N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < DQ_STAGES; ++i) {
      tc::mbar_init(&afull[i], 1);
      tc::mbar_init(&bfull[i], 256);
      tc::mbar_init(&sempty[i], 1);
    }
    tc::mbar_init(dfull, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 4) tc::tmem_alloc(tmem_slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    if (lane == 0) {
      const uint32_t idesc0 = tc::idesc_bf16_f32_bmn(PB_H, 256);
      const uint32_t idesc1 = tc::idesc_bf16_f32_bmn(PB_H, 64);
      bool ok = true;
      for (int j = 0; ok && j < ntiles; ++j) {
        const int st = j % DQ_STAGES;
        if (!tc::mbar_wait(&afull[st], (j / DQ_STAGES) & 1, abort_flag) ||
            !tc::mbar_wait(&bfull[st], (j / DQ_STAGES) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_proxy_async_smem();  // the gathered rows were written through the generic proxy
        tc::fence_after_sync();
        const uint32_t sa = base + st * DQ_STAGE, sb = sa + DQ_A;
#pragma unroll
        for (int ks = 0; ks < DQ_N / 16; ++ks) {
          const uint64_t ad = tc::desc_sw128(sa + ks * 32);
          const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
          tc::mma_bf16_ss(tmem, ad, tc::desc_sw128_mn(sb + ks * 2048, DQ_BBLK), idesc0, acc);
          if (nblk == 5)
            tc::mma_bf16_ss(tmem + 256, ad, tc::desc_sw128_mn(sb + 4 * DQ_BBLK + ks * 2048, DQ_BBLK), idesc1, acc);
        }
        tc::mma_commit(&sempty[st]);
      }
      tc::mma_commit(dfull);
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ gather (256 threads): 64 rows x 4 parts
    const int pt = warp < 4 ? tid : tid - 32;
    const int row = pt >> 2, part = pt & 3;
    if (pt == 0) tc::prefetch_tmap(&tm_ds);
    const int per = nblk * 2;  // 16-byte chunks per part (8 or 10)
    const char* kvb = reinterpret_cast<const char*>(a.kv);
    bool ok = true;
    int id_next = row < a.topk ? __ldg(idx_row + row) : -1;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % DQ_STAGES;
      const int id = id_next;
      const int slot_next = (j + 1) * DQ_N + row;
      id_next = slot_next < a.topk ? __ldg(idx_row + slot_next) : -1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&sempty[st], ((j / DQ_STAGES) & 1) ^ 1u, abort_flag))) {
        ok = false;
        break;
      }
      if (pt == 0) {
        // the dS tile of this stage (A operand) by TMA
        tc::mbar_arrive_expect_tx(&afull[st], DQ_A);
        tc::tma_load_2d(base + st * DQ_STAGE, &tm_ds, &afull[st], j * DQ_N, lq * PB_H);
      }
      const bool valid = id >= 0 && id < n;
      const char* src_row = kvb + ((int64_t)(valid ? s0 + id : 0) * D + ch0) * 2;
      const uint32_t dst = base + st * DQ_STAGE + DQ_A + row * 128;
      for (int q = 0; q < per; ++q) {
        const int c16 = part * per + q;
        const int cb = c16 >> 3, jj = c16 & 7;
        cp_async16(dst + cb * DQ_BBLK + ((jj ^ (row & 7)) << 4), src_row + c16 * 16, valid ? 16u : 0u);
      }
      cp_async_commit();
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&bfull[st]))
                   : "memory");
    }
    cp_async_wait<0>();
    if (!ok) *abort_flag = 1;
    if (warp < 4) {
      // ---------------------------------------------------------- drain dQ (thread = head)
      const int h = tid;
      __nv_bfloat16* drow = a.dq + ((int64_t)t * PB_H + h) * D + ch0;
      const bool done = __all_sync(0xffffffffu, tc::mbar_wait(dfull, 0, abort_flag));
      if (done) {
        tc::fence_after_sync();
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        for (int cb = 0; cb < nch / 32; ++cb) {
          uint32_t o[32];
          __syncwarp();
          tc::tmem_ld32(tmem + lane_base + cb * 32, o);
          tc::tmem_ld_wait();
          uint4* dst = reinterpret_cast<uint4*>(drow + cb * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pack_bf16(__uint_as_float(o[8 * q]), __uint_as_float(o[8 * q + 1])),
                                pack_bf16(__uint_as_float(o[8 * q + 2]), __uint_as_float(o[8 * q + 3])),
                                pack_bf16(__uint_as_float(o[8 * q + 4]), __uint_as_float(o[8 * q + 5])),
                                pack_bf16(__uint_as_float(o[8 * q + 6]), __uint_as_float(o[8 * q + 7])));
        }
      } else {
        *abort_flag = 1;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && tid == 0) raise_flag(a.flags, TSA_FLAG_TIMEOUT);
  if (warp == 4) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int D>
static cudaError_t launch_pds_t(const MlaBwdArgs& a, int nq, cudaStream_t stream) {
  CUtensorMap tdo;
  cudaError_t e = make_tmap_bf16_2d(&tdo, a.dout, (uint64_t)a.T * PB_H, 512, PB_H, 64);
  if (e != cudaSuccess) return e;
  constexpr int smem = PbLayout<D>::SMEM;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  if ((e = cudaFuncSetAttribute(mla_bwd_pds_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
      cudaSuccess)
    return e;
  mla_bwd_pds_tc_kernel<D><<<dim3(nq), PB_THREADS, smem, stream>>>(tdo, a);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_dq_t(const MlaBwdArgs& a, int nq, cudaStream_t stream) {
  CUtensorMap tds;
  cudaError_t e = make_tmap_bf16_2d(&tds, a.ds_out, (uint64_t)nq * PB_H, a.kp, PB_H, 64);
  if (e != cudaSuccess) return e;
  static_assert(DQ_SMEM <= 227 * 1024, "shared memory budget");
  if ((e = cudaFuncSetAttribute(mla_bwd_dq_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM)) !=
      cudaSuccess)
    return e;
  mla_bwd_dq_tc_kernel<D><<<dim3(2 * nq), DQ_THREADS, DQ_SMEM, stream>>>(tds, a);
  return cudaGetLastError();
}

cudaError_t launch_mla_bwd_pds_tc(const MlaBwdArgs& a, int D, int nq, cudaStream_t stream) {
  if (nq <= 0) return cudaSuccess;
  if (a.H != PB_H || a.kp % 128 != 0 || a.p_out == nullptr || a.ds_out == nullptr) return cudaErrorInvalidValue;
  return D == 576 ? launch_pds_t<576>(a, nq, stream) : launch_pds_t<512>(a, nq, stream);
}

cudaError_t launch_mla_bwd_dq_tc(const MlaBwdArgs& a, int D, int nq, cudaStream_t stream) {
  if (nq <= 0) return cudaSuccess;
  if (a.H != PB_H || a.kp % 128 != 0 || a.ds_out == nullptr) return cudaErrorInvalidValue;
  return D == 576 ? launch_dq_t<576>(a, nq, stream) : launch_dq_t<512>(a, nq, stream);
}

}  // namespace tsa
