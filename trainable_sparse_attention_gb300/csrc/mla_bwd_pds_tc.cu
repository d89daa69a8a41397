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
// mla_bwd_sp_tc_kernel, two passes with one CTA per query.  A tcgen05 MMA
// costs the same for N = 32 and N = 64 (about 45 cycles for M = 128), so the
// selected rows are taken 64 at a time; q (576 channels) and dO (512) do not
// both fit the 512 TMEM columns next to two 64-column accumulators, and dO in
// shared memory would leave no room for a deep gather ring.  Hence:
//   pass 1: S = q K^T with the q rows in TMEM (A operand), P = exp(scale S - L)
//           written in bf16;
//   pass 2: dP = dO V^T with the dO rows in TMEM, dS = scale P (dP - Dlt)
//           from the bf16 P of pass 1, written in bf16.
// Each pass streams its gathered 64-row tiles through a three-stage ring
// (cp.async, 8 producer warps) and double-buffers the accumulator in TMEM;
// warps 0-7 (two per TMEM lane quadrant, thread = head, 32 of the 64 key
// columns each) write [query][head][slot] rows, slots padded to kp with
// zeros.  No softmax state is carried between tiles: L is known, so every
// tile is final when it is computed.
//
// mla_bwd_dq_tc_kernel: dQ = dS K over the gathered rows.  The 128 x D fp32
// accumulator does not fit one SM's 512 TMEM columns for D = 576, so two CTAs
// share a query, split by channel (CTA 0: [0, 256), CTA 1: [256, D)); each
// gathers only its slice of the selected rows as the MN-major B operand and
// streams the dS tiles (A, K-major) by TMA.
//
// The recompute passes copy a selected row with consecutive lanes on
// consecutive 16-byte chunks, so the cp.async of a warp coalesce into whole
// lines; the dQ kernel fetches its rows with TMA gathers of 4 rows x 64
// channels (tile::gather4).  Each kernel uses the copy path that measured
// faster for it: TMA gathers in the recompute passes, or split half and half
// with cp.async, made the backward 1-2 % slower, while in the dQ kernel they
// took a quarter off its time.
#include "kernels.cuh"
#include "tc.cuh"

namespace tsa {

cudaError_t make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                              uint32_t box_cols);

namespace {

constexpr int PB_H = 128;        // heads = MMA M
constexpr int SP_H = PB_H;
constexpr int SP_N = 64;         // keys per tile (MMA N)
constexpr int SP_STAGES = 3;
constexpr int SP_PRODUCERS = 256;
constexpr int SP_THREADS = 288 + SP_PRODUCERS;  // warps 0-7 epilogue, warp 8 MMA, warps 9-16 gather
constexpr int SP_ACC = 288;      // first TMEM column of the two accumulators (after the A operand)

constexpr int SP_PTILE = SP_H * 128;  // one P tile of the dS pass: 128 heads x 64 slots bf16

template <int D, bool DS>
constexpr int sp_smem() {
  return 1024 + SP_STAGES * ((DS ? 512 : D) / 64) * (SP_N * 128) + (DS ? 2 * SP_PTILE : 0) + 256;
}

constexpr int DQ_N = 64;          // slots per tile (MMA K per tile)
constexpr int DQ_STAGES = 4;
constexpr int DQ_THREADS = 544;   // warps 0-3 and 5-16 gather (thread 0 also loads the dS tiles, 0-3 drain dQ), warp 4 MMA
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

// One launch of either pass over queries q0 .. q0+gridDim.x (one CTA each).
// DS = false: S = q K^T (A = q rows in TMEM, KC = D channels), writes P.
// DS = true:  dP = dO V^T (A = dO rows in TMEM, KC = 512 value channels),
//             reads P, writes dS = scale P (dP - Dlt).
template <int D, bool DS>
__global__ void __launch_bounds__(SP_THREADS, 1)
    mla_bwd_sp_tc_kernel(const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ MlaBwdArgs a) {
  constexpr int KC = DS ? 512 : D;   // channels of the contraction
  constexpr int KB = KC / 64;        // 64-channel blocks of a gathered row
  constexpr int ACOLS = KC / 2;      // TMEM columns of the A operand (bf16 pairs)
  constexpr int KV_BLOCK = SP_N * 128;
  constexpr int KV_STAGE = KB * KV_BLOCK;
  constexpr int OFF_P = SP_STAGES * KV_STAGE;            // dS pass: two P tiles (TMA, 128-byte swizzle)
  constexpr int OFF_BAR = OFF_P + (DS ? 2 * SP_PTILE : 0);
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + OFF_BAR);
  uint64_t* aready = bars;                      // [1] A rows stored into TMEM (12 warps)
  uint64_t* kv_full = bars + 1;                 // [STAGES] asynchronous producer arrivals
  uint64_t* kv_empty = kv_full + SP_STAGES;     // [STAGES]
  uint64_t* acc_full = kv_empty + SP_STAGES;    // [2] a tile's S (or dP) in TMEM
  uint64_t* acc_empty = acc_full + 2;           // [2] (4 warps)
  uint64_t* pfull = acc_empty + 2;              // [2] dS pass: P tile landed (TMA)
  uint64_t* pempty = pfull + 2;                 // [2] dS pass: P tile read (4 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int lq = blockIdx.x;
  const int t = a.q0 + lq;
  const int sq = seq_of(a.st, t);
  const int s0 = a.st.cu[sq];
  const int n = a.st.cu[sq + 1] - s0;
  const int* idx_row = a.idx + (int64_t)t * a.topk;
  const int ntiles = (a.topk + SP_N - 1) / SP_N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int p_issued = 0;  // dS pass: P tiles whose TMA loads thread 0 issued

  if (tid == 0) {
    tc::mbar_init(aready, 16);
    for (int i = 0; i < SP_STAGES; ++i) {
      tc::mbar_init(&kv_full[i], SP_PRODUCERS);
      tc::mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_empty[i], 8);
      tc::mbar_init(&pfull[i], 1);
      tc::mbar_init(&pempty[i], 8);
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 8) tc::tmem_alloc(tmem_slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // A rows -> TMEM columns [0, KC/2), 32 columns (64 channels) per store.  The
  // four warps that share a TMEM lane quadrant (epilogue warps q and q+4, the
  // two producer warps of that quadrant) split the KB blocks of their 32 rows.
  auto load_a_rows = [&](int share) {
    const int h = (warp & 3) * 32 + lane;
    const uint4* arow = DS ? reinterpret_cast<const uint4*>(a.dout + ((int64_t)t * SP_H + h) * 512)
                           : reinterpret_cast<const uint4*>(a.q + ((int64_t)t * SP_H + h) * D);
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    for (int c = share; c < KB; c += 4) {
      uint32_t r[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = __ldg(arow + c * 8 + i);
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
    if (lane == 0) tc::mbar_arrive(aready);
  };

  if (warp >= 9) {
    // ------------------------------------------------------------ gather producers (8 warps)
    // Warp w copies rows 8w .. 8w+7 of each 64-row tile; lane l copies the
    // 16-byte chunks l, l+32, ... of a row, so one instruction covers 512
    // contiguous bytes of the row.  The chunks land in the 128-byte-swizzled
    // K-major tile, and each thread's copies arrive asynchronously on the
    // stage's barrier when they land.  The slot indices of the next tile are
    // loaded one tile ahead (lane r < 8 holds row 8w + r).
    const int w8 = (warp - 9) * 8;
    constexpr int NCH = KC / 8;  // 16-byte chunks per row
    const char* kvb = reinterpret_cast<const char*>(a.kv);
    bool ok = true;
    const int npre = ntiles < SP_STAGES ? ntiles : SP_STAGES;
    int id_next = (lane < 8 && w8 + lane < a.topk) ? __ldg(idx_row + w8 + lane) : -1;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % SP_STAGES;
      const int id_mine = id_next;
      const int slot_next = (j + 1) * SP_N + w8 + lane;
      id_next = (lane < 8 && slot_next < a.topk) ? __ldg(idx_row + slot_next) : -1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&kv_empty[st], ((j / SP_STAGES) & 1) ^ 1u, abort_flag))) {
        ok = false;
        break;
      }
      if (!DS && lane < 8 && id_mine >= n) raise_flag(a.flags, TSA_FLAG_INDEX_RANGE);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int id = __shfl_sync(0xffffffffu, id_mine, r);
        const int row = w8 + r;
        const bool valid = id >= 0 && id < n;
        const char* src_row = kvb + (int64_t)(valid ? s0 + id : 0) * D * 2;
        const uint32_t dst = base + st * KV_STAGE + row * 128;
#pragma unroll
        for (int c16 = lane; c16 < NCH; c16 += 32) {
          const int cb = c16 >> 3, jj = c16 & 7;
          cp_async16(dst + cb * KV_BLOCK + ((jj ^ (row & 7)) << 4), src_row + c16 * 16, valid ? 16u : 0u);
        }
      }
      cp_async_commit();
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&kv_full[st]))
                   : "memory");
      // the first tiles are in flight: help load the A rows
      if (j == npre - 1) load_a_rows(warp < 13 ? 2 : 3);
    }
    cp_async_wait<0>();
    if (!ok) *abort_flag = 1;
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(SP_H, SP_N);
      bool ok = tc::mbar_wait(aready, 0, abort_flag);
      tc::fence_after_sync();
      for (int j = 0; ok && j < ntiles; ++j) {
        const int st = j % SP_STAGES, b = j & 1;
        if (!tc::mbar_wait(&kv_full[st], (j / SP_STAGES) & 1, abort_flag) ||
            !tc::mbar_wait(&acc_empty[b], ((j >> 1) & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_proxy_async_smem();  // the gathered tile was written through the generic proxy
        tc::fence_after_sync();
        const uint32_t d = tmem + SP_ACC + b * SP_N;
        const uint32_t kv = base + st * KV_STAGE;
        for (int c = 0; c < KB; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_ts(d, tmem + (c * 4 + kk) * 8, tc::desc_sw128(kv + c * KV_BLOCK + kk * 32), idesc,
                            (c | kk) != 0 ? 1u : 0u);
        }
        tc::mma_commit(&kv_empty[st]);
        tc::mma_commit(&acc_full[b]);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-7)
    // Thread (h, hf): head h = 32 (warp % 4) + lane (its TMEM lane), key
    // columns 32 hf .. +31 of each 64-key tile, hf = warp / 4.
    const int qd = warp & 3, hf = warp >> 2;
    const int h = qd * 32 + lane;
    const int cofs = hf * 32;
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const float NEG_INF = __int_as_float(0xff800000);
    const float Lh = a.lse[(int64_t)t * SP_H + h];
    const float lse2 = Lh * kLog2e;
    const bool live = Lh != NEG_INF;  // a row without valid slots has P = dS = 0
    const float dl = DS ? a.dlt[(int64_t)t * SP_H + h] : 0.f;
    load_a_rows(hf);
    static_assert(ACOLS <= SP_ACC, "A operand overlaps the accumulators");
    __nv_bfloat16* prow = a.p_out + ((int64_t)lq * SP_H + h) * a.kp;
    __nv_bfloat16* dsrow = a.ds_out + ((int64_t)lq * SP_H + h) * a.kp;
    bool ok = true;
    int idn = cofs + lane < a.topk ? __ldg(idx_row + cofs + lane) : -1;
    if (DS && tid == 0) {
      // P tiles 0 and 1 (TMA); later tiles are issued as the ring frees up
      tc::prefetch_tmap(&tm_p);
      for (int jj = 0; jj < 2 && jj < ntiles; ++jj) {
        tc::mbar_arrive_expect_tx(&pfull[jj], SP_PTILE);
        tc::tma_load_2d_hint(base + OFF_P + jj * SP_PTILE, &tm_p, &pfull[jj], jj * SP_N, lq * SP_H,
                             tc::policy_evict_first());
        ++p_issued;
      }
    }
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1;
      const uint32_t mask = __ballot_sync(0xffffffffu, idn >= 0 && idn < n);
      if (!DS) {
        const int sn = (j + 1) * SP_N + cofs + lane;
        idn = sn < a.topk ? __ldg(idx_row + sn) : -1;
      }
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&acc_full[b], (j >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      uint32_t x[32];
      tc::tmem_ld32(tmem + lane_base + SP_ACC + b * SP_N + cofs, x);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[b]);
      uint32_t pk[16];
      if (!DS) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float p0 = 0.f, p1 = 0.f;
          if (live && ((mask >> i) & 1u)) p0 = ex2(fmaf(__uint_as_float(x[i]), a.scale_log2, -lse2));
          if (live && ((mask >> (i + 1)) & 1u)) p1 = ex2(fmaf(__uint_as_float(x[i + 1]), a.scale_log2, -lse2));
          pk[i / 2] = pack_bf16(p0, p1);
        }
      } else {
        // this thread's 32 P values of tile j from the TMA ring (128-byte swizzled rows)
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&pfull[b], (j >> 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        uint4 pn[4];
        const unsigned char* ps = gbase + OFF_P + b * SP_PTILE + h * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) pn[c] = *reinterpret_cast<const uint4*>(ps + (((4 * hf + c) ^ (h & 7)) << 4));
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(pn);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pw[i / 2]));
          pk[i / 2] = pack_bf16(a.scale * p.x * (__uint_as_float(x[i]) - dl),
                                a.scale * p.y * (__uint_as_float(x[i + 1]) - dl));
        }
        // The slot is released only after its values have been consumed, and
        // the generic-proxy reads are ordered before the TMA (async-proxy)
        // refill that the release allows: without both, a refill could land
        // before a read and hand this thread tile j+2's P.
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&pempty[b]);
        if (tid == 0 && j + 2 < ntiles) {
          // refill this slot with tile j+2 once all eight warps have read tile j
          if (tc::mbar_wait(&pempty[b], (j >> 1) & 1, abort_flag)) {
            tc::mbar_arrive_expect_tx(&pfull[b], SP_PTILE);
            tc::tma_load_2d_hint(base + OFF_P + b * SP_PTILE, &tm_p, &pfull[b], (j + 2) * SP_N, lq * SP_H,
                                 tc::policy_evict_first());
            ++p_issued;
          } else {
            *abort_flag = 1;
          }
        }
      }
      // streaming stores (evict-first in L2): read back once per consumer
      uint4* dst = reinterpret_cast<uint4*>((DS ? dsrow : prow) + j * SP_N + cofs);
#pragma unroll
      for (int c = 0; c < 4; ++c) __stcs(dst + c, make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
    }
    if (!ok) *abort_flag = 1;
    // zero the padding slots [ntiles * 64, kp) (each half its own 32-column runs)
    __nv_bfloat16* orow = DS ? dsrow : prow;
    for (int c = ntiles * SP_N + cofs; c < a.kp; c += SP_N)
      for (int e = 0; e < 32; e += 8) *reinterpret_cast<uint4*>(orow + c + e) = make_uint4(0u, 0u, 0u, 0u);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && tid == 0) {
    raise_flag(a.flags, TSA_FLAG_TIMEOUT);
    // after an abort a P tile may still be landing: wait (bounded by time
    // only) for the last tile issued into each slot before the CTA exits
    volatile int keep_waiting = 0;
    for (int g = p_issued > 2 ? p_issued - 2 : 0; g < p_issued; ++g)
      (void)tc::mbar_wait(&pfull[g & 1], (g >> 1) & 1, &keep_waiting);
  }
  if (warp == 8) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// grid.x = 2 * nq: query q0 + blockIdx.x / 2, channel half blockIdx.x % 2.
template <int D>
__global__ void __launch_bounds__(DQ_THREADS, 1)
    mla_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_ds, const __grid_constant__ CUtensorMap tm_kv,
                         const __grid_constant__ MlaBwdArgs a) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + DQ_OFF_BAR);
  uint64_t* afull = bars;                     // [STAGES] dS tile (TMA)
  uint64_t* bfull = afull + DQ_STAGES;        // [STAGES] one expect-tx arrival per gather warp
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
  int a_issued = 0;  // dS tiles whose TMA loads thread 0 issued

  if (tid == 0) {
    for (int i = 0; i < DQ_STAGES; ++i) {
      tc::mbar_init(&afull[i], 1);
      tc::mbar_init(&bfull[i], 16);
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
        tc::fence_proxy_async_smem();  // kept from the cp.async version: the rows now arrive by TMA (async proxy) and need no proxy fence
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
    // ------------------------------------------------------------ gather (16 warps)
    // Warp g (0..15 over warps 0-3, 5-16) fetches rows 4g .. 4g+3 of each
    // 64-row tile with TMA gathers of 4 rows x one 64-channel block of its
    // channel slice (tile::gather4, 128-byte swizzle, the MN-major B layout),
    // lane c < nblk issuing block c.  A slot that is -1 (or outside its
    // sequence) has dS = 0 and fetches some row of its sequence, picked by
    // slot number so that the padding of short rows does not send every CTA
    // to the same row (a hot spot in L2).
    const int g = warp < 4 ? warp : warp - 1;
    const int w8 = g * 4;
    bool ok = true;
    int issued = 0;
    if (tid == 0) tc::prefetch_tmap(&tm_ds);
    int id_next = (lane < 4 && w8 + lane < a.topk) ? __ldg(idx_row + w8 + lane) : -1;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % DQ_STAGES;
      const int id_mine = id_next;
      const int slot_next = (j + 1) * DQ_N + w8 + lane;
      id_next = (lane < 4 && slot_next < a.topk) ? __ldg(idx_row + slot_next) : -1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&sempty[st], ((j / DQ_STAGES) & 1) ^ 1u, abort_flag))) {
        ok = false;
        break;
      }
      if (tid == 0) {
        // the dS tile of this stage (A operand) by TMA
        tc::mbar_arrive_expect_tx(&afull[st], DQ_A);
        tc::tma_load_2d_hint(base + st * DQ_STAGE, &tm_ds, &afull[st], j * DQ_N, lq * PB_H, tc::policy_evict_first());
        ++a_issued;
      }
      const int row_mine = s0 + ((id_mine >= 0 && id_mine < n) ? id_mine : (j * DQ_N + w8 + lane) % n);
      // this warp's bytes (4 rows x nblk blocks of 128 bytes) are expected before its gathers are issued
      if (lane == 0) tc::mbar_arrive_expect_tx(&bfull[st], nblk * 4 * 128);
      __syncwarp();
      const int r0 = __shfl_sync(0xffffffffu, row_mine, 0);
      const int r1 = __shfl_sync(0xffffffffu, row_mine, 1);
      const int r2 = __shfl_sync(0xffffffffu, row_mine, 2);
      const int r3 = __shfl_sync(0xffffffffu, row_mine, 3);
      if (lane < nblk)
        tc::tma_gather4(base + st * DQ_STAGE + DQ_A + lane * DQ_BBLK + w8 * 128, &tm_kv, &bfull[st], ch0 + lane * 64,
                        r0, r1, r2, r3);
      issued = j + 1;
    }
    if (!ok) *abort_flag = 1;
    // the gathers still in flight land before the CTA can exit (bounded by
    // time only, so this also runs after an abort)
    {
      volatile int keep_waiting = 0;
      for (int gg = issued > DQ_STAGES ? issued - DQ_STAGES : 0; gg < issued; ++gg)
        (void)tc::mbar_wait(&bfull[gg % DQ_STAGES], (gg / DQ_STAGES) & 1, &keep_waiting);
    }
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
  if (*abort_flag && tid == 0) {
    raise_flag(a.flags, TSA_FLAG_TIMEOUT);
    // after an abort a dS tile may still be landing: wait (bounded by time
    // only) for the last tile issued into each stage before the CTA exits
    volatile int keep_waiting = 0;
    for (int g = a_issued > DQ_STAGES ? a_issued - DQ_STAGES : 0; g < a_issued; ++g)
      (void)tc::mbar_wait(&afull[g % DQ_STAGES], (g / DQ_STAGES) & 1, &keep_waiting);
  }
  if (warp == 4) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool DS>
static cudaError_t launch_sp_t(const MlaBwdArgs& a, int nq, cudaStream_t stream) {
  constexpr int smem = sp_smem<D, DS>();
  static_assert(smem <= 227 * 1024, "shared memory budget");
  CUtensorMap tp;
  cudaError_t e = make_tmap_bf16_2d(&tp, a.p_out, (uint64_t)nq * SP_H, a.kp, SP_H, 64);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mla_bwd_sp_tc_kernel<D, DS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mla_bwd_sp_tc_kernel<D, DS><<<dim3(nq), SP_THREADS, smem, stream>>>(tp, a);
  note_launch();
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_dq_t(const MlaBwdArgs& a, int nq, cudaStream_t stream) {
  CUtensorMap tds, tkv;
  cudaError_t e = make_tmap_bf16_2d(&tds, a.ds_out, (uint64_t)nq * PB_H, a.kp, PB_H, 64);
  if (e != cudaSuccess) return e;
  // kv [T, D] bf16, boxes of one row x 64 channels for tile::gather4
  if ((e = make_tmap_bf16_2d(&tkv, a.kv, static_cast<uint64_t>(a.T), D, 1, 64)) != cudaSuccess) return e;
  static_assert(DQ_SMEM <= 227 * 1024, "shared memory budget");
  if ((e = cudaFuncSetAttribute(mla_bwd_dq_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM)) !=
      cudaSuccess)
    return e;
  mla_bwd_dq_tc_kernel<D><<<dim3(2 * nq), DQ_THREADS, DQ_SMEM, stream>>>(tds, tkv, a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_mla_bwd_pds_tc(const MlaBwdArgs& a, int D, int nq, cudaStream_t stream) {
  if (nq <= 0) return cudaSuccess;
  if (a.H != PB_H || a.kp % 128 != 0 || a.p_out == nullptr || a.ds_out == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = D == 576 ? launch_sp_t<576, false>(a, nq, stream) : launch_sp_t<512, false>(a, nq, stream);
  if (e != cudaSuccess) return e;
  return D == 576 ? launch_sp_t<576, true>(a, nq, stream) : launch_sp_t<512, true>(a, nq, stream);
}

cudaError_t launch_mla_bwd_dq_tc(const MlaBwdArgs& a, int D, int nq, cudaStream_t stream) {
  if (nq <= 0) return cudaSuccess;
  if (a.H != PB_H || a.kp % 128 != 0 || a.ds_out == nullptr) return cudaErrorInvalidValue;
  return D == 576 ? launch_dq_t<576>(a, nq, stream) : launch_dq_t<512>(a, nq, stream);
}

}  // namespace tsa
