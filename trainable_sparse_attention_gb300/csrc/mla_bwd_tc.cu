// Sparse MLA backward for 128 heads on tcgen05: the dKV GEMM and its scatter.
//
// Megatron-LM PR #3674 "Enable DSA CP/absorbed/THD paths with TileLang fused
// ops" (sparse MLA backward) and Megatron-LM PR #7617 "Support NoPE shapes and
// unaligned top-k in TileLang sparse MLA" ("Validation": the backward
// accumulates dKV atomically).
//
// For one query t with selected rows idx[t, 0..topk) the key/value gradient is
//   dKV[idx[t, s], c] += sum_h dS[t, h, s] q[t, h, c] + P[t, h, s] dO[t, h, c]
// (the dO term only for the 512 value channels; dS already carries the
// softmax scale).  The preceding launch leaves P and dS of a chunk of queries
// in bf16 in the workspace, laid out [query][head][slot] with the slots padded
// to a multiple of 128 by zeros.
//
// Here one CTA owns (query, 128-channel block) and computes the block
// transposed, D[c, s] (M = 128 channels, N = 128 slots per tile, K = 128
// heads), so that TMEM lane = channel: every warp holds 32 consecutive channels
// of a slot row and its fp32 reductions into dKV cover whole 128-byte lines.
// The q / dO blocks are the fixed A operand (MN-major, loaded once by TMA);
// the dS / P tiles stream through a two-stage TMA pipeline as the MN-major B
// operand; the accumulator is double-buffered in TMEM so that the drain of
// tile j overlaps the MMAs of tile j+1.  Sixteen drain warps (four per TMEM lane
// quadrant) keep enough reductions in flight.  All 128 heads are summed before the
// scatter, so each selected row receives one reduction per query.
#include "kernels.cuh"
#include "tc.cuh"

namespace tsa {

cudaError_t make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                              uint32_t box_cols);

namespace {

constexpr int BH = 128;           // heads = MMA K of this GEMM
constexpr int DK_NS = 128;        // slots per tile (MMA N)
constexpr int DK_STAGES = 2;
constexpr int DK_THREADS = 576;   // warps 0-15 drain, warp 16 TMA producer, warp 17 MMA
constexpr int DK_DRAIN = 16;      // drain warps: TMEM lane quadrant w % 4, 32-slot piece w / 4
constexpr int DK_BOX = BH * 128;  // one 64-column box of 128 rows: 16 KB
constexpr int DK_A = 2 * DK_BOX;  // one 128-channel A block (q or dO): 32 KB
constexpr int DK_B = 2 * DK_BOX;  // one 128-slot B tile (dS or P): 32 KB
constexpr int DK_XP = 16 * 32 * 4;  // per-warp transpose buffer (16 slots x 32 channels): 2 KB
constexpr int DK_OFF_AQ = 0;
constexpr int DK_OFF_AO = DK_OFF_AQ + DK_A;
constexpr int DK_OFF_B = DK_OFF_AO + DK_A;
constexpr int DK_OFF_X = DK_OFF_B + DK_STAGES * 2 * DK_B;
constexpr int DK_OFF_BAR = DK_OFF_X + DK_DRAIN * DK_XP;
constexpr int DK_SMEM = 1024 + DK_OFF_BAR + 256;
static_assert(DK_SMEM <= 227 * 1024, "dKV kernel shared memory");

__device__ __forceinline__ void red_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

}  // namespace

// grid.x = nq * nblk: query q0 + blockIdx.x / nblk, channel block blockIdx.x % nblk.
__global__ void __launch_bounds__(DK_THREADS, 1)
    mla_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tm_ds, const __grid_constant__ CUtensorMap tm_p,
                          const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ MlaBwdTcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + DK_OFF_BAR);
  uint64_t* afull = bars;                      // [1]
  uint64_t* bfull = bars + 1;                  // [STAGES]
  uint64_t* bempty = bfull + DK_STAGES;        // [STAGES]
  uint64_t* dfull = bempty + DK_STAGES;        // [2]
  uint64_t* dempty = dfull + 2;                // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int nblk = (a.D + 127) / 128;
  const int lq = blockIdx.x / nblk;
  const int t = a.q0 + lq;
  const int ch0 = (blockIdx.x % nblk) * 128;
  const int nch = min(128, a.D - ch0);  // 128, or 64 for the rope block of D = 576
  const bool has_v = ch0 < 512;         // the block holds value channels (the dO term applies)
  // The rope block of D = 576 (64 channels) leaves accumulator lanes 64..127
  // empty: with the indexer's teacher requested, its P term runs against a
  // constant A whose channel 64 is 1/128 for every head, so accumulator lane 64
  // is (1/128) sum_h P[h, slot], the head mean of the probabilities.
  const bool has_t = a.teacher != nullptr && nch == 64;
  const int ntiles = a.kp / DK_NS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int b_issued = 0;  // P / dS tiles whose TMA loads the producer issued

  if (tid == 0) {
    tc::mbar_init(afull, 1);
    for (int i = 0; i < DK_STAGES; ++i) {
      tc::mbar_init(&bfull[i], 1);
      tc::mbar_init(&bempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&dfull[i], 1);
      tc::mbar_init(&dempty[i], DK_DRAIN);
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (nch < 128) {
    // the second 64-channel box of a 64-channel block is never loaded: zero it (rows 64..127 of A)
    uint4* z = reinterpret_cast<uint4*>(gbase + DK_OFF_AQ + DK_BOX);
    for (int i = tid; i < DK_BOX / 16; i += DK_THREADS) z[i] = make_uint4(0u, 0u, 0u, 0u);
    if (has_t) {
      // the teacher's constant A (MN-major, head rows of 128 bytes, 128-byte
      // swizzle): zero, then 1/128 (bf16 0x3C00) at channel 64 of every head
      // row -- element 0 of the second box, whose 16-byte chunk 0 sits at
      // chunk (0 ^ (row & 7)) of the row
      uint4* zo = reinterpret_cast<uint4*>(gbase + DK_OFF_AO);
      for (int i = tid; i < 2 * DK_BOX / 16; i += DK_THREADS) zo[i] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      for (int h = tid; h < BH; h += DK_THREADS)
        *reinterpret_cast<unsigned short*>(gbase + DK_OFF_AO + DK_BOX + h * 128 + ((h & 7) << 4)) = 0x3C00u;
    }
    tc::fence_proxy_async_smem();
  }
  if (warp == 17) tc::tmem_alloc(tmem_slot, 256);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 16) {
    if (lane == 0) {
      const uint32_t sAq = base + DK_OFF_AQ, sAo = base + DK_OFF_AO;
      const int qboxes = nch / 64;
      tc::mbar_arrive_expect_tx(afull, (qboxes + (has_v ? 2 : 0)) * DK_BOX);
      for (int c = 0; c < qboxes; ++c) tc::tma_load_2d(sAq + c * DK_BOX, &tm_q, afull, ch0 + c * 64, t * BH);
      if (has_v)
        for (int c = 0; c < 2; ++c) tc::tma_load_2d(sAo + c * DK_BOX, &tm_do, afull, ch0 + c * 64, t * BH);
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % DK_STAGES;
        if (!tc::mbar_wait(&bempty[st], ((j / DK_STAGES) & 1) ^ 1u, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        tc::mbar_arrive_expect_tx(&bfull[st], (has_v || has_t ? 2 : 1) * DK_B);
        const uint32_t dst = base + DK_OFF_B + st * 2 * DK_B;
        const uint64_t pol = tc::policy_evict_first();  // P / dS tiles: read by this query's CTAs only
        for (int c = 0; c < 2; ++c) {
          tc::tma_load_2d_hint(dst + c * DK_BOX, &tm_ds, &bfull[st], j * DK_NS + c * 64, lq * BH, pol);
          if (has_v || has_t)
            tc::tma_load_2d_hint(dst + DK_B + c * DK_BOX, &tm_p, &bfull[st], j * DK_NS + c * 64, lq * BH, pol);
        }
        ++b_issued;
      }
    }
  } else if (warp == 17) {
    if (lane == 0) {
      // A (q / dO block, channels contiguous) and B (dS / P tile, slots contiguous) are both MN-major.
      const uint32_t idesc = tc::idesc_bf16_f32(128, DK_NS) | (1u << 15) | (1u << 16);
      const uint32_t sAq = base + DK_OFF_AQ, sAo = base + DK_OFF_AO;
      bool ok = tc::mbar_wait(afull, 0, abort_flag);
      for (int j = 0; ok && j < ntiles; ++j) {
        const int st = j % DK_STAGES, acc = j & 1;
        if (!tc::mbar_wait(&bfull[st], (j / DK_STAGES) & 1, abort_flag) ||
            !tc::mbar_wait(&dempty[acc], ((j >> 1) & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + acc * DK_NS;
        const uint32_t bS = base + DK_OFF_B + st * 2 * DK_B, bP = bS + DK_B;
#pragma unroll
        for (int ks = 0; ks < BH / 16; ++ks)
          tc::mma_bf16_ss(d, tc::desc_sw128_mn(sAq + ks * 2048, DK_BOX), tc::desc_sw128_mn(bS + ks * 2048, DK_BOX),
                          idesc, ks > 0 ? 1u : 0u);
        if (has_v || has_t) {
#pragma unroll
          for (int ks = 0; ks < BH / 16; ++ks)
            tc::mma_bf16_ss(d, tc::desc_sw128_mn(sAo + ks * 2048, DK_BOX), tc::desc_sw128_mn(bP + ks * 2048, DK_BOX),
                            idesc, 1u);
        }
        tc::mma_commit(&bempty[st]);
        tc::mma_commit(&dfull[acc]);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ drain
    // warp w: channels 32 (w % 4) .. +31 (its TMEM lane quadrant), slots
    // 32 (w / 4) .. +31 of each tile, transposed through shared memory in two
    // halves of 16 slots.  The slot rows of the next tile are loaded while
    // this one drains.
    const int qd = warp & 3, pc = warp >> 2;
    const int sq = seq_of(a.st, t);
    const int s0 = a.st.cu[sq];
    const int n = a.st.cu[sq + 1] - s0;
    const int* idx_row = a.idx + (int64_t)t * a.topk;
    float* xb = reinterpret_cast<float*>(gbase + DK_OFF_X + warp * DK_XP);  // [16 slots][32 channels]
    const bool live = qd * 32 < nch;
    const int cq = (lane & 7) * 4;  // this lane's 4 channels within the warp's 32 in the scatter
    float* dkv_base = a.dkv_acc + ch0 + qd * 32 + cq;
    auto rows_of = [&](int j) -> int {
      const int slot = j * DK_NS + pc * 32 + lane;
      if (slot >= a.topk) return -1;
      const int id = __ldg(idx_row + slot);
      return (id >= 0 && id < n) ? s0 + id : -1;
    };
    int nx = live ? rows_of(0) : -1;
    for (int j = 0; j < ntiles; ++j) {
      const int acc = j & 1;
      const int my = nx;
      if (live && j + 1 < ntiles) nx = rows_of(j + 1);
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&dfull[acc], (j >> 1) & 1, abort_flag))) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      if (has_t && qd == 2) {
        // accumulator lane 64 (this quadrant's lane 0): the teacher of slots pc*32 .. +31 of the tile
        uint32_t r[32];
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(qd * 32) << 16) + acc * DK_NS + pc * 32, r);
        tc::tmem_ld_wait();
        if (lane == 0) {
          float* trow = a.teacher + (int64_t)t * a.topk + j * DK_NS + pc * 32;
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (j * DK_NS + pc * 32 + k < a.topk) trow[k] = __uint_as_float(r[k]);
        }
      }
      if (live) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(qd * 32) << 16) + acc * DK_NS + pc * 32, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // transpose through shared memory: xb[slot][channel]
#pragma unroll
          for (int i = 0; i < 16; ++i) xb[i * 32 + lane] = __uint_as_float(r[16 * hh + i]);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int sl = 4 * k + (lane >> 3);
            const int row = __shfl_sync(0xffffffffu, my, 16 * hh + sl);
            const float4 v = *reinterpret_cast<const float4*>(xb + sl * 32 + cq);
            if (row >= 0) red_v4(dkv_base + (int64_t)row * a.D, v.x, v.y, v.z, v.w);
          }
          __syncwarp();
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&dempty[acc]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && tid == 0) raise_flag(a.flags, TSA_FLAG_TIMEOUT);
  if (*abort_flag && warp == 16 && lane == 0) {
    // after an abort the q / dO boxes or a P / dS tile may still be landing:
    // wait (bounded by time only) for them before the CTA exits
    volatile int keep_waiting = 0;
    (void)tc::mbar_wait(afull, 0, &keep_waiting);
    for (int g = b_issued > DK_STAGES ? b_issued - DK_STAGES : 0; g < b_issued; ++g)
      (void)tc::mbar_wait(&bfull[g % DK_STAGES], (g / DK_STAGES) & 1, &keep_waiting);
  }
  if (warp == 17) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 256);
  }
}

cudaError_t launch_mla_bwd_dkv_tc(const MlaBwdTcArgs& a, int nq, cudaStream_t stream) {
  if (nq <= 0) return cudaSuccess;
  CUtensorMap tds, tp, tq, tdo;
  cudaError_t e;
  if ((e = make_tmap_bf16_2d(&tds, a.ds, (uint64_t)nq * BH, a.kp, BH, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16_2d(&tp, a.p, (uint64_t)nq * BH, a.kp, BH, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16_2d(&tq, a.q, (uint64_t)a.T * BH, a.D, BH, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16_2d(&tdo, a.dout, (uint64_t)a.T * BH, 512, BH, 64)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(mla_bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DK_SMEM)) !=
      cudaSuccess)
    return e;
  const int nblk = (a.D + 127) / 128;
  mla_bwd_dkv_tc_kernel<<<dim3(nq * nblk), DK_THREADS, DK_SMEM, stream>>>(tds, tp, tq, tdo, a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tsa
