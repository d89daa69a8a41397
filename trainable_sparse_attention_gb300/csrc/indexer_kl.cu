// Indexer training on the selected slots: the sparse KL loss against the
// attention teacher, and the backward of the indexer score (tcgen05 + TMEM +
// TMA gathers).
//
// Megatron-LM issue #7060 "Add trainable QSA sparse attention with a TileLang
// backend" ("Describe the problem": sparse KL supervision for training the
// indexer; "Describe the solution you'd like": sparse Stage-2 teacher / KL loss
// for indexer training) and Megatron-LM PR #3674 "Enable DSA CP/absorbed/THD
// paths with TileLang fused ops" (Copilot overview: sparse-KL streaming for the
// indexer loss; file table: fused indexer backward).  The pages print no
// formula; the reading taken (the same as the CPU reference's):
//
//   student  I[t,j] = score_scale * sum_h w[t,h] * ReLU(q_I[t,h] . k_I[s0 + idx[t,j]])
//   p[t,:]   = softmax over t's valid slots of I[t,:]
//   loss[t]  = KL(a[t,:] || p[t,:]) = sum_j a log(a / p)   (a = the teacher, 0 log 0 = 0)
//   dI[t,j]  = p - a on valid slots, 0 elsewhere            (the teacher is a target)
//   backward, with D = q_I[t,h] . k_I[s] and G = dI[t,j] (any caller-given weight):
//     dw[t,h]   = score_scale * sum_j G * ReLU(D)
//     dq_I[t,h] = score_scale * sum_j G * w[t,h] * [D > 0] * k_I[s]
//     dk_I[s]  += score_scale * sum_h G * w[t,h] * [D > 0] * q_I[t,h]
//
// One CTA per query.  The selected key rows k_I[s0 + idx[t, j]] are copied
// 128 at a time (cp.async into the 128-byte-swizzled K-major layout) through a
// two- or three-stage ring, and
//   D^T = K_sel q_I[t]^T        (M = 128 slots, N = NP heads, K = d_I = 128)
// lands in TMEM with slots on lanes, so every epilogue thread owns one slot and
// works on its own row of head values (ReLU, head weight, the head sum of the
// score, the [D > 0] mask of the backward) without leaving registers.
//
// KL kernel: the scores of all slots of the row are kept in shared memory; at
// the end the row's log-sum-exp, loss and dI are computed by the whole CTA.
// Backward kernel: the epilogue writes C[j,h] = score_scale G_j w_h [D > 0] in
// bf16 to shared memory (the same bytes serve as the MN-major B operand of
// dq^T and the K-major B operand of dk^T), and two more MMAs per tile give
//   dq_I[t]^T += K_sel^T C      (M = d_I, N = NP, K = 128 slots; accumulated over tiles)
//   dk^T       = q_I[t]^T C^T   (M = d_I, N = 128 slots, K = NP)
// dk^T has channels on TMEM lanes; each warp turns its 32 channels x 32 slots
// around in shared memory so that its fp32 reductions into the caller's dk
// accumulator are 16-byte vectors, 8 lanes covering one 128-byte line of a key
// row.  dw is the
// slot sum of G ReLU(D): a recursive-halving shuffle sum per tile, combined over
// the four epilogue warps at the end.
//
// Heads are padded to NP = 64 or 128 (w = 0 on the padding, so padded heads add
// exactly nothing).  Warp roles (192 threads): warps 0-3 epilogue (TMEM lane
// quadrants; slot of the tile = 32 w + lane), warp 4 producer, warp 5 TMEM
// allocator + MMA issuer.  Every wait is bounded; a timeout raises
// TSA_FLAG_TIMEOUT and the CTA winds down, releasing its TMEM.
#include <algorithm>

#include "kernels.cuh"
#include "tc.cuh"

namespace tsa {

cudaError_t make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                              uint32_t box_cols);

namespace {

constexpr int KL_M = 128;       // slots per tile
constexpr int KL_DI = 128;      // indexer head dimension (the only one built here)
constexpr int KL_THREADS = 192;
constexpr int KL_KBOX = KL_M * 128;          // one 64-channel box of a gathered tile: 16 KB
constexpr int KL_KSTAGE = 2 * KL_KBOX;       // d_I = 128: two boxes

// NP = 64: two CTAs per SM (two gather stages, at most 256 TMEM columns each,
// D^T single-buffered in the backward), so that one query's pipeline fill and
// final row pass overlap the other's tiles.  NP = 128: one CTA per SM.
template <int NP, bool BWD>
struct KlLayout {
  static constexpr int CTAS = NP == 64 ? 2 : 1;          // resident CTAs per SM
  static constexpr int STAGES = NP == 64 ? 2 : 3;        // gather ring
  static constexpr int DB = (BWD && NP == 64) ? 1 : 2;   // D^T buffers
  static constexpr int QBOX = NP * 128;                  // one 64-channel box of q_I[t] (NP rows)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * QBOX;
  static constexpr int OFF_C = OFF_K + STAGES * KL_KSTAGE;
  static constexpr int CBOX = KL_M * 128;                // 64 heads of C for the tile's 128 slots
  static constexpr int C_BYTES = BWD ? (NP / 64) * CBOX : 0;
  static constexpr int OFF_W = OFF_C + C_BYTES;          // head weights [NP]
  static constexpr int OFF_SC = OFF_W + NP * 4;          // KL: scores of the row [kTopkMaxK]
  static constexpr int SC_BYTES = BWD ? 4 * 4 * NP : kTopkMaxK * 4;  // BWD: dw partials [4 warps][NP]
  static constexpr int OFF_RED = OFF_SC + SC_BYTES;      // block reductions [8]
  static constexpr int OFF_BAR = OFF_RED + 64;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  // TMEM columns: D^T (DB buffers), then (backward) dq^T and dk^T
  static constexpr int T_D = 0;
  static constexpr int T_DQ = DB * NP;
  static constexpr int T_DK = T_DQ + NP;
  static constexpr int USED_COLS = BWD ? T_DK + KL_M : DB * NP;
  static constexpr int TMEM_COLS = USED_COLS <= 128 ? 128 : USED_COLS <= 256 ? 256 : 512;
  static_assert(CTAS * TMEM_COLS <= 512, "TMEM columns of the resident CTAs");
  static_assert(CTAS * (SMEM + 1024) <= 228 * 1024, "shared memory of the resident CTAs");
};

// Sum over the 32 lanes of N values per lane by recursive halving: afterwards
// lane L holds in v[i] (i < N/32, or v[0] for N < 32) the total of original
// index i + (N/32) * L (N >= 32).
template <int N, int O>
__device__ __forceinline__ void lane_sum_halving(float* v, int lane) {
  if constexpr (O >= 1) {
    static_assert(N >= 2, "needs at least two values per lane");
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float send = up ? v[i] : v[N / 2 + i];
      const float keep = up ? v[N / 2 + i] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
    lane_sum_halving<N / 2, O / 2>(v, lane);
  }
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

}  // namespace


template <int NP, bool BWD>
__global__ void __launch_bounds__(KL_THREADS, KlLayout<NP, BWD>::CTAS)
    indexer_sel_kernel(const __grid_constant__ CUtensorMap tm_q, const __nv_bfloat16* __restrict__ kI,
                       const __grid_constant__ IndexerSelArgs a) {
  using L = KlLayout<NP, BWD>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + L::OFF_Q, sK = base + L::OFF_K, sC = base + L::OFF_C;
  float* Ws = reinterpret_cast<float*>(gbase + L::OFF_W);
  float* sc = reinterpret_cast<float*>(gbase + L::OFF_SC);
  float* red = reinterpret_cast<float*>(gbase + L::OFF_RED);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + L::OFF_BAR);
  uint64_t* qfull = bars;                      // [1] q_I[t] landed
  uint64_t* kfull = bars + 1;                  // [STAGES] gathered tile landed
  uint64_t* kempty = kfull + L::STAGES;        // [STAGES] its MMAs are done
  uint64_t* dfull = kempty + L::STAGES;        // [DB] D^T ready
  uint64_t* dempty = dfull + 2;                // [DB] epilogue read D^T (4 warps)
  uint64_t* cfull = dempty + 2;                // [1] C tile written (4 warps)
  uint64_t* cempty = cfull + 1;                // [1] MMAs reading C done
  uint64_t* dkfull = cempty + 1;               // [1] dk^T ready
  uint64_t* dkempty = dkfull + 1;              // [1] dk^T drained (4 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dkempty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int t = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sq = seq_of(a.st, t);
  const int s0 = a.st.cu[sq];
  const int n = a.st.cu[sq + 1] - s0;
  const int ntiles = (a.topk + KL_M - 1) / KL_M;
  const int* idx_row = a.idx + (int64_t)t * a.topk;

  if (tid == 0) {
    tc::mbar_init(qfull, 1);
    for (int i = 0; i < L::STAGES; ++i) {
      tc::mbar_init(&kfull[i], 32);  // one cp.async arrival per producer lane
      tc::mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&dfull[i], 1);
      tc::mbar_init(&dempty[i], 4);
    }
    tc::mbar_init(cfull, 4);
    tc::mbar_init(cempty, 1);
    tc::mbar_init(dkfull, 1);
    tc::mbar_init(dkempty, 4);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  for (int h = tid; h < NP; h += KL_THREADS) Ws[h] = h < a.H_I ? a.w[(int64_t)t * a.H_I + h] : 0.f;
  if (warp == 5) tc::tmem_alloc(tmem_slot, L::TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // q_I[t] once by TMA (NP rows from row t * H_I; rows past this query's heads
    // meet w = 0), then each tile's 128 slot rows of k_I by cp.async: 16 lanes
    // per row, so that a warp instruction copies two whole 256-byte rows, each
    // 16-byte chunk straight to its place in the 128-byte-swizzled K-major tile
    // (chunk j of row r at r * 128 + (j ^ (r & 7)) * 16 of its 64-channel box).
    // Lane l holds the slot indices of rows 4l .. 4l+3; they travel to the
    // copying lanes by shuffle.  A slot that is -1 or outside the sequence is
    // zero-filled; the epilogue masks it.  (One TMA gather4 per 4 rows had
    // bound these kernels.)  Each lane's copies of a tile arrive on its kfull.
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::mbar_arrive_expect_tx(qfull, 2 * L::QBOX);
      for (int c = 0; c < 2; ++c) tc::tma_load_2d(sQ + c * L::QBOX, &tm_q, qfull, c * 64, t * a.H_I);
    }
    const int c16 = lane & 15, h = lane >> 4;
    const int cb = c16 >> 3, jj = c16 & 7;
    const char* ksrc = reinterpret_cast<const char*>(kI);
    bool ok = true;
    // the slot indices of tile j + 1 are loaded while tile j's stage frees up
    int id_next[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) id_next[i] = 4 * lane + i < a.topk ? __ldg(idx_row + 4 * lane + i) : -1;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % L::STAGES;
      int id[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        id[i] = id_next[i];
        const int slot = (j + 1) * KL_M + 4 * lane + i;
        id_next[i] = slot < a.topk ? __ldg(idx_row + slot) : -1;
      }
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&kempty[st], ((j / L::STAGES) & 1) ^ 1u, abort_flag))) {
        ok = false;
        break;
      }
      int r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (id[i] >= n) raise_flag(a.flags, TSA_FLAG_INDEX_RANGE);
        r[i] = (id[i] >= 0 && id[i] < n) ? s0 + id[i] : -1;
      }
      const uint32_t dst = sK + st * KL_KSTAGE + cb * KL_KBOX;
#pragma unroll 8
      for (int m = 0; m < KL_M / 2; ++m) {
        // row 2m + h is row 2 (m & 1) + h of lane m / 2
        const int ra = __shfl_sync(0xffffffffu, r[2 * (m & 1)], m >> 1);
        const int rb = __shfl_sync(0xffffffffu, r[2 * (m & 1) + 1], m >> 1);
        const int src = h ? rb : ra;
        const int row = 2 * m + h;
        cp_async16(dst + row * 128 + ((jj ^ (row & 7)) << 4), ksrc + (int64_t)(src >= 0 ? src : s0) * (KL_DI * 2) + c16 * 16,
                   src >= 0 ? 16u : 0u);
      }
      cp_async_commit();
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&kfull[st])) : "memory");
    }
    if (!ok) *abort_flag = 1;
    cp_async_wait<0>();  // this lane's copies land before the CTA can exit
    if (lane == 0) {     // and the q_I block (bounded by time only)
      volatile int keep_waiting = 0;
      (void)tc::mbar_wait(qfull, 0, &keep_waiting);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_d = tc::idesc_bf16_f32(KL_M, NP);
      constexpr uint32_t id_dq = tc::idesc_bf16_f32(KL_DI, NP) | (1u << 15) | (1u << 16);  // A, B MN-major
      constexpr uint32_t id_dk = tc::idesc_bf16_f32(KL_DI, KL_M) | (1u << 15);               // A MN-major
      bool ok = tc::mbar_wait(qfull, 0, abort_flag);
      for (int j = 0; ok && j < ntiles; ++j) {
        const int st = j % L::STAGES, acc = j % L::DB;
        if (!tc::mbar_wait(&kfull[st], (j / L::STAGES) & 1, abort_flag) ||
            (j >= L::DB && !tc::mbar_wait(&dempty[acc], ((j / L::DB) & 1) ^ 1u, abort_flag))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        tc::fence_proxy_async_smem();  // the rows arrived by cp.async (generic proxy); the MMAs read them
        const uint32_t kst = sK + st * KL_KSTAGE;
        // D^T = K_sel q_I^T (both K-major)
#pragma unroll
        for (int ks = 0; ks < KL_DI / 16; ++ks) {
          const int c = ks >> 2, kk = ks & 3;
          tc::mma_bf16_ss(tmem + L::T_D + acc * NP, tc::desc_sw128(kst + c * KL_KBOX + kk * 32),
                          tc::desc_sw128(sQ + c * L::QBOX + kk * 32), id_d, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(&dfull[acc]);
        if constexpr (BWD) {
          // the epilogue's C tile of this slot tile, and the drained dk^T of the previous one
          if (!tc::mbar_wait(cfull, j & 1, abort_flag) || (j > 0 && !tc::mbar_wait(dkempty, (j - 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          // dq^T += K_sel^T C  (K = the 128 slots, 16 per MMA)
#pragma unroll
          for (int ks = 0; ks < KL_M / 16; ++ks)
            tc::mma_bf16_ss(tmem + L::T_DQ, tc::desc_sw128_mn(kst + ks * 2048, KL_KBOX),
                            tc::desc_sw128_mn(sC + ks * 2048, L::CBOX), id_dq, (j > 0 || ks > 0) ? 1u : 0u);
          // dk^T = q_I^T C^T  (K = the NP heads)
#pragma unroll
          for (int ks = 0; ks < NP / 16; ++ks) {
            const int c = ks >> 2, kk = ks & 3;
            tc::mma_bf16_ss(tmem + L::T_DK, tc::desc_sw128_mn(sQ + ks * 2048, L::QBOX),
                            tc::desc_sw128(sC + c * L::CBOX + kk * 32), id_dk, ks > 0 ? 1u : 0u);
          }
          tc::mma_commit(cempty);
          tc::mma_commit(dkfull);
        }
        tc::mma_commit(&kempty[st]);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-3)
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int slot_in_tile = warp * 32 + lane;
    float dwacc[NP / 32];
#pragma unroll
    for (int i = 0; i < NP / 32; ++i) dwacc[i] = 0.f;
    for (int j = 0; j < ntiles; ++j) {
      const int acc = j % L::DB;
      const int slot = j * KL_M + slot_in_tile;
      const int id = slot < a.topk ? __ldg(idx_row + slot) : -1;
      const bool valid = id >= 0 && id < n;
      float g = 0.f;
      if constexpr (BWD) g = valid ? a.score_scale * __ldg(a.dscore + (int64_t)t * a.topk + slot) : 0.f;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&dfull[acc], (j / L::DB) & 1, abort_flag))) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      float part[4] = {0.f, 0.f, 0.f, 0.f};
      float dwv[BWD ? NP : 1];
#pragma unroll
      for (int cb = 0; cb < NP / 32; ++cb) {
        uint32_t r[32];
        __syncwarp();
        tc::tmem_ld32(tmem + lane_base + L::T_D + acc * NP + cb * 32, r);
        tc::tmem_ld_wait();
        if constexpr (!BWD) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            part[i & 3] = fmaf(Ws[cb * 32 + i], fmaxf(__uint_as_float(r[i]), 0.f), part[i & 3]);
        } else {
          // C[slot, h] = g w_h [D > 0] in bf16 into the swizzled tile; dw terms g ReLU(D)
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float d0 = __uint_as_float(r[i]), d1 = __uint_as_float(r[i + 1]);
            const float c0 = d0 > 0.f ? g * Ws[cb * 32 + i] : 0.f;
            const float c1 = d1 > 0.f ? g * Ws[cb * 32 + i + 1] : 0.f;
            pk[i / 2] = pack_bf16(c0, c1);
            dwv[cb * 32 + i] = g * fmaxf(d0, 0.f);
            dwv[cb * 32 + i + 1] = g * fmaxf(d1, 0.f);
          }
          if (j > 0 && cb == 0) {
            // the previous tile's dq / dk MMAs must be done with C before it is overwritten
            if (!__all_sync(0xffffffffu, tc::mbar_wait(cempty, (j - 1) & 1, abort_flag))) {
              *abort_flag = 1;
              break;
            }
          }
          unsigned char* crow = gbase + L::OFF_C + ((cb * 32) / 64) * L::CBOX;
          const int c0 = ((cb * 32) % 64) / 8;  // first 16-byte chunk of these 32 heads in the row
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(crow + sw128(slot_in_tile, c0 + q)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      if (*abort_flag) break;
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&dempty[acc]);
      if constexpr (!BWD) {
        const float s = (part[0] + part[1]) + (part[2] + part[3]);
        if (slot < a.topk) sc[slot] = valid ? s * a.score_scale + 0.f : -INFINITY;
      } else {
        tc::fence_proxy_async_smem();  // C (generic writes) before the MMAs (async proxy) read it
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(cfull);
        // dw: slot sum of this warp's 32 slots, recursive halving; lane l then holds heads (NP/32) l + i
        lane_sum_halving<NP, 16>(dwv, lane);
#pragma unroll
        for (int i = 0; i < NP / 32; ++i) dwacc[i] += dwv[i];
        // dk^T tile: this warp's 32 channels (TMEM lanes) x the tile's 128 slots, one reduction per
        // (slot, channel): every warp instruction covers one 128-byte line of a key row
        // key rows of the tile's slots cb*32 + lane (cb = 0..3), one per lane and
        // block, loaded before the wait and broadcast below
        int rowq[KL_M / 32];
#pragma unroll
        for (int cb = 0; cb < KL_M / 32; ++cb) {
          const int sl = j * KL_M + cb * 32 + lane;
          const int idc = sl < a.topk ? __ldg(idx_row + sl) : -1;
          rowq[cb] = (idc >= 0 && idc < n) ? s0 + idc : -1;
        }
        if (!__all_sync(0xffffffffu, tc::mbar_wait(dkfull, j & 1, abort_flag))) {
          *abort_flag = 1;
          break;
        }
        tc::fence_after_sync();
        // Each 32-slot block goes through shared memory (this warp's 32 rows of
        // the C tile, whose MMAs are complete) so that a lane adds four
        // channels of one key row with a 16-byte reduction: 8 lanes cover the
        // warp's 128-byte line of a row, 4 rows per instruction.
        const int ch0 = warp * 32;
        float* tb = reinterpret_cast<float*>(gbase + L::OFF_C + warp * (32 * 128));
#pragma unroll
        for (int cb = 0; cb < KL_M / 32; ++cb) {
          uint32_t r[32];
          __syncwarp();
          tc::tmem_ld32(tmem + lane_base + L::T_DK + cb * 32, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) tb[k * 32 + lane] = __uint_as_float(r[k]);  // [slot][channel]
          __syncwarp();
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const int k = 4 * m + (lane >> 3);
            const int rk = __shfl_sync(0xffffffffu, rowq[cb], k);
            const float4 v = *reinterpret_cast<const float4*>(tb + k * 32 + 4 * (lane & 7));
            if (rk >= 0) red_add_v4(a.dk_acc + (int64_t)rk * KL_DI + ch0 + 4 * (lane & 7), v.x, v.y, v.z, v.w);
          }
          __syncwarp();  // read before the next block overwrites it
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(dkempty);
      }
    }
    if constexpr (BWD) {
      float* dwp = sc;  // [4 warps][NP]
#pragma unroll
      for (int i = 0; i < NP / 32; ++i) dwp[warp * NP + (NP / 32) * lane + i] = dwacc[i];
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  if (aborted && tid == 0) raise_flag(a.flags, TSA_FLAG_TIMEOUT);
  if (!aborted) {
    if constexpr (!BWD) {
      // ---- the row's KL: max, log-sum-exp, loss, dI = p - a
      float m = -INFINITY;
      for (int s = tid; s < a.topk; s += KL_THREADS) m = fmaxf(m, sc[s]);
      m = warp_max(m);
      if (lane == 0) red[warp] = m;
      __syncthreads();
      m = red[0];
      for (int w = 1; w < KL_THREADS / 32; ++w) m = fmaxf(m, red[w]);
      __syncthreads();
      float z = 0.f;
      if (m != -INFINITY)
        for (int s = tid; s < a.topk; s += KL_THREADS) z += sc[s] == -INFINITY ? 0.f : expf(sc[s] - m);
      z = warp_sum(z);
      if (lane == 0) red[warp] = z;
      __syncthreads();
      z = 0.f;
      for (int w = 0; w < KL_THREADS / 32; ++w) z += red[w];
      __syncthreads();
      const float lz = m != -INFINITY ? m + logf(z) : 0.f;  // log-sum-exp of the valid scores
      float lsum = 0.f;
      const float* arow = a.teacher + (int64_t)t * a.topk;
      float* grow = a.dscore_out + (int64_t)t * a.topk;
      // four teacher loads per thread in flight at a time
      for (int s4 = tid; s4 < a.topk; s4 += 4 * KL_THREADS) {
        float av[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int s = s4 + u * KL_THREADS;
          av[u] = s < a.topk ? __ldg(arow + s) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int s = s4 + u * KL_THREADS;
          if (s >= a.topk) break;
          const float z_s = sc[s];
          float gval = 0.f;
          if (z_s != -INFINITY) {
            const float lp = z_s - lz;
            gval = expf(lp) - av[u];
            if (av[u] > 0.f) lsum += av[u] * (logf(av[u]) - lp);
          }
          grow[s] = gval;
        }
      }
      lsum = warp_sum(lsum);
      if (lane == 0) red[warp] = lsum;
      __syncthreads();
      if (tid == 0) {
        float tot = 0.f;
        for (int w = 0; w < KL_THREADS / 32; ++w) tot += red[w];
        a.loss[t] = tot;
      }
    } else {
      // ---- dq_I[t] from TMEM (lane = channel), dw[t] from the warps' partials
      if (warp < 4) {
        tc::fence_after_sync();
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const int ch = warp * 32 + lane;
#pragma unroll 1
        for (int cb = 0; cb < NP / 32; ++cb) {
          uint32_t r[32];
          __syncwarp();
          tc::tmem_ld32(tmem + lane_base + L::T_DQ + cb * 32, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int h = cb * 32 + i;
            if (h < a.H_I) a.dq[((int64_t)t * a.H_I + h) * KL_DI + ch] = __float2bfloat16_rn(__uint_as_float(r[i]));
          }
        }
      }
      for (int h = tid; h < a.H_I; h += KL_THREADS) {
        const float* dwp = sc;
        a.dw[(int64_t)t * a.H_I + h] = (dwp[h] + dwp[NP + h]) + (dwp[2 * NP + h] + dwp[3 * NP + h]);
      }
    }
  }
  if (warp == 5) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- teacher from staged P

// The teacher of the 128-head backward: the staged bf16 probabilities of one
// chunk of queries, P[lq][h][kp] (slots >= topk are zero), averaged over the
// heads: teacher[q0 + lq][j] = (1/128) sum_h P[lq][h][j].  One CTA per query;
// thread i sums slots 8i .. 8i+7 (16-byte loads, consecutive threads on
// consecutive bytes of a head's row).
__global__ void __launch_bounds__(256) mla_teacher_from_p_kernel(const __nv_bfloat16* __restrict__ P, int H,
                                                                 int kp, int topk, int q0,
                                                                 float* __restrict__ teacher) {
  const int lq = blockIdx.x;
  const uint4* rowp = reinterpret_cast<const uint4*>(P + (int64_t)lq * H * kp);
  const int vpr = kp / 8;  // 16-byte vectors per head row
  const float inv_h = 1.f / static_cast<float>(H);
  for (int v = threadIdx.x; v * 8 < topk; v += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int h = 0; h < H; ++h) {
      const uint4 x = __ldg(rowp + (int64_t)h * vpr + v);
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(p2[i]);
        acc[2 * i] += f.x;
        acc[2 * i + 1] += f.y;
      }
    }
    float* out = teacher + (int64_t)(q0 + lq) * topk + v * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (v * 8 + i < topk) out[i] = acc[i] * inv_h;
  }
}

cudaError_t launch_mla_teacher_from_p(const __nv_bfloat16* P, int nq, int H, int kp, int topk, int q0,
                                      float* teacher, cudaStream_t stream) {
  if (nq <= 0) return cudaSuccess;
  if (kp % 8 != 0 || kp < topk) return cudaErrorInvalidValue;
  mla_teacher_from_p_kernel<<<nq, 256, 0, stream>>>(P, H, kp, topk, q0, teacher);
  note_launch();
  return cudaGetLastError();
}

// ---------------------------------------------------------------- host side

bool indexer_sel_supported(int H_I, int d_I) {
  return d_I == KL_DI && H_I >= 1 && H_I <= 128;
}

template <int NP, bool BWD>
static cudaError_t launch_sel_t(const IndexerSelArgs& a, const void* q, const void* k, int T_total,
                                cudaStream_t stream) {
  using L = KlLayout<NP, BWD>;
  static_assert(L::SMEM <= 227 * 1024, "indexer selection kernel shared memory");
  CUtensorMap tq;
  cudaError_t e = make_tmap_bf16_2d(&tq, q, (uint64_t)T_total * a.H_I, KL_DI, NP, 64);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(indexer_sel_kernel<NP, BWD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                L::SMEM)) != cudaSuccess)
    return e;
  indexer_sel_kernel<NP, BWD><<<a.T, KL_THREADS, L::SMEM, stream>>>(tq, static_cast<const __nv_bfloat16*>(k), a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_indexer_sel(const IndexerSelArgs& a, const void* q, const void* k, bool bwd,
                               cudaStream_t stream) {
  if (a.T <= 0 || a.topk <= 0) return cudaSuccess;
  if (a.topk > kTopkMaxK) return cudaErrorInvalidValue;
  if (a.H_I <= 64) return bwd ? launch_sel_t<64, true>(a, q, k, a.T, stream) : launch_sel_t<64, false>(a, q, k, a.T, stream);
  return bwd ? launch_sel_t<128, true>(a, q, k, a.T, stream) : launch_sel_t<128, false>(a, q, k, a.T, stream);
}

}  // namespace tsa
