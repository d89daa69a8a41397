// Block Sparse-GQA forward and backward on tcgen05 (TMEM accumulators, TMA
// tile::gather4 staging, mbarrier pipelines), key-centric.
//
// Megatron-LM issue #7060 "Add trainable QSA sparse attention with a TileLang
// backend" ("Describe the solution you'd like": Sparse-GQA forward and backward
// kernels over exact block top-k selections, BSHD and packed THD).
//
// A query selects nsel blocks per kv group, each a run of block_size keys it
// attends causally.  Gathered per query, every (query, group, block) triple
// moves a block_size x d tile of K and of V for only G = Hq / Hkv heads of the
// query (8 bytes of gather per flop at G = 8): the work is bound by row copies,
// and the G rows of one query fill at most 16 of the 128 rows of an MMA.
// Inverted, it is dense: the selections are turned into one list per (block,
// group) of the queries that chose that block (count, scan, fill), and a CTA
// takes a chunk of a list.  The block's K and V are staged once; the chunk's
// queries pass through in batches of 128 (query, head) rows -- 128 / G queries
// of G heads -- so every MMA is M = 128 rows x N = 64 keys:
//
//   forward, per batch:   S = Q K^T (TMEM), P = exp(scale S - m) on the causal
//                         keys (rows on TMEM lanes: one thread per row, the row
//                         maximum and sum never leave the thread), P to TMEM as
//                         bf16, O = P V (A operand read from TMEM);
//                         the normalised partial O / l (bf16) and its
//                         log-sum-exp (fp32) go to the slot (query, group, j)
//                         of the selection in the caller's workspace;
//   combine:              per (query, head), the partials of the selected
//                         blocks are merged in slot order: the result does not
//                         depend on the order of the inverted lists, so the
//                         forward replays bit for bit;
//   backward, per batch:  S = Q K^T and dP = dO V^T (TMEM), P = exp(scale S - lse)
//                         and dS = scale P (dP - Delta) written to shared memory
//                         in bf16, then dV^T += dO^T P and dK^T += Q^T dS
//                         (accumulated in TMEM over the whole chunk, reduced once
//                         per chunk) and dQ^T = K^T dS^T, whose channels sit on
//                         TMEM lanes; each warp turns its 32 channels x 32 rows
//                         around in shared memory so that its fp32 reductions
//                         into the dQ accumulator are 16-byte vectors, 8 lanes
//                         per 128-byte line.  The backward's batches flow
//                         through three groups of warps at once: two loader
//                         warps copy the next batches' Q and dO rows with
//                         cp.async (the TMA gathers' one-instruction-per-4-rows
//                         rate bound the kernel), eight row warps turn S / dP
//                         into P / dS, and four drain warps reduce the previous
//                         batch's dQ^T from the second of two TMEM buffers.
//
// Head dimension 64 runs as 128 with channels 64..127 zero in shared memory,
// and blocks of 32 keys as 64-key tiles whose upper half is masked: the MMA
// shapes stay M = 128, N = 64 / 128.
#include <algorithm>

#include "kernels.cuh"
#include "tc.cuh"

namespace tsa {

cudaError_t make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                              uint32_t box_cols);

namespace {

constexpr int GT_ROWS = 128;              // (query, head) rows per batch = MMA M
constexpr int GT_KEYS = 64;               // key tile = MMA N (a 32-key block is padded)
constexpr int GT_DP = 128;                // head dimension in shared memory (64 is zero padded)
constexpr int GT_THREADS = 192;           // warps 0-3 rows / drain, warp 4 producer, warp 5 MMA
constexpr int GT_QBOX = GT_ROWS * 128;    // 128 rows x 64 channels bf16: 16 KB
constexpr int GT_QT = 2 * GT_QBOX;        // a Q (or dO) batch: 32 KB
constexpr int GT_KBOX = GT_KEYS * 128;    // 64 keys x 64 channels: 8 KB
constexpr int GT_KT = 2 * GT_KBOX;        // the K (or V) tile: 16 KB
constexpr int GT_PT = GT_ROWS * 128;      // P or dS: 128 rows x 64 keys bf16: 16 KB

// forward: K, V, two Q buffers, two row tables
constexpr int GF_OFF_K = 0;
constexpr int GF_OFF_V = GF_OFF_K + GT_KT;
constexpr int GF_OFF_Q = GF_OFF_V + GT_KT;
constexpr int GF_OFF_TAB = GF_OFF_Q + 2 * GT_QT;       // int [2][128]: selection entry of each row, -1 = none
constexpr int GF_OFF_BAR = GF_OFF_TAB + 2 * GT_ROWS * 4;
constexpr int GF_SMEM = 1024 + GF_OFF_BAR + 256;
// TMEM (forward): S 64 columns, P 32 (bf16 pairs), O 128
constexpr int GF_T_S = 0, GF_T_P = 64, GF_T_O = 128, GF_TMEM = 256;

__device__ __forceinline__ int gt_block_seq(const GqaTcArgs& a, int gb) {
  int lo = 0, hi = a.st.num_seqs - 1;  // last sequence whose first block is <= gb
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.blk_base[mid] <= gb) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void red_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

}  // namespace

// ---------------------------------------------------------------- selection inversion

// Selection entries e = (t, g, j) that name a causal block of t's sequence:
// count them per (query segment t / qseg, global block, group), or (FILL)
// append e itself (the flat index (t * Hkv + g) * nsel + j, which is also the
// entry's partial slot) to that list.  Lists are numbered segment-major, so the
// grid takes the lists of one segment of queries before the next: the
// backward's CTAs running together then reduce into one segment's slice of the
// dQ accumulator, which fits in L2.  Entries outside the sequence raise
// TSA_FLAG_INDEX_RANGE and are dropped.
template <bool FILL>
__global__ void gqa_tc_inv_kernel(const __grid_constant__ GqaTcArgs a) {
  const int64_t total = static_cast<int64_t>(a.T) * a.Hkv * a.nsel;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = __ldg(a.blk + e);
    if (b < 0) continue;
    const int t = static_cast<int>(e / (static_cast<int64_t>(a.Hkv) * a.nsel));
    const int g = static_cast<int>((e / a.nsel) % a.Hkv);
    const int s = seq_of(a.st, t);
    const int p = t - a.st.cu[s];
    const int n = a.st.cu[s + 1] - a.st.cu[s];
    if (static_cast<int64_t>(b) * a.bs >= n) {
      if (!FILL) raise_flag(a.flags, TSA_FLAG_INDEX_RANGE);
      continue;
    }
    if (static_cast<int64_t>(b) * a.bs > p) continue;  // not a causal block of this query
    const int idx = ((t / a.qseg) * a.nblk + a.blk_base[s] + b) * a.Hkv + g;
    if (!FILL) {
      atomicAdd(a.cnt + idx, 1);
    } else {
      const int pos = atomicAdd(a.cur + idx, 1);
      a.list[a.off[idx] + pos] = static_cast<int>(e);
    }
  }
}

// Exclusive scans of the list sizes (offsets) and of the chunks per list;
// clears the fill cursors.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) gqa_tc_scan_kernel(const __grid_constant__ GqaTcArgs a, int nB, int chunk) {
  __shared__ int warp_tot[2][32];
  __shared__ int carry[2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < 2) carry[threadIdx.x] = 0;
  __syncthreads();
  for (int base = 0; base < nB; base += 1024) {
    const int i = base + threadIdx.x;
    const int c = i < nB ? a.cnt[i] : 0;
    const int ch = (c + chunk - 1) / chunk;
    if (i < nB) a.cur[i] = 0;
    int x = c, y = ch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xv = __shfl_up_sync(0xffffffffu, x, o), yv = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) { x += xv; y += yv; }
    }
    if (lane == 31) { warp_tot[0][warp] = x; warp_tot[1][warp] = y; }
    __syncthreads();
    int px = carry[0], py = carry[1];
    for (int w = 0; w < warp; ++w) { px += warp_tot[0][w]; py += warp_tot[1][w]; }
    if (i < nB) { a.off[i] = px + x - c; a.choff[i] = py + y - ch; }
    __syncthreads();
    if (threadIdx.x == 1023) { carry[0] = px + x; carry[1] = py + y; }
    __syncthreads();
  }
  if (threadIdx.x == 0) { a.off[nB] = carry[0]; a.choff[nB] = carry[1]; }
}

// The chunk of CTA c: its list (block, group) and entry range.  Returns false if c is past the last chunk.
struct GtChunk {
  int g, s0, n, kbase, e0, e1;
};
__device__ __forceinline__ bool gt_chunk(const GqaTcArgs& a, int c, int chunk, GtChunk& ck) {
  const int nB = a.nblk * a.Hkv;
  const int nL = a.nseg * nB;
  if (c >= a.choff[nL]) return false;
  int lo = 0, hi = nL - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.choff[mid] <= c) lo = mid; else hi = mid - 1;
  }
  const int bg = lo % nB;  // (block, group) of the list
  const int gb = bg / a.Hkv;
  ck.g = bg % a.Hkv;
  const int sq = gt_block_seq(a, gb);
  ck.s0 = a.st.cu[sq];
  ck.n = a.st.cu[sq + 1] - ck.s0;
  ck.kbase = (gb - a.blk_base[sq]) * a.bs;
  ck.e0 = a.off[lo] + (c - a.choff[lo]) * chunk;
  ck.e1 = min(a.off[lo + 1], ck.e0 + chunk);
  return true;
}

// ---------------------------------------------------------------- forward: partials

// Producer helper: gather the block's 64 key rows (K or V, [T * Hkv, d] view)
// into a 64 x 128-channel tile; rows past the block or the sequence repeat the
// block's first row (masked by the consumers).
__device__ __forceinline__ void gt_gather_kv(uint32_t dst, const CUtensorMap* map, uint64_t* bar, const GqaTcArgs& a,
                                             const GtChunk& ck, int lane) {
  if (lane < 16) {
    int r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int key = 4 * lane + i;
      const int kp = ck.kbase + key;
      const bool ok = key < a.bs && kp < ck.n;
      r[i] = (ck.s0 + (ok ? kp : ck.kbase)) * a.Hkv + ck.g;
    }
    tc::tma_gather4(dst + 4 * lane * 128, map, bar, 0, r[0], r[1], r[2], r[3]);
    if (a.d == 128) tc::tma_gather4(dst + GT_KBOX + 4 * lane * 128, map, bar, 64, r[0], r[1], r[2], r[3]);
  }
}

// Producer helpers: the rows of one batch (entries eb .. eb + qb of the chunk,
// G heads each); lane l owns rows 4l .. 4l+3.  gt_batch_rows computes their
// source rows of the [T * Hq, d] view and, if tab is given, records for each
// row its selection entry (t * Hkv + g) * nsel + j, or with tab_rows that
// source row t * Hq + h, or -1; gt_gather_batch issues the gathers into a
// 128-row Q (or dO) buffer.
__device__ __forceinline__ void gt_batch_rows(const GqaTcArgs& a, const GtChunk& ck, int eb, int* tab, bool tab_rows,
                                              int lane, int (&r)[4]) {
  const int G = a.G, qb = GT_ROWS / G;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = 4 * lane + i;
    const int qi = row / G, hh = row - qi * G;
    const int ei = eb + qi;
    const bool ok = qi < qb && ei < ck.e1;
    const int e = ok ? __ldg(a.list + ei) : -1;
    r[i] = (ok ? e / (a.Hkv * a.nsel) : 0) * a.Hq + ck.g * G + hh;
    if (tab != nullptr) tab[row] = ok ? (tab_rows ? r[i] : e) : -1;
  }
}
__device__ __forceinline__ void gt_gather_batch(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int d,
                                                const int (&r)[4], int lane) {
  tc::tma_gather4(dst + 4 * lane * 128, map, bar, 0, r[0], r[1], r[2], r[3]);
  if (d == 128) tc::tma_gather4(dst + GT_QBOX + 4 * lane * 128, map, bar, 64, r[0], r[1], r[2], r[3]);
}

__global__ void __launch_bounds__(GT_THREADS, 2)
    gqa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ GqaTcArgs a, int chunk) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t sK = base + GF_OFF_K, sV = base + GF_OFF_V, sQ = base + GF_OFF_Q;
  int* tab = reinterpret_cast<int*>(gbase + GF_OFF_TAB);  // [2][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + GF_OFF_BAR);
  uint64_t* kvfull = bars;        // [1]
  uint64_t* qfull = bars + 1;     // [2]
  uint64_t* qempty = qfull + 2;   // [2] S MMA done with the Q buffer and rows done with its table
  uint64_t* sfull = qempty + 2;   // [1]
  uint64_t* sempty = sfull + 1;   // [1] rows read S (4 warps)
  uint64_t* pfull = sempty + 1;   // [1] rows wrote P (4 warps)
  uint64_t* pempty = pfull + 1;   // [1] PV done with P
  uint64_t* ofull = pempty + 1;   // [1]
  uint64_t* oempty = ofull + 1;   // [1] rows read O (4 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(oempty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  GtChunk ck;
  if (!gt_chunk(a, blockIdx.x, chunk, ck)) return;  // uniform
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qb = GT_ROWS / a.G;
  const int nbatch = (ck.e1 - ck.e0 + qb - 1) / qb;
  int issued = 0;  // producer: batches whose gathers were issued

  if (tid == 0) {
    tc::mbar_init(kvfull, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&qfull[i], 1);
      tc::mbar_init(&qempty[i], 1 + 4);  // the MMA commit and the four row warps
    }
    tc::mbar_init(sfull, 1);
    tc::mbar_init(sempty, 4);
    tc::mbar_init(pfull, 4);
    tc::mbar_init(pempty, 1);
    tc::mbar_init(ofull, 1);
    tc::mbar_init(oempty, 4);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (a.d == 64) {
    // channels 64..127 of every operand tile are never loaded: zero them once
    for (int i = tid; i < GT_KBOX / 16; i += GT_THREADS) {
      reinterpret_cast<uint4*>(gbase + GF_OFF_K + GT_KBOX)[i] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(gbase + GF_OFF_V + GT_KBOX)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int i = tid; i < GT_QBOX / 16; i += GT_THREADS) {
      reinterpret_cast<uint4*>(gbase + GF_OFF_Q + GT_QBOX)[i] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(gbase + GF_OFF_Q + GT_QT + GT_QBOX)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_proxy_async_smem();
  }
  if (warp == 5) tc::tmem_alloc(tmem_slot, GF_TMEM);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t kv_bytes = (a.d == 128 ? 2 : 1) * 2 * GT_KBOX;
  const uint32_t q_bytes = (a.d == 128 ? 2 : 1) * GT_QBOX;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
      tc::prefetch_tmap(&tm_v);
      tc::mbar_arrive_expect_tx(kvfull, kv_bytes);
    }
    __syncwarp();
    gt_gather_kv(sK, &tm_k, kvfull, a, ck, lane);
    gt_gather_kv(sV, &tm_v, kvfull, a, ck, lane);
    bool ok = true;
    for (int i = 0; i < nbatch; ++i) {
      const int buf = i & 1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&qempty[buf], ((i >> 1) & 1) ^ 1u, abort_flag))) {
        ok = false;
        break;
      }
      // the row table is read by the row warps after they see qfull: every lane
      // writes its rows' entries before lane 0's arrival releases them
      int r[4];
      gt_batch_rows(a, ck, ck.e0 + i * qb, tab + buf * GT_ROWS, false, lane, r);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_expect_tx(&qfull[buf], q_bytes);
      __syncwarp();
      gt_gather_batch(sQ + buf * GT_QT, &tm_q, &qfull[buf], a.d, r, lane);
      issued = i + 1;
    }
    if (!ok) *abort_flag = 1;
    if (lane == 0) {  // copies still in flight land before the CTA exits (bounded by time only)
      volatile int keep_waiting = 0;
      (void)tc::mbar_wait(kvfull, 0, &keep_waiting);
      for (int g = issued > 2 ? issued - 2 : 0; g < issued; ++g)
        (void)tc::mbar_wait(&qfull[g & 1], (g >> 1) & 1, &keep_waiting);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = tc::idesc_bf16_f32(GT_ROWS, GT_KEYS);
      constexpr uint32_t id_o = tc::idesc_bf16_f32_bmn(GT_ROWS, GT_DP);
      bool ok = tc::mbar_wait(kvfull, 0, abort_flag);
      for (int i = 0; ok && i < nbatch; ++i) {
        const int buf = i & 1;
        const uint32_t ph = i & 1;
        if (!tc::mbar_wait(&qfull[buf], (i >> 1) & 1, abort_flag) ||
            (i > 0 && !tc::mbar_wait(sempty, ph ^ 1u, abort_flag))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t qt = sQ + buf * GT_QT;
#pragma unroll
        for (int ks = 0; ks < GT_DP / 16; ++ks) {
          const int c = ks >> 2, kk = ks & 3;
          tc::mma_bf16_ss(tmem + GF_T_S, tc::desc_sw128(qt + c * GT_QBOX + kk * 32),
                          tc::desc_sw128(sK + c * GT_KBOX + kk * 32), id_s, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(sfull);
        tc::mma_commit(&qempty[buf]);
        if (!tc::mbar_wait(pfull, ph, abort_flag) || (i > 0 && !tc::mbar_wait(oempty, ph ^ 1u, abort_flag))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < GT_KEYS / 16; ++ks)
          tc::mma_bf16_ts(tmem + GF_T_O, tmem + GF_T_P + ks * 8, tc::desc_sw128_mn(sV + ks * 2048, GT_KBOX), id_o,
                          ks > 0 ? 1u : 0u);
        tc::mma_commit(pempty);
        tc::mma_commit(ofull);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ rows (warps 0-3): softmax and partials
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int row = warp * 32 + lane;
    const int hh = row % a.G;
    for (int i = 0; i < nbatch; ++i) {
      const int buf = i & 1;
      const uint32_t ph = i & 1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&qfull[buf], (i >> 1) & 1, abort_flag)) ||
          !__all_sync(0xffffffffu, tc::mbar_wait(sfull, ph, abort_flag))) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      const int e = tab[buf * GT_ROWS + row];  // the producer wrote it before arriving on qfull
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&qempty[buf]);  // the table may be rewritten for batch i + 2
      const int t = e >= 0 ? e / (a.Hkv * a.nsel) : 0;
      const int p = t - ck.s0;
      // causal keys of this row in the tile: key c < lim
      const int lim = e < 0 ? 0 : min(min(a.bs, ck.n - ck.kbase), p - ck.kbase + 1);
      uint32_t sr[GT_KEYS];
      __syncwarp();
      tc::tmem_ld32(tmem + lane_base + GF_T_S, sr);
      tc::tmem_ld32(tmem + lane_base + GF_T_S + 32, sr + 32);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(sempty);
      float m = -INFINITY;
#pragma unroll
      for (int c = 0; c < GT_KEYS; ++c)
        if (c < lim) m = fmaxf(m, __uint_as_float(sr[c]) * a.scale_log2);
      float l = 0.f;
      uint32_t pk[GT_KEYS / 2];
#pragma unroll
      for (int c = 0; c < GT_KEYS; c += 2) {
        const float p0 = c < lim ? exp2f(__uint_as_float(sr[c]) * a.scale_log2 - m) : 0.f;
        const float p1 = c + 1 < lim ? exp2f(__uint_as_float(sr[c + 1]) * a.scale_log2 - m) : 0.f;
        l += p0 + p1;
        pk[c / 2] = pack_bf16(p0, p1);
      }
      // P -> TMEM once PV of the previous batch is done with it
      if (i > 0 && !__all_sync(0xffffffffu, tc::mbar_wait(pempty, ph ^ 1u, abort_flag))) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      __syncwarp();
      tc::tmem_st32(tmem + lane_base + GF_T_P, pk);
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(pfull);
      if (!__all_sync(0xffffffffu, tc::mbar_wait(ofull, ph, abort_flag))) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      // partial O / l (bf16: a convex combination of value rows) and its
      // log2-sum-exp (fp32) into the selection slot of this row
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* dst = e >= 0 ? a.part_o + ((int64_t)e * a.G + hh) * a.d : nullptr;
#pragma unroll 1
      for (int cb = 0; cb < a.d / 32; ++cb) {
        uint32_t r[32];
        __syncwarp();
        tc::tmem_ld32(tmem + lane_base + GF_T_O + cb * 32, r);
        tc::tmem_ld_wait();
        if (dst != nullptr) {
#pragma unroll
          for (int k = 0; k < 32; k += 8)
            *reinterpret_cast<uint4*>(dst + cb * 32 + k) =
                make_uint4(pack_bf16(__uint_as_float(r[k]) * inv, __uint_as_float(r[k + 1]) * inv),
                           pack_bf16(__uint_as_float(r[k + 2]) * inv, __uint_as_float(r[k + 3]) * inv),
                           pack_bf16(__uint_as_float(r[k + 4]) * inv, __uint_as_float(r[k + 5]) * inv),
                           pack_bf16(__uint_as_float(r[k + 6]) * inv, __uint_as_float(r[k + 7]) * inv));
        }
      }
      if (e >= 0) a.part_l[(int64_t)e * a.G + hh] = l > 0.f ? m + log2f(l) : -INFINITY;
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(oempty);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && tid == 0) raise_flag(a.flags, TSA_FLAG_TIMEOUT);
  if (warp == 5) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, GF_TMEM);
  }
}

// Merge of the partials: one warp per (query, head), the selected blocks in
// slot order (fixed, so the result is bit-identical across runs).  Lane j holds
// slot j's log-sum-exp (32 slots per round) and the weights come from warp
// reductions.  Up to 32 selected blocks, the partial rows are loaded together
// with the log-sum-exps (one memory latency per row); more blocks take two
// passes, the partial rows eight slots at a time.
__global__ void __launch_bounds__(256, 2) gqa_combine_kernel(const __grid_constant__ GqaTcArgs a) {
  const int64_t rowid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (rowid >= (int64_t)a.T * a.Hq) return;
  const int t = static_cast<int>(rowid / a.Hq), h = static_cast<int>(rowid % a.Hq);
  const int g = h / a.G, hh = h % a.G;
  const int s = seq_of(a.st, t);
  const int p = t - a.st.cu[s];
  const int n = a.st.cu[s + 1] - a.st.cu[s];
  const int32_t* brow = a.blk + ((int64_t)t * a.Hkv + g) * a.nsel;
  const int64_t e0 = ((int64_t)t * a.Hkv + g) * a.nsel;
  const int nv = a.d / 4;  // four channels per lane
  float M = -INFINITY, W = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto accumulate = [&](const uint2& r, float w) {
    const float2 o01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 o23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    acc.x = fmaf(w, o01.x, acc.x);
    acc.y = fmaf(w, o01.y, acc.y);
    acc.z = fmaf(w, o23.x, acc.z);
    acc.w = fmaf(w, o23.y, acc.w);
  };
  if (a.nsel <= 32) {
    // one round: the block ids, the log-sum-exps and every slot's partial row
    // are loaded together (one memory latency); a slot without a partial
    // (invalid or not causal) gets weight 0 and its row, whatever it holds, is
    // never summed
    uint2 raw[32];
#pragma unroll
    for (int k = 0; k < 32; ++k)
      raw[k] = (k < a.nsel && lane < nv)
                   ? __ldg(reinterpret_cast<const uint2*>(a.part_o + ((e0 + k) * a.G + hh) * a.d) + lane)
                   : make_uint2(0u, 0u);
    const int b = lane < a.nsel ? __ldg(brow + lane) : -1;
    const float lj = lane < a.nsel ? __ldg(a.part_l + (e0 + lane) * a.G + hh) : -INFINITY;
    const bool ok = b >= 0 && (int64_t)b * a.bs < n && (int64_t)b * a.bs <= p;
    M = warp_max(ok ? lj : -INFINITY);
    if (M != -INFINITY) {
      const float wl = ok ? exp2f(lj - M) : 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float w = __shfl_sync(0xffffffffu, wl, k);
        if (w != 0.f) accumulate(raw[k], w);
      }
      W = warp_sum(wl);
    }
  } else {
    // pass 1: the maximum log-sum-exp over the valid slots
    for (int j0 = 0; j0 < a.nsel; j0 += 32) {
      const int j = j0 + lane;
      const int b = j < a.nsel ? __ldg(brow + j) : -1;
      const bool ok = b >= 0 && (int64_t)b * a.bs < n && (int64_t)b * a.bs <= p;
      M = fmaxf(M, ok ? __ldg(a.part_l + (e0 + j) * a.G + hh) : -INFINITY);
    }
    M = warp_max(M);
    if (M != -INFINITY) {
      for (int j0 = 0; j0 < a.nsel; j0 += 32) {
        const int j = j0 + lane;
        const int b = j < a.nsel ? __ldg(brow + j) : -1;
        const bool ok = b >= 0 && (int64_t)b * a.bs < n && (int64_t)b * a.bs <= p;
        const float wl = ok ? exp2f(__ldg(a.part_l + (e0 + j) * a.G + hh) - M) : 0.f;
        W += wl;
        const int cnt = min(32, a.nsel - j0);
        for (int k0 = 0; k0 < cnt; k0 += 8) {
          uint2 raw[8];
          float wk[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {  // slot order within a round: k0 + u
            const int k = k0 + u;
            wk[u] = __shfl_sync(0xffffffffu, wl, k & 31);
            raw[u] = make_uint2(0u, 0u);
            if (k < cnt && wk[u] != 0.f && lane < nv)
              raw[u] = __ldg(reinterpret_cast<const uint2*>(a.part_o + ((e0 + j0 + k) * a.G + hh) * a.d) + lane);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (k0 + u < cnt && wk[u] != 0.f) accumulate(raw[u], wk[u]);
        }
      }
      W = warp_sum(W);
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  if (lane < nv) {
    __nv_bfloat16* orow = a.out + ((int64_t)t * a.Hq + h) * a.d + 4 * lane;
    *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16(acc.x * inv, acc.y * inv), pack_bf16(acc.z * inv, acc.w * inv));
  }
  if (lane == 0) a.lse[(int64_t)t * a.Hq + h] = W > 0.f ? (M + log2f(W)) * kLn2 : -INFINITY;
}

// ---------------------------------------------------------------- host side

namespace {

// Inversion of the selections into per-(block, group) lists, shared by the
// forward and the backward.
cudaError_t gt_invert(const GqaTcArgs& a, int chunk, cudaStream_t stream) {
  const int nB = a.nseg * a.nblk * a.Hkv;  // lists
  const int64_t entries = static_cast<int64_t>(a.T) * a.Hkv * a.nsel;
  cudaError_t e;
  const unsigned ig = static_cast<unsigned>(std::min<int64_t>((entries + 255) / 256, 4096));
  if ((e = cudaMemsetAsync(a.cnt, 0, sizeof(int) * nB, stream)) != cudaSuccess) return e;
  gqa_tc_inv_kernel<false><<<ig, 256, 0, stream>>>(a);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gqa_tc_scan_kernel<<<1, 1024, 0, stream>>>(a, nB, chunk);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gqa_tc_inv_kernel<true><<<ig, 256, 0, stream>>>(a);
  note_launch();
  return cudaGetLastError();
}

constexpr int GT_FWD_CHUNK = 256;  // list entries (queries) per forward CTA

}  // namespace

cudaError_t launch_gqa_fwd_tc(const GqaTcArgs& a, cudaStream_t stream) {
  const int nB = a.nseg * a.nblk * a.Hkv;  // lists
  const int64_t entries = static_cast<int64_t>(a.T) * a.Hkv * a.nsel;
  if (entries <= 0 || nB <= 0) return cudaSuccess;
  cudaError_t e = gt_invert(a, GT_FWD_CHUNK, stream);
  if (e != cudaSuccess) return e;
  CUtensorMap tq, tk, tv;
  if ((e = make_tmap_bf16_2d(&tq, a.q, (uint64_t)a.T * a.Hq, a.d, 1, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16_2d(&tk, a.k, (uint64_t)a.T * a.Hkv, a.d, 1, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16_2d(&tv, a.v, (uint64_t)a.T * a.Hkv, a.d, 1, 64)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(gqa_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GF_SMEM)) !=
      cudaSuccess)
    return e;
  // chunks: at most one partial chunk per list plus entries / chunk full ones
  const int64_t grid = nB + (entries + GT_FWD_CHUNK - 1) / GT_FWD_CHUNK;
  gqa_fwd_tc_kernel<<<static_cast<unsigned>(grid), GT_THREADS, GF_SMEM, stream>>>(tq, tk, tv, a, GT_FWD_CHUNK);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(a.T) * a.Hq;
  gqa_combine_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(a);
  note_launch();
  return cudaGetLastError();
}

// ---------------------------------------------------------------- backward

namespace {

// K, V, two Q and two dO buffers, P, dS, two row tables
constexpr int GB_OFF_K = 0;
constexpr int GB_OFF_V = GB_OFF_K + GT_KT;
constexpr int GB_OFF_Q = GB_OFF_V + GT_KT;
constexpr int GB_OFF_DO = GB_OFF_Q + 2 * GT_QT;
constexpr int GB_OFF_P = GB_OFF_DO + 2 * GT_QT;
constexpr int GB_OFF_DS = GB_OFF_P + GT_PT;
constexpr int GB_OFF_TAB = GB_OFF_DS + GT_PT;          // int [2][128]
constexpr int GB_OFF_BAR = GB_OFF_TAB + 2 * GT_ROWS * 4;
constexpr int GB_SMEM = 1024 + GB_OFF_BAR + 256;
static_assert(GB_SMEM <= 227 * 1024, "GQA backward shared memory");
constexpr int GB_THREADS = 480;  // warps 0-7 rows (two per TMEM lane quadrant), 8-11 dQ drains, 12-13 loaders, 14 MMA
constexpr int GB_W_DRAIN = 8, GB_W_LOAD = 12, GB_W_MMA = 14;
constexpr int GB_LOADERS = 64;   // loader threads: one regular and one cp.async arrival each on qfull
// TMEM: S, dP, dV^T, dK^T (accumulated over the chunk), dQ^T double-buffered
constexpr int GB_T_S = 0, GB_T_DP = 64, GB_T_DV = 128, GB_T_DK = 192, GB_T_DQ = 256, GB_TMEM = 512;
constexpr int GT_BWD_CHUNK = 512;  // list entries (queries) per backward CTA

}  // namespace

__global__ void __launch_bounds__(GB_THREADS, 1)
    gqa_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ GqaTcArgs a, int chunk) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t sK = base + GB_OFF_K, sV = base + GB_OFF_V, sQ = base + GB_OFF_Q, sO = base + GB_OFF_DO;
  const uint32_t sP = base + GB_OFF_P, sS = base + GB_OFF_DS;
  int* tab = reinterpret_cast<int*>(gbase + GB_OFF_TAB);  // [2][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + GB_OFF_BAR);
  uint64_t* kvfull = bars;          // [1]
  uint64_t* qfull = bars + 1;       // [2] Q, dO and the row table of a batch landed (loader arrivals)
  uint64_t* qempty = qfull + 2;     // [2] MMAs done with Q / dO, row and drain warps done with the table
  uint64_t* sfull = qempty + 2;     // [1] S and dP ready
  uint64_t* sempty = sfull + 1;     // [1] rows read S and dP (8 warps)
  uint64_t* psfull = sempty + 1;    // [1] rows wrote P and dS (8 warps)
  uint64_t* psempty = psfull + 1;   // [1] MMAs done reading P and dS
  uint64_t* dqfull = psempty + 1;   // [2] dQ^T of a batch complete
  uint64_t* dqempty = dqfull + 2;   // [2] drain warps read it (4 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dqempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  GtChunk ck;
  if (!gt_chunk(a, blockIdx.x, chunk, ck)) return;  // uniform
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qb = GT_ROWS / a.G;
  const int nbatch = (ck.e1 - ck.e0 + qb - 1) / qb;

  if (tid == 0) {
    tc::mbar_init(kvfull, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&qfull[i], 2 * GB_LOADERS);
      tc::mbar_init(&qempty[i], 1 + 8 + 4);  // the MMA commit, the eight row and the four drain warps
      tc::mbar_init(&dqfull[i], 1);
      tc::mbar_init(&dqempty[i], 4);
    }
    tc::mbar_init(sfull, 1);
    tc::mbar_init(sempty, 8);
    tc::mbar_init(psfull, 8);
    tc::mbar_init(psempty, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (a.d == 64) {
    // channels 64..127 of every operand tile are never loaded: zero them once
    for (int i = tid; i < GT_KBOX / 16; i += GB_THREADS) {
      reinterpret_cast<uint4*>(gbase + GB_OFF_K + GT_KBOX)[i] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(gbase + GB_OFF_V + GT_KBOX)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int i = tid; i < GT_QBOX / 16; i += GB_THREADS)
      for (int b = 0; b < 2; ++b) {
        reinterpret_cast<uint4*>(gbase + GB_OFF_Q + b * GT_QT + GT_QBOX)[i] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(gbase + GB_OFF_DO + b * GT_QT + GT_QBOX)[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    tc::fence_proxy_async_smem();
  }
  if (warp == GB_W_MMA) tc::tmem_alloc(tmem_slot, GB_TMEM);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t kv_bytes = (a.d == 128 ? 2 : 1) * 2 * GT_KBOX;

  if (warp == GB_W_LOAD || warp == GB_W_LOAD + 1) {
    // ------------------------------------------------------------ loaders (2 warps)
    // The block's K and V rows by TMA gathers, once per chunk.  Then per batch,
    // loader warp wl owns batch rows 64 wl .. +63: lane l finds the sources of
    // rows 64 wl + 2l and +1 and writes them to the row table, and the warp
    // copies the rows' Q and dO by cp.async, 16 lanes per row (two whole rows
    // per instruction; the sources travel by shuffle), each 16-byte chunk
    // straight to its place in the 128-byte-swizzled K-major tile (chunk j of
    // row r at r * 128 + (j ^ (r & 7)) * 16 of its 64-channel box).  Rows
    // without a query are zero-filled.  Each thread arrives on qfull once after
    // its table entries and once (noinc) when its copies have landed.
    const int wl = warp - GB_W_LOAD;
    if (wl == 0) {
      if (lane == 0) {
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
        tc::mbar_arrive_expect_tx(kvfull, kv_bytes);
      }
      __syncwarp();
      gt_gather_kv(sK, &tm_k, kvfull, a, ck, lane);
      gt_gather_kv(sV, &tm_v, kvfull, a, ck, lane);
    }
    const int nch = a.d / 8;  // 16-byte chunks per row: 16 or 8
    const int c16 = lane & 15, h = lane >> 4;
    const int cb = c16 >> 3, jj = c16 & 7;
    const char* qsrc = reinterpret_cast<const char*>(a.q);
    const char* osrc = reinterpret_cast<const char*>(a.dout);
    bool ok = true;
    for (int i = 0; i < nbatch; ++i) {
      const int buf = i & 1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&qempty[buf], ((i >> 1) & 1) ^ 1u, abort_flag))) {
        ok = false;
        break;
      }
      int src[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int row = 64 * wl + 2 * lane + k;
        const int qi = row / a.G, hh = row - qi * a.G;
        const int ei = ck.e0 + i * qb + qi;
        const bool okr = qi < qb && ei < ck.e1;
        const int e = okr ? __ldg(a.list + ei) : -1;
        src[k] = okr ? (e / (a.Hkv * a.nsel)) * a.Hq + ck.g * a.G + hh : -1;
        tab[buf * GT_ROWS + row] = src[k];
      }
      tc::mbar_arrive(&qfull[buf]);  // this thread's table entries
      const uint32_t qdst = sQ + buf * GT_QT, odst = sO + buf * GT_QT;
#pragma unroll 4
      for (int m = 0; m < 32; ++m) {
        const int s0 = __shfl_sync(0xffffffffu, src[0], m), s1 = __shfl_sync(0xffffffffu, src[1], m);
        const int sr = h ? s1 : s0;
        const int row = 64 * wl + 2 * m + h;
        if (c16 < nch) {
          const int64_t off = (int64_t)(sr >= 0 ? sr : 0) * a.d * 2 + c16 * 16;
          const uint32_t o = cb * GT_QBOX + row * 128 + ((jj ^ (row & 7)) << 4);
          cp_async16(qdst + o, qsrc + off, sr >= 0 ? 16u : 0u);
          cp_async16(odst + o, osrc + off, sr >= 0 ? 16u : 0u);
        }
      }
      cp_async_commit();
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&qfull[buf])) : "memory");
    }
    cp_async_wait<0>();  // this thread's copies land before the CTA can exit
    if (!ok) *abort_flag = 1;
    if (wl == 0 && lane == 0) {  // the K / V gathers land before the CTA exits (bounded by time only)
      volatile int keep_waiting = 0;
      (void)tc::mbar_wait(kvfull, 0, &keep_waiting);
    }
  } else if (warp == GB_W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = tc::idesc_bf16_f32(GT_ROWS, GT_KEYS);
      constexpr uint32_t id_kv = tc::idesc_bf16_f32(GT_DP, GT_KEYS) | (1u << 15) | (1u << 16);  // A, B MN-major
      constexpr uint32_t id_q = tc::idesc_bf16_f32(GT_DP, GT_ROWS) | (1u << 15);                // A MN-major
      // S = Q K^T and dP = dO V^T of batch i (K = the head dimension)
      auto issue_s = [&](int i) {
        const int buf = i & 1;
        const uint32_t qt = sQ + buf * GT_QT, ot = sO + buf * GT_QT;
        tc::fence_proxy_async_smem();  // the rows arrived by cp.async (generic proxy); the MMAs read them
#pragma unroll
        for (int ks = 0; ks < GT_DP / 16; ++ks) {
          const int c = ks >> 2, kk = ks & 3;
          tc::mma_bf16_ss(tmem + GB_T_S, tc::desc_sw128(qt + c * GT_QBOX + kk * 32),
                          tc::desc_sw128(sK + c * GT_KBOX + kk * 32), id_s, ks > 0 ? 1u : 0u);
          tc::mma_bf16_ss(tmem + GB_T_DP, tc::desc_sw128(ot + c * GT_QBOX + kk * 32),
                          tc::desc_sw128(sV + c * GT_KBOX + kk * 32), id_s, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(sfull);
      };
      // batch i's rows landed and the rows have read S / dP of batch i - 1
      auto s_ready = [&](int i, bool block) {
        const int buf = i & 1;
        if (block)
          return tc::mbar_wait(&qfull[buf], (i >> 1) & 1, abort_flag) &&
                 (i < 1 || tc::mbar_wait(sempty, (i - 1) & 1, abort_flag));
        return tc::mbar_try_wait(&qfull[buf], (i >> 1) & 1) && (i < 1 || tc::mbar_try_wait(sempty, (i - 1) & 1));
      };
      bool ok = tc::mbar_wait(kvfull, 0, abort_flag) && (nbatch == 0 || s_ready(0, true));
      if (ok && nbatch > 0) {
        tc::fence_after_sync();
        issue_s(0);
      }
      for (int i = 0; ok && i < nbatch; ++i) {
        const int buf = i & 1;
        // S / dP of the next batch first if the rows have read this one's and
        // its rows are here, so the row warps find it ready
        bool next_done = false;
        if (i + 1 < nbatch && s_ready(i + 1, false)) {
          tc::fence_after_sync();
          issue_s(i + 1);
          next_done = true;
        }
        // the rows' P and dS of this batch, and dQ^T buffer i & 1 drained (batch i - 2)
        if (!tc::mbar_wait(psfull, i & 1, abort_flag) ||
            (i > 1 && !tc::mbar_wait(&dqempty[buf], ((i >> 1) & 1) ^ 1u, abort_flag))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t qt = sQ + buf * GT_QT, ot = sO + buf * GT_QT;
        // dV^T += dO^T P, dK^T += Q^T dS (K = the batch's 128 rows)
#pragma unroll
        for (int ks = 0; ks < GT_ROWS / 16; ++ks) {
          tc::mma_bf16_ss(tmem + GB_T_DV, tc::desc_sw128_mn(ot + ks * 2048, GT_QBOX),
                          tc::desc_sw128_mn(sP + ks * 2048, GT_PT), id_kv, (i > 0 || ks > 0) ? 1u : 0u);
          tc::mma_bf16_ss(tmem + GB_T_DK, tc::desc_sw128_mn(qt + ks * 2048, GT_QBOX),
                          tc::desc_sw128_mn(sS + ks * 2048, GT_PT), id_kv, (i > 0 || ks > 0) ? 1u : 0u);
        }
        tc::mma_commit(&qempty[buf]);
        // dQ^T = K^T dS^T (K = the 64 keys) into buffer i & 1
#pragma unroll
        for (int ks = 0; ks < GT_KEYS / 16; ++ks)
          tc::mma_bf16_ss(tmem + GB_T_DQ + buf * GT_ROWS, tc::desc_sw128_mn(sK + ks * 2048, GT_KBOX),
                          tc::desc_sw128(sS + ks * 32), id_q, ks > 0 ? 1u : 0u);
        tc::mma_commit(psempty);
        tc::mma_commit(&dqfull[buf]);
        if (i + 1 < nbatch && !next_done) {
          if (!s_ready(i + 1, true)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          issue_s(i + 1);
        }
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp < GB_W_DRAIN) {
    // ------------------------------------------------------------ rows (warps 0-7)
    // warp w: TMEM lane quadrant qd = w % 4 (batch rows), keys 32 hf .. +31 of
    // S / dP with hf = w / 4
    const int qd = warp & 3, hf = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const int row = qd * 32 + lane;
    for (int i = 0; i < nbatch; ++i) {
      const int buf = i & 1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&qfull[buf], (i >> 1) & 1, abort_flag)) ||
          !__all_sync(0xffffffffu, tc::mbar_wait(sfull, i & 1, abort_flag))) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      const int qrow = tab[buf * GT_ROWS + row];  // its row t * Hq + h of q / dO, or -1
      const int t = qrow >= 0 ? qrow / a.Hq : 0;
      const int lim = qrow < 0 ? 0 : min(min(a.bs, ck.n - ck.kbase), t - ck.s0 - ck.kbase + 1);
      const float lse2 = qrow >= 0 ? __ldg(a.lse_in + qrow) * kLog2e : 0.f;
      const float dl = qrow >= 0 ? __ldg(a.dlt + qrow) : 0.f;
      uint32_t sr[32], dr[32];
      __syncwarp();
      tc::tmem_ld32(tmem + lane_base + GB_T_S + hf * 32, sr);
      tc::tmem_ld32(tmem + lane_base + GB_T_DP + hf * 32, dr);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(sempty);
      uint32_t pk[16], dk[16];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        const int k0 = hf * 32 + c;
        const float p0 = k0 < lim ? exp2f(__uint_as_float(sr[c]) * a.scale_log2 - lse2) : 0.f;
        const float p1 = k0 + 1 < lim ? exp2f(__uint_as_float(sr[c + 1]) * a.scale_log2 - lse2) : 0.f;
        pk[c / 2] = pack_bf16(p0, p1);
        dk[c / 2] = pack_bf16(a.scale * p0 * (__uint_as_float(dr[c]) - dl),
                              a.scale * p1 * (__uint_as_float(dr[c + 1]) - dl));
      }
      // P and dS into shared memory once the previous batch's MMAs have read them
      if (i > 0 && !__all_sync(0xffffffffu, tc::mbar_wait(psempty, (i - 1) & 1, abort_flag))) {
        *abort_flag = 1;
        break;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        *reinterpret_cast<uint4*>(gbase + GB_OFF_P + sw128(row, hf * 4 + q)) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        *reinterpret_cast<uint4*>(gbase + GB_OFF_DS + sw128(row, hf * 4 + q)) =
            make_uint4(dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
      }
      tc::fence_proxy_async_smem();  // generic writes before the MMAs (async proxy) read them
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(psfull);
        tc::mbar_arrive(&qempty[buf]);  // done with the batch's row table
      }
    }
  } else {
    // ------------------------------------------------------------ dQ drains (warps 8-11)
    // warp 8 + qd: channels 32 qd .. +31 (its TMEM lane quadrant of dQ^T) of all
    // 128 batch rows, 32 rows at a time.  Each 32-row block is turned around in
    // shared memory so that a lane adds four channels of one row with a 16-byte
    // reduction: 8 lanes cover the warp's 128-byte line of a row, 4 rows per
    // instruction.  The space is this warp's 4 KB of the batch's own Q buffer
    // (its first 64-channel box, which the producer reloads for every batch):
    // every MMA that reads it is complete once dQ^T is, and the producer refills
    // it only after this warp has released the batch.
    const int qd = warp - GB_W_DRAIN;
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const bool live = qd * 32 < a.d;  // d = 64: quadrants 2, 3 hold the zero padding
    for (int i = 0; i < nbatch; ++i) {
      const int buf = i & 1;
      // qfull orders the producer's row-table writes before this warp's reads
      // (the phase cannot move on before this warp releases the batch)
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&qfull[buf], (i >> 1) & 1, abort_flag)) ||
          !__all_sync(0xffffffffu, tc::mbar_wait(&dqfull[buf], (i >> 1) & 1, abort_flag))) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      const int* tb = tab + buf * GT_ROWS;
      float* xb = reinterpret_cast<float*>(gbase + GB_OFF_Q + buf * GT_QT + qd * (32 * 32 * 4));  // [row][channel]
#pragma unroll 1
      for (int cb = 0; cb < GT_ROWS / 32; ++cb) {
        uint32_t r[32];
        __syncwarp();
        tc::tmem_ld32(tmem + lane_base + GB_T_DQ + buf * GT_ROWS + cb * 32, r);
        tc::tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int k = 0; k < 32; ++k) xb[k * 32 + lane] = __uint_as_float(r[k]);
          __syncwarp();
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const int k = 4 * m + (lane >> 3);
            const int qr = tb[cb * 32 + k];
            const float4 v = *reinterpret_cast<const float4*>(xb + k * 32 + 4 * (lane & 7));
            if (qr >= 0) red_add_v4(a.dq_acc + (int64_t)qr * a.d + qd * 32 + 4 * (lane & 7), v.x, v.y, v.z, v.w);
          }
          __syncwarp();  // read before the next block overwrites it
        }
      }
      tc::fence_proxy_async_smem();  // the transpose writes before the producer's next TMA into the buffer
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&dqempty[buf]);
        tc::mbar_arrive(&qempty[buf]);  // the buffers and the row table may be rewritten for batch i + 2
      }
    }
    // ---- this chunk's dK, dV of the block's keys: channels 32 qd .. +31, all 64 keys
    if (!*abort_flag && nbatch > 0) {
      // the last dQ^T commit follows every MMA of the chunk
      const int last = nbatch - 1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&dqfull[last & 1], (last >> 1) & 1, abort_flag))) {
        *abort_flag = 1;
      } else {
        tc::fence_after_sync();
        const int ch = qd * 32 + lane;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t rk[32], rv[32];
          __syncwarp();
          tc::tmem_ld32(tmem + lane_base + GB_T_DK + hf * 32, rk);
          tc::tmem_ld32(tmem + lane_base + GB_T_DV + hf * 32, rv);
          tc::tmem_ld_wait();
          if (ch < a.d) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int key = hf * 32 + k;
              const int kp = ck.kbase + key;
              if (key < a.bs && kp < ck.n) {
                const int64_t o = ((int64_t)(ck.s0 + kp) * a.Hkv + ck.g) * a.d + ch;
                red_f32(a.dk_acc + o, __uint_as_float(rk[k]));
                red_f32(a.dv_acc + o, __uint_as_float(rv[k]));
              }
            }
          }
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && tid == 0) raise_flag(a.flags, TSA_FLAG_TIMEOUT);
  if (warp == GB_W_MMA) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, GB_TMEM);
  }
}

cudaError_t launch_gqa_bwd_tc(const GqaTcArgs& a, cudaStream_t stream) {
  const int nB = a.nseg * a.nblk * a.Hkv;  // lists
  const int64_t entries = static_cast<int64_t>(a.T) * a.Hkv * a.nsel;
  if (entries <= 0 || nB <= 0) return cudaSuccess;
  cudaError_t e = gt_invert(a, GT_BWD_CHUNK, stream);
  if (e != cudaSuccess) return e;
  CUtensorMap tk, tv;
  if ((e = make_tmap_bf16_2d(&tk, a.k, (uint64_t)a.T * a.Hkv, a.d, 1, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16_2d(&tv, a.v, (uint64_t)a.T * a.Hkv, a.d, 1, 64)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(gqa_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GB_SMEM)) !=
      cudaSuccess)
    return e;
  const int64_t grid = nB + (entries + GT_BWD_CHUNK - 1) / GT_BWD_CHUNK;
  const unsigned nblocks = static_cast<unsigned>(grid);
  gqa_bwd_tc_kernel<<<nblocks, GB_THREADS, GB_SMEM, stream>>>(tk, tv, a, GT_BWD_CHUNK);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tsa
