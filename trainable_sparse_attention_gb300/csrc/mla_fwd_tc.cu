// Sparse MLA forward for H = 128 heads on tcgen05 (TMEM accumulators, 2-CTA
// cluster, TMA gathers into swizzled tiles).  Tensor-parallel head counts
// H < 128 (64 for a two-way split of 128 heads) run on the same kernel with the
// heads padded to the MMA's 128 rows: rows h >= H get a zero q row and write
// nothing (Megatron-LM PR #7617 backport commit message: the FlashMLA route pads
// TP-local heads to the kernel's head tile).
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
// slice of the selected rows, and computes the partial logits Q_r K_r^T over
// it.  The two 128 x 32 partials are swapped through distributed shared memory
// and added; fp32 addition is commutative, so both CTAs hold bit-identical
// logits and take identical softmax decisions.  No MMA is repeated and every
// selected row is read once.
//
// Per CTA, TMEM columns [0,256) = O slice, [256,320) = two 32-key S buffers,
// [320, 320 + 32 kb) = the q slice (the A operand of QK^T, loaded once),
// [480,512) = two P buffers (the A operand of PV, written by the softmax with
// tcgen05.st: no shared memory and no proxy fence between softmax and PV).
// Warps 0-3: softmax, one warp per TMEM lane quadrant (thread = head = TMEM
// lane) owning all 32 key columns of a tile, so a row's maximum and sum stay
// in one thread (two warps per quadrant, agreeing on each tile's maximum
// through shared memory, were slower); each rescales and writes its row of
// the O slice.  Warp 4: TMEM owner and QK^T issuer of the even tiles, warp 11
// of the odd ones; warp 5: PV issuer (separate issuing threads, so that QK^T
// waiting for a gather never delays a ready PV); warps 6-9: TMA gathers
// (tile::gather4, issued from several lanes at once) of the selected rows into
// a 6-stage ring of 32-key tiles; warp 10: sender, one bulk copy per tile of
// the staged partial logits into the peer's exchange buffer (per-thread stores
// into the peer's shared memory held up the softmax warps' next shared-memory
// accesses by ~0.5 us per tile).
//
// The softmax is software-pipelined: a tile's partial logits are staged for
// the peer before the peer's half of the previous tile is awaited, so the
// exchange (a bulk copy lands ~0.6 us after its issue) overlaps a whole
// normalisation; four exchange buffers keep the peer's sends ordered by the
// exchange itself (the peer stages tile j only after it received this CTA's
// tile j - 2, staged after this CTA read buffer j % 4 for tile j - 4).  P is
// double-buffered so PV(j) never waits for the softmax of tile j+1.  The
// running max is rescaled lazily (only when it grows by more than 2^8), so the
// O slice in TMEM is rarely touched.  Every wait is bounded; a timeout raises
// TSA_FLAG_TIMEOUT and both CTAs wind down.
#include "kernels.cuh"
#include "tc.cuh"

namespace tsa {

cudaError_t make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                              uint32_t box_cols);

namespace {

constexpr int MT_H = 128;        // heads = MMA M
constexpr int MT_N = 32;         // keys per tile
constexpr int MT_STAGES = 6;     // even: tile j's stage is used only by tiles of j's parity
constexpr int MT_SOFTMAX = 4;    // softmax warps, one per TMEM lane quadrant
constexpr int MT_W_QK = 4;       // QK^T issuer of the even tiles and TMEM owner
constexpr int MT_W_PV = 5;       // PV issuer
constexpr int MT_W_PROD = 6;     // first of the four gather producer warps
constexpr int MT_W_SEND = 10;    // sender of the staged partial logits
constexpr int MT_W_QK2 = 11;     // QK^T issuer of the odd tiles (another SM sub-partition than warp 4)
constexpr int MT_THREADS = 384;
constexpr int MT_DV = 512;
constexpr int MT_OCOLS = 256;    // value channels per CTA (TMEM columns [0, 256))
constexpr int MT_SCOL = 256;     // TMEM column of the two S buffers
constexpr int MT_QCOL = 320;     // TMEM column of the q slice (up to 160 columns)
constexpr int MT_PCOL = 480;     // TMEM column of the two P buffers (32 keys of bf16 pairs = 16 columns each)
constexpr int MT_XBUF = 4;       // exchange buffers: the peer's half of tile j lands in buffer j % 4
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct MtLayout {
  static constexpr int KB0 = 4;                      // CTA 0: channels [0, 256)
  static constexpr int KB1 = (D - 256) / 64;         // CTA 1: channels [256, D)
  static constexpr int KBMAX = KB1 > KB0 ? KB1 : KB0;
  static constexpr int KV_BLOCK = MT_N * 128;        // one 64-channel column block of a tile
  static constexpr int KV_STAGE = KBMAX * KV_BLOCK;
  static constexpr int X_BYTES = MT_H * MT_N * 4;    // one exchange buffer
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_X = OFF_KV + MT_STAGES * KV_STAGE;
  static constexpr int OFF_SB = OFF_X + MT_XBUF * X_BYTES;  // two staging buffers of this CTA's partials (same layout as X)
  static constexpr int OFF_BAR = OFF_SB + 2 * X_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 512;
  static_assert(MT_QCOL + 32 * KBMAX <= MT_PCOL && MT_PCOL + 2 * 16 <= 512, "TMEM columns");
  static_assert(MT_STAGES % 2 == 0, "each QK^T issuer owns the stages of its tiles");
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace

template <int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MT_THREADS, 1)
    mla_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ MlaFwdArgs a) {
  using L = MtLayout<D>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t sKV = base + L::OFF_KV;
  // [4][128][32] partial logits written by the peer; chunk q (4 floats) of row h
  // sits at chunk q ^ (h & 7), so the 16-byte stores and loads of a warp spread
  // over all banks
  float* X = reinterpret_cast<float*>(gbase + L::OFF_X);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + L::OFF_BAR);
  uint64_t* qready = bars;                            // q slice stored into TMEM (8 warps)
  uint64_t* kv_full = bars + 1;                       // [STAGES]
  uint64_t* kv_empty = kv_full + MT_STAGES;           // [STAGES]
  uint64_t* s_full = kv_empty + MT_STAGES;            // [2]
  uint64_t* s_empty = s_full + 2;                     // [2] (one arrival per softmax warp)
  uint64_t* p_full = s_empty + 2;                     // [2] (one arrival per softmax warp)
  uint64_t* p_empty = p_full + 2;                     // [2] (PV of that buffer completed)
  uint64_t* xfull = p_empty + 2;                      // [4] the peer's half of tile j landed in my X[j % 4]
  uint64_t* sb_full = xfull + MT_XBUF;                // [2] staging buffer written (one arrival per softmax warp)
  uint64_t* sb_empty = sb_full + 2;                   // [2] bulk copy of the staging buffer has read it
  uint64_t* mask_full = sb_empty + 2;                 // [STAGES] valid-slot bits of the stage written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mask_full + MT_STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* masks = tmem_slot + 2;                    // [STAGES] valid-slot bits of each staged tile

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
    tc::mbar_init(qready, MT_SOFTMAX);
    for (int i = 0; i < MT_STAGES; ++i) {
      tc::mbar_init(&kv_full[i], 4);  // one expect-tx arrival per producer warp; its gathers complete the bytes
      tc::mbar_init(&kv_empty[i], 1);
      tc::mbar_init(&mask_full[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&s_empty[i], MT_SOFTMAX);
      tc::mbar_init(&p_full[i], MT_SOFTMAX);
      tc::mbar_init(&p_empty[i], 1);
    }
    for (int i = 0; i < MT_XBUF; ++i) tc::mbar_init(&xfull[i], 1);  // own expect_tx arrival + the peer's bulk copy
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sb_full[i], MT_SOFTMAX);
      tc::mbar_init(&sb_empty[i], 1);
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
    for (int i = 0; i < MT_XBUF; ++i) tc::mbar_arrive_expect_tx(&xfull[i], L::X_BYTES);  // tiles 0 .. 3
  }
  if (warp == MT_W_QK) tc::tmem_alloc(tmem_slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  __syncwarp();
  tc::cluster_sync();  // the peer's barriers exist before any remote arrival
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp >= MT_W_PROD && warp < MT_W_PROD + 4) {
    // ------------------------------------------------------------ gather producers (4 warps)
    // Warp w fetches rows 8w .. 8w+7 of each 32-row tile with TMA gathers of
    // 4 rows x one 64-channel block (tile::gather4, 128-byte swizzle, the
    // K-major layout the MMA reads): lane l < 2 kb issues the gather of row
    // group l / kb and channel block l % kb, so the warp's 8 or 10 gathers are
    // in flight together and no copy goes through the load/store pipe.  A slot
    // that is -1 (or outside its sequence) fetches the sequence's first row
    // instead; the softmax masks it (P = 0), so nothing of it reaches the
    // output.  The slot indices of the next tile are loaded one tile ahead
    // (lane r < 8 holds row 8w + r).
    const int w8 = (warp - MT_W_PROD) * 8;
    bool ok = true;
    int issued = 0;  // tiles whose gathers this warp has issued
    int id_next = (lane < 8 && w8 + lane < a.topk) ? __ldg(idx_row + w8 + lane) : -1;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % MT_STAGES;
      const int id_mine = id_next;
      const int slot_next = (j + 1) * MT_N + w8 + lane;
      id_next = (lane < 8 && slot_next < a.topk) ? __ldg(idx_row + slot_next) : -1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&kv_empty[st], ((j / MT_STAGES) & 1) ^ 1u, abort_flag))) {
        ok = false;
        break;
      }
      if (lane < 8 && id_mine >= n) raise_flag(a.flags, TSA_FLAG_INDEX_RANGE);
      const bool valid = id_mine >= 0 && id_mine < n;
      const int row_mine = s0 + (valid ? id_mine : 0);
      // this warp's bytes (8 rows x kb blocks of 128 bytes) are expected before its gathers are issued
      if (lane == 0) tc::mbar_arrive_expect_tx(&kv_full[st], kb * 8 * 128);
      __syncwarp();
      const int grp = lane / kb, c = lane - grp * kb;  // row group (4 rows) and channel block of this lane
      const int r0 = __shfl_sync(0xffffffffu, row_mine, (4 * grp) & 31);
      const int r1 = __shfl_sync(0xffffffffu, row_mine, (4 * grp + 1) & 31);
      const int r2 = __shfl_sync(0xffffffffu, row_mine, (4 * grp + 2) & 31);
      const int r3 = __shfl_sync(0xffffffffu, row_mine, (4 * grp + 3) & 31);
      if (lane < 2 * kb)
        tc::tma_gather4(sKV + st * L::KV_STAGE + c * L::KV_BLOCK + (w8 + 4 * grp) * 128, &tm_kv, &kv_full[st],
                        ch0 + c * 64, r0, r1, r2, r3);
      issued = j + 1;
      // valid-slot bits of this warp's 8 rows: byte w of the stage's mask word
      const uint32_t bal = __ballot_sync(0xffffffffu, lane < 8 && valid);
      if (lane == 0) {
        reinterpret_cast<volatile unsigned char*>(&masks[st])[warp - MT_W_PROD] = static_cast<unsigned char>(bal & 0xffu);
        tc::mbar_arrive(&mask_full[st]);
      }
    }
    if (!ok) *abort_flag = 1;
    // the gathers still in flight land before the CTA can exit (bounded by
    // time only, so this also runs after an abort)
    volatile int keep_waiting = 0;
    for (int g = issued > MT_STAGES ? issued - MT_STAGES : 0; g < issued; ++g)
      (void)tc::mbar_wait(&kv_full[g % MT_STAGES], (g / MT_STAGES) & 1, &keep_waiting);
  } else if (warp == MT_W_QK || warp == MT_W_QK2) {
    // ------------------------------------------------------------ QK^T issuers (A = q slice in TMEM)
    // One thread keeps only one tcgen05.mma in issue at a time (~50 ns each,
    // whatever N is), so the 16 to 20 MMAs of a tile's QK^T take most of a
    // tile period from one thread; two threads on different SM sub-partitions
    // take the even and the odd tiles (S buffer j & 1), and each tile's MMAs
    // still accumulate in order on one thread.  With an even number of stages
    // each issuer also owns the stages of its tiles.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(MT_H, MT_N);
      bool ok = tc::mbar_wait(qready, 0, abort_flag);
      tc::fence_after_sync();
      // QK^T of each of this issuer's tiles, as soon as its rows have landed and
      // its S buffer is free (the softmax frees one as soon as it has read it).
      for (int j = warp == MT_W_QK ? 0 : 1; ok && j < ntiles; j += 2) {
        const int st = j % MT_STAGES, b = j & 1;
        if (!tc::mbar_wait(&kv_full[st], (j / MT_STAGES) & 1, abort_flag) ||
            !tc::mbar_wait(&s_empty[b], ((j >> 1) & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + MT_SCOL + b * MT_N;
        for (int c = 0; c < kb; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_ts(d, tmem + MT_QCOL + (c * 4 + kk) * 8,
                            tc::desc_sw128(sKV + st * L::KV_STAGE + c * L::KV_BLOCK + kk * 32), idesc_qk,
                            (c | kk) != 0 ? 1u : 0u);
        }
        tc::mma_commit(&s_full[b]);
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == MT_W_SEND) {
    // ------------------------------------------------------------ sender
    // One bulk copy per tile moves this CTA's staged partial logits into the
    // peer's exchange buffer, completing on the peer's barrier; the staging
    // buffer is handed back once the copy has read it.
    if (lane == 0) {
      const uint32_t x_peer = tc::mapa(smem_u32(X), peer);
      const uint32_t peer_xfull = tc::mapa(smem_u32(xfull), peer);
      bool ok = true;
      for (int j = 0; ok && j < ntiles; ++j) {
        const int b = j & 1;
        if (!tc::mbar_wait(&sb_full[b], (j >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const int xb = j & (MT_XBUF - 1);
        tc::bulk_copy_to_peer(x_peer + xb * L::X_BYTES, base + L::OFF_SB + b * L::X_BYTES, L::X_BYTES,
                              peer_xfull + xb * 8);
        tc::bulk_commit();
        tc::bulk_wait_read0();
        tc::mbar_arrive(&sb_empty[b]);
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == MT_W_PV) {
    // ------------------------------------------------------------ PV issuer
    // QK^T(j) completed before the softmax published P(j), so the commits of
    // this thread (kv_empty after PV(j)) also cover every MMA that read stage j.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32_bmn(MT_H, MT_OCOLS);
      bool ok = true;
      for (int j = 0; ok && j < ntiles; ++j) {
        const int pb = j & 1;
        if (!tc::mbar_wait(&p_full[pb], (j >> 1) & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        const int st = j % MT_STAGES;
#pragma unroll
        for (int ks = 0; ks < MT_N / 16; ++ks) {
          const uint64_t bd = tc::desc_sw128_mn(sKV + st * L::KV_STAGE + ks * 2048, L::KV_BLOCK);
          tc::mma_bf16_ts(tmem, tmem + MT_PCOL + pb * 16 + ks * 8, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc::mma_commit(&kv_empty[st]);
        tc::mma_commit(&p_empty[pb]);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-3)
    // Thread h (warp h / 32 reads its TMEM lane quadrant) owns row h: all 32
    // key columns of every tile, so a row's maximum and sum never leave the
    // thread.  Iteration j: fetch tile j's partial logits from TMEM and stage
    // them for the sender, then add the peer's half of tile j-1 to this CTA's
    // and normalise tile j-1.
    const int h = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // q slice row h -> TMEM columns [MT_QCOL, MT_QCOL + 32 kb)
    {
      // heads h >= H (a tensor-parallel slice padded to the MMA's 128 rows) get a
      // zero q row: their logits are 0, and nothing of them is written
      const bool real = h < a.H;
      const uint4* qrow = reinterpret_cast<const uint4*>(a.q + ((int64_t)t * a.H + (real ? h : 0)) * D + ch0);
      for (int c = 0; c < kb; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = real ? __ldg(qrow + c * 8 + i) : make_uint4(0u, 0u, 0u, 0u);
          r[4 * i] = v.x;
          r[4 * i + 1] = v.y;
          r[4 * i + 2] = v.z;
          r[4 * i + 3] = v.w;
        }
        __syncwarp();
        tc::tmem_st32(tmem + lane_base + MT_QCOL + c * 32, r);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(qready);
    }
    float m_use = NEG_INF, l = 0.f;  // running max and row sum
    bool ok = true;
    uint32_t cur[32];  // this CTA's partial logits of tile j - 1 (staged in the previous iteration)
#pragma unroll 2
    for (int j = 0; j <= ntiles; ++j) {
      uint32_t nxt[32];
      if (j < ntiles) {
        // tile j's partial logits, staged for the sender at once (same swizzled
        // layout as the peer's exchange buffer), before this thread waits for
        // the peer's half of tile j - 1: the exchange then takes a tile period
        // per two tiles instead of setting every period.  Staging buffer b is
        // free once the bulk copy of tile j - 2 has read it.
        const int b = j & 1;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&s_full[b], (j >> 1) & 1, abort_flag))) { ok = false; break; }
        tc::fence_after_sync();
        __syncwarp();
        tc::tmem_ld32(tmem + lane_base + MT_SCOL + b * MT_N, nxt);
        tc::tmem_ld_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s_empty[b]);
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&sb_empty[b], ((j >> 1) & 1) ^ 1u, abort_flag))) {
          ok = false;
          break;
        }
        unsigned char* srow = gbase + L::OFF_SB + b * L::X_BYTES + h * (MT_N * 4);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(srow + ((q ^ (h & 7)) << 4)) =
              make_uint4(nxt[4 * q], nxt[4 * q + 1], nxt[4 * q + 2], nxt[4 * q + 3]);
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sb_full[b]);
      }
      // tile j - 1: this CTA's half plus the peer's
      float x2[32];
      if (j > 0) {
        const int jj = j - 1, bb = jj & 1, xb = jj & (MT_XBUF - 1);
        if (!__all_sync(0xffffffffu, tc::mbar_wait_cluster(&xfull[xb], (jj >> 2) & 1, abort_flag))) {
          ok = false;
          break;
        }
        const float4* xr = reinterpret_cast<const float4*>(X + xb * (MT_H * MT_N) + h * MT_N);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 v = xr[q ^ (h & 7)];  // 16-byte chunks of a row are swizzled by the row
          x2[4 * q] = __uint_as_float(cur[4 * q]) + v.x;
          x2[4 * q + 1] = __uint_as_float(cur[4 * q + 1]) + v.y;
          x2[4 * q + 2] = __uint_as_float(cur[4 * q + 2]) + v.z;
          x2[4 * q + 3] = __uint_as_float(cur[4 * q + 3]) + v.w;
        }
        // the next use of X[xb] is tile jj + 4; the peer sends it only after it
        // received this CTA's tile jj + 2, which this CTA stages after reading X[xb]
        if (h == 0 && jj + MT_XBUF < ntiles) tc::mbar_arrive_expect_tx(&xfull[xb], L::X_BYTES);
      }
      if (j > 0) {
        const int jj = j - 1, bb = jj & 1;
        // valid-slot bits published by the producers with this stage
        const int st = jj % MT_STAGES;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&mask_full[st], (jj / MT_STAGES) & 1, abort_flag))) {
          ok = false;
          break;
        }
        // the logits stay unscaled here: the softmax scale (> 0) goes into the
        // exponent's FMA, and rounding is monotone, so the scaled maximum is the
        // maximum of the scaled logits
        const uint32_t mask = masks[st];
        if (mask != 0xffffffffu) {
#pragma unroll
          for (int i = 0; i < 32; ++i) x2[i] = ((mask >> i) & 1u) ? x2[i] : NEG_INF;
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(fmaxf(x2[i], x2[i + 8]), fmaxf(x2[i + 16], x2[i + 24]));
        const float tmax = a.scale_log2 * fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                                fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        float alpha = 1.f;
        const bool resc = tmax > m_use + kRescaleLog2;
        if (resc) {
          alpha = (m_use == NEG_INF) ? 0.f : ex2(m_use - tmax);
          m_use = tmax;
          l *= alpha;
        }
        const float mu = (m_use == NEG_INF) ? 0.f : m_use;
        uint32_t pk[16];
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = ex2(fmaf(x2[i], a.scale_log2, -mu)), p1 = ex2(fmaf(x2[i + 1], a.scale_log2, -mu));
          ps[(i >> 1) & 3] += p0 + p1;
          pk[i / 2] = pack_bf16(p0, p1);
        }
        l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        // P buffer bb is free once PV(jj-2) completed
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&p_empty[bb], ((jj >> 1) & 1) ^ 1u, abort_flag))) {
          ok = false;
          break;
        }
        // a raised running max rescales this row of the O slice, which PV(jj-1) must have finished
        if (jj > 0 && __any_sync(0xffffffffu, resc)) {
          const int pb = (jj - 1) & 1;
          if (!__all_sync(0xffffffffu, tc::mbar_wait(&p_empty[pb], ((jj - 1) >> 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          for (int cb = 0; cb < MT_OCOLS / 32; ++cb) {
            uint32_t o[32];
            const uint32_t oc = tmem + lane_base + cb * 32;
            tc::tmem_ld32(oc, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tc::tmem_st32(oc, o);
          }
          tc::tmem_st_wait();
        }
        // P row h, 32 keys = 16 columns of TMEM P buffer bb (the A operand of PV)
        __syncwarp();
        tc::tmem_st16(tmem + lane_base + MT_PCOL + bb * 16, pk);
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&p_full[bb]);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) cur[i] = nxt[i];
    }
    if (!ok) *abort_flag = 1;
    // epilogue: O row / l -> bf16, lse
    const int lb = (ntiles - 1) & 1;
    const bool last_ok = ok && __all_sync(0xffffffffu, tc::mbar_wait(&p_empty[lb], ((ntiles - 1) >> 1) & 1, abort_flag));
    const bool real_head = h < a.H;
    __nv_bfloat16* orow = a.out + ((int64_t)t * a.H + (real_head ? h : 0)) * MT_DV + ch0;
    if (last_ok) {
      // every lane takes part in the (warp-collective) TMEM loads; only the
      // rows of real heads are stored
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      for (int cb = 0; cb < MT_OCOLS / 32; ++cb) {
        uint32_t o[32];
        __syncwarp();
        tc::tmem_ld32(tmem + lane_base + cb * 32, o);
        tc::tmem_ld_wait();
        uint4* dst = reinterpret_cast<uint4*>(orow + cb * 32);
        if (real_head)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(pack_bf16(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                              pack_bf16(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                              pack_bf16(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                              pack_bf16(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
      }
      if (rank == 0 && real_head) a.lse[(int64_t)t * a.H + h] = l > 0.f ? (m_use + log2f(l)) * kLn2 : NEG_INF;
    } else {
      // wound down after a timeout: zero output row, -inf lse
      *abort_flag = 1;
      if (real_head) {
        for (int c = 0; c < MT_OCOLS; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
        if (rank == 0) a.lse[(int64_t)t * a.H + h] = NEG_INF;
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && tid == 0) raise_flag(a.flags, TSA_FLAG_TIMEOUT);
  __syncwarp();
  tc::cluster_sync();  // the peer no longer writes into this CTA's shared memory
  if (warp == MT_W_QK) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int D>
static cudaError_t launch_tc_t(const MlaFwdArgs& a, cudaStream_t stream) {
  constexpr int smem = MtLayout<D>::SMEM;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  // kv [T, D] bf16, boxes of one row x 64 channels (128 bytes) for tile::gather4
  CUtensorMap tm_kv;
  cudaError_t e = make_tmap_bf16_2d(&tm_kv, a.kv, static_cast<uint64_t>(a.T), D, 1, 64);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mla_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mla_fwd_tc_kernel<D><<<dim3(2 * a.T), MT_THREADS, smem, stream>>>(tm_kv, a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_mla_fwd_tc(const MlaFwdArgs& a, int D, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  return D == 576 ? launch_tc_t<576>(a, stream) : launch_tc_t<512>(a, stream);
}

}  // namespace tsa
