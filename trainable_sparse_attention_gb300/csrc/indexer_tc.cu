// Indexer score on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   I_g[t,s] = score_scale * sum_{h in g} w[t,h] * ReLU(q_I[t,h] . k_I[s]),  s <= t
//
// Megatron-LM issue #7060 "Add trainable QSA sparse attention with a TileLang
// backend" ("Describe the solution you'd like": trainable indexer, ReLU
// scores, streaming bounded-memory runner) and Megatron-LM PR #3674 (fused
// indexer forward + logits cleaning).
//
// A query block is QB = 256 / H_I consecutive queries: their q_I rows form the
// MMA's B operand (N = 256 columns = (query, head)); key tiles of 128 keys (the
// A operand, M = 128) stream through a 2-stage TMA ring.  Two stages keep the
// CTA's shared memory (~139 KB at d_I = 128) small enough for one top-k CTA to
// run beside it on the same SM: the streamed runner selects chunk i while this
// kernel scores chunk i + 1 (with four stages and the two kernels in turn the
// T = 65536 indexer + top-k took 31.3 ms, with two stages side by side 29.9 ms).  Keys sit on TMEM
// lanes, so each epilogue thread owns one key and reduces the heads of a group
// inside its own registers: ReLU, head weight and group sum never leave the
// thread, and only causal scores are written ("cleaned" logits are never
// produced).  The 2 x 256-column TMEM accumulator is double-buffered so the
// epilogue of tile i overlaps the MMAs of tile i+1.
//
// The kernel is persistent: one CTA per SM walks a contiguous share of the
// launch's (query block, causal key tile) pairs, so TMEM allocation and
// pipeline fill are paid once per SM rather than once per short work item.
// When its share moves to the next query block, the new q_I block is loaded
// as soon as the MMAs of the previous one are done, and the head weights go
// to the other half of a double buffer.
//
// Block scores (block_size bs in {16, 32, 64, 128}, the QSA block top-k input)
// come from the same MMAs with a different epilogue: each thread masks its
// key's group scores to -inf where the key is not causal for the query, and the
// maximum over the bs consecutive keys of a block is taken across TMEM lanes --
// inside a warp by recursive halving (at each xor-shuffle step a lane keeps half
// of its values and takes the partner's copy of that half, so 64 values need 62
// shuffles instead of 320), across the 2 or 4 warps of a 64- or 128-key block
// through shared memory, handed over on an mbarrier (bounded wait).  Only the
// block maxima are written: the [T, T] token scores never exist.
//
// Warp roles (320 threads): warps 0-7 epilogue (warp w: TMEM lanes 32 (w % 4)
// .. +31, accumulator columns 128 (w / 4) .. +127, so two warps share each
// sub-partition and hide each other's latencies), warp 8 TMA producer, warp 9
// TMEM allocator + MMA issuer (one elected thread).  Every
// wait is bounded; a timeout raises TSA_FLAG_TIMEOUT and the CTA winds down,
// releasing its TMEM.
#include <algorithm>

#include "kernels.cuh"
#include "tc.cuh"

namespace tsa {

namespace {

constexpr int IT_M = 128;
constexpr int IT_N = 256;
constexpr int IT_STAGES = 2;  // see the header: room for a top-k CTA beside this one
constexpr int IT_THREADS = 320;

template <int DI>
struct ItLayout {
  static constexpr int KB = DI / 64;                    // 128-byte column blocks along d_I
  static constexpr int B_BYTES = KB * IT_N * 128;       // q_I block
  static constexpr int A_BYTES = KB * IT_M * 128;       // one key tile
  static constexpr int XBUF = 2 * 8 * 4 * 32 * 4;        // block epilogue partials [acc][warp][<=4][32 lanes]
  static constexpr int USED = 1024 + B_BYTES + IT_STAGES * A_BYTES + 2 * IT_N * 4 + XBUF + 256;
  // at least 120 KB so that a single CTA (the only TMEM owner) fits on an SM
  static constexpr int SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
};

}  // namespace

// The work of one launch is the list of (query block, key tile) pairs, query
// blocks of QB queries in order and, inside a block, its causal key tiles
// 0 .. nkt(qb)-1.  CTA c of G takes the contiguous share [c W / G, (c+1) W / G)
// of the W pairs; every role walks the same share with this iterator.
struct ItWalk {
  int qb, kt, nkt, tr;  // query block, key tile, key tiles of the block, block changes so far
  bool first, last;     // first / last pair of its query block in this share
};

__device__ __forceinline__ int it_nkt(const IndexerArgs& a, int QB, int qb) {
  const int qn = min(QB, a.nq - qb * QB);
  return (a.p_begin + qb * QB + qn - 1) / IT_M + 1;
}

// (c0, c1) += (a0 * b0, a1 * b1), one packed fp32 FMA (each lane rounds as fmaf).
__device__ __forceinline__ void fma2(float& c0, float& c1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%0, %1};\n"
      " fma.rn.f32x2 rc, ra, rb, rc;\n mov.b64 {%0, %1}, rc;\n}"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Recursive-halving maximum over aligned groups of 2*O lanes (O a power of two):
// N values per lane in, and after log2(min(N, 2*O)) halving steps each lane
// holds N / 2^steps of them, each the maximum over its lane group.  The value
// v[i] of lane L then belongs to the original index i + NF * ((L & (2O-1)) >> R),
// with NF the values left and R = log2(2O) - steps (lanes differing only in
// their R low bits hold the same values).
template <int N, int O>
__device__ __forceinline__ void lane_group_max(float* v, int lane) {
  if constexpr (O >= 1) {
    if constexpr (N >= 2) {
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = up ? v[i] : v[N / 2 + i];
        const float keep = up ? v[N / 2 + i] : v[i];
        v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, O));
      }
      lane_group_max<N / 2, O / 2>(v, lane);
    } else {
      v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], O));
      lane_group_max<1, O / 2>(v, lane);
    }
  }
}

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// Block-maximum epilogue of one warp for one key tile.  vals[NSEG]: the masked
// scores of this lane's key for the warp's NSEG (query, group) segments.  G = the
// lanes of one block inside the warp (16, or 32 for blocks of 32 keys and more).
// Blocks of 64 / 128 keys span 2 / 4 warps: the partner warps leave their
// partials in xbuf and arrive on xbar; the first warp of the block waits
// (bounded) and writes.  Returns false if that wait gave up.
template <int NSEG, int G>
__device__ __forceinline__ bool block_max_epilogue(float* vals, const IndexerArgs& a, int lane, int warp, int qd,
                                                   int ch, int acc, uint32_t aph, int kt, int q0, int qn,
                                                   int p_first, float* xbuf, uint64_t* xbar,
                                                   volatile int* abort_flag) {
  constexpr int LG = ilog2(G), LN = ilog2(NSEG);
  constexpr int HS = LG < LN ? LG : LN;  // halving steps
  constexpr int NF = NSEG >> HS;         // values left per lane
  constexpr int R = LG - HS;
  lane_group_max<NSEG, G / 2>(vals, lane);
  const int sub = (lane & (G - 1)) >> R;
  const bool dup = (lane & ((1 << R) - 1)) != 0;
  const int bs = a.bs;
  int blk;  // local block of this lane's key
  if (bs <= 32) {
    blk = (kt * IT_M + qd * 32 + lane) / bs;
  } else {
    const int bsw = bs / 32;  // warps per block
    const int grp = qd / bsw;
    uint64_t* xb = &xbar[(acc * 2 + ch) * 2 + grp];
    float* mine = xbuf + (acc * 8 + warp) * (4 * 32);
    if (qd % bsw != 0) {  // partner: hand the partials over and go on
#pragma unroll
      for (int i = 0; i < NF; ++i) mine[i * 32 + lane] = vals[i];
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(xb);
      return true;
    }
    if (!__all_sync(0xffffffffu, tc::mbar_wait(xb, aph, abort_flag))) return false;
    for (int p = 1; p < bsw; ++p) {
      const float* other = mine + p * (4 * 32);  // warp + p: same column half, next lane quadrant
#pragma unroll
      for (int i = 0; i < NF; ++i) vals[i] = fmaxf(vals[i], other[i * 32 + lane]);
    }
    blk = (kt * IT_M + qd * 32) / bs;
  }
  if (!dup) {
#pragma unroll
    for (int i = 0; i < NF; ++i) {
      const int sg = ch * NSEG + i + NF * sub;  // (query, group) segment of the block's half
      const int qq = sg / a.groups, gg = sg % a.groups;
      if (qq < qn && blk * bs <= p_first + qq)
        a.out[((int64_t)(q0 + qq) * a.groups + gg) * a.width + blk] = vals[i];
    }
  }
  return true;
}

template <int DI, int HG, bool BLK>
__global__ void __launch_bounds__(IT_THREADS, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ IndexerArgs a, int total) {
  using L = ItLayout<DI>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t sB = base;
  const uint32_t sA = base + L::B_BYTES;
  float* Ws = reinterpret_cast<float*>(gbase + L::B_BYTES + IT_STAGES * L::A_BYTES);  // [2][IT_N]
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(Ws + 2 * IT_N) + L::XBUF);
  uint64_t* full = bars;                       // [IT_STAGES] key tile landed
  uint64_t* empty = bars + IT_STAGES;          // [IT_STAGES]
  uint64_t* bfull = empty + IT_STAGES;         // [1] q_I block landed (one phase per block change)
  uint64_t* bempty = bfull + 1;                // [1] MMAs of the previous block done
  uint64_t* accf = bempty + 1;                 // [2]
  uint64_t* acce = accf + 2;                   // [2]
  uint64_t* wsfull = acce + 2;                 // [2] head weights of a block written (32 lanes)
  uint64_t* wsempty = wsfull + 2;              // [2] epilogue done with a weight buffer (8 warps)
  uint64_t* xbar = wsempty + 2;                // [2 acc][2 halves][2 blocks] block partials handed over
  float* xbuf = reinterpret_cast<float*>(gbase + L::B_BYTES + IT_STAGES * L::A_BYTES + 2 * IT_N * 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int H_I = a.H_I;
  const int QB = IT_N / H_I;
  const int nqb = (a.nq + QB - 1) / QB;
  const int w0 = static_cast<int>((static_cast<int64_t>(total) * blockIdx.x) / gridDim.x);
  const int w1 = static_cast<int>((static_cast<int64_t>(total) * (blockIdx.x + 1)) / gridDim.x);
  const int nitems = w1 - w0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // producer lane: key tiles issued, and the walk index of the last q_I block issued (-1: none)
  int a_issued = 0, b_last_tr = -1;
  if (nitems <= 0) return;  // uniform

  // start of the share: (qb, kt) of pair w0
  ItWalk start;
  {
    int qb = 0, acc = 0, nk = it_nkt(a, QB, 0);
    while (qb + 1 < nqb && acc + nk <= w0) {
      acc += nk;
      ++qb;
      nk = it_nkt(a, QB, qb);
    }
    start.qb = qb;
    start.kt = w0 - acc;
    start.nkt = nk;
    start.tr = 0;
    start.first = true;
    start.last = (start.kt + 1 == nk) || nitems == 1;
  }
  auto advance = [&](ItWalk& w, int i) {  // w describes item i; move to item i+1
    if (++w.kt == w.nkt) {
      ++w.qb;
      w.kt = 0;
      w.nkt = it_nkt(a, QB, w.qb);
      ++w.tr;
      w.first = true;
    } else {
      w.first = false;
    }
    w.last = (w.kt + 1 == w.nkt) || (i + 2 == nitems);
  };

  if (tid == 0) {
    for (int i = 0; i < IT_STAGES; ++i) { tc::mbar_init(&full[i], 1); tc::mbar_init(&empty[i], 1); }
    tc::mbar_init(bfull, 1);
    tc::mbar_init(bempty, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&accf[i], 1);
      tc::mbar_init(&acce[i], 8);
      tc::mbar_init(&wsfull[i], 32);
      tc::mbar_init(&wsempty[i], 8);
    }
    // partner warps of a block: 1 (64-key blocks) or 3 (128-key blocks)
    for (int i = 0; i < 8; ++i) tc::mbar_init(&xbar[i], a.bs >= 64 ? a.bs / 32 - 1 : 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 9) tc::tmem_alloc(tmem_slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer: head weights (all lanes), TMA (lane 0)
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
    }
    bool ok = true;
    ItWalk w = start;
    for (int it = 0; ok && it < nitems; ++it) {
      if (w.first) {
        const int q0 = w.qb * QB, qn = min(QB, a.nq - q0);
        const int p_first = a.p_begin + q0;
        // head weights of this block (buffer tr & 1, free once the block two changes back is done)
        const int wb = w.tr & 1;
        if (w.tr >= 2 && !__all_sync(0xffffffffu, tc::mbar_wait(&wsempty[wb], ((w.tr - 2) >> 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        for (int c = lane; c < IT_N; c += 32) {
          const int qq = c / H_I, h = c % H_I;
          Ws[wb * IT_N + c] = (qq < qn) ? a.w[(int64_t)(a.seq_start + p_first + qq) * H_I + h] : 0.f;
        }
        tc::mbar_arrive(&wsfull[wb]);
        if (lane == 0) {
          // q_I block (B operand) once the MMAs of the previous block are done
          if (w.tr >= 1 && !tc::mbar_wait(bempty, (w.tr - 1) & 1, abort_flag)) ok = false;
          if (ok) {
            tc::mbar_arrive_expect_tx(bfull, L::B_BYTES);
            for (int c = 0; c < L::KB; ++c)
              tc::tma_load_2d(sB + c * (IT_N * 128), &tm_q, bfull, c * 64, (a.seq_start + p_first) * H_I);
            b_last_tr = w.tr;
          }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      if (lane == 0) {
        const int st = it % IT_STAGES;
        const uint32_t ph = (it / IT_STAGES) & 1;
        if (!tc::mbar_wait(&empty[st], ph ^ 1u, abort_flag)) {
          ok = false;
        } else {
          tc::mbar_arrive_expect_tx(&full[st], L::A_BYTES);
          const int row = a.seq_start + w.kt * IT_M;
          for (int c = 0; c < L::KB; ++c)
            tc::tma_load_2d(sA + st * L::A_BYTES + c * (IT_M * 128), &tm_k, &full[st], c * 64, row);
          a_issued = it + 1;
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      advance(w, it);
    }
    if (!ok) *abort_flag = 1;
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(IT_M, IT_N);
      bool ok = true;
      ItWalk w = start;
      for (int it = 0; ok && it < nitems; ++it) {
        const int st = it % IT_STAGES;
        const uint32_t ph = (it / IT_STAGES) & 1;
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if ((w.first && !tc::mbar_wait(bfull, w.tr & 1, abort_flag)) || !tc::mbar_wait(&full[st], ph, abort_flag) ||
            !tc::mbar_wait(&acce[acc], aph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + acc * IT_N;
#pragma unroll
        for (int ks = 0; ks < DI / 16; ++ks) {
          const int c = ks >> 2, kk = ks & 3;
          const uint64_t ad = tc::desc_sw128(sA + st * L::A_BYTES + c * (IT_M * 128) + kk * 32);
          const uint64_t bd = tc::desc_sw128(sB + c * (IT_N * 128) + kk * 32);
          tc::mma_bf16_ss(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(&empty[st]);
        tc::mma_commit(&accf[acc]);
        if (w.last) tc::mma_commit(bempty);  // the q_I block may be replaced once these MMAs are done
        advance(w, it);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-7)
    const int qd = warp & 3, ch = warp >> 2;  // lane quadrant, column half
    const int key_in_tile = qd * 32 + lane;
    ItWalk w = start;
    for (int it = 0; it < nitems; ++it) {
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      const int wb = w.tr & 1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&accf[acc], aph, abort_flag)) ||
          (w.first && !__all_sync(0xffffffffu, tc::mbar_wait(&wsfull[wb], (w.tr >> 1) & 1, abort_flag)))) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      const int q0 = w.qb * QB, qn = min(QB, a.nq - q0);
      const int p_first = a.p_begin + q0;
      const float4* W4 = reinterpret_cast<const float4*>(Ws + wb * IT_N + ch * (IT_N / 2));  // 16-byte aligned
      const uint32_t taddr = tmem + (static_cast<uint32_t>(qd * 32) << 16) + acc * IT_N + ch * (IT_N / 2);
      const int s = w.kt * IT_M + key_in_tile;
      // four partial sums of the current (query, group) segment break the FMA
      // dependency chain; the TMEM load of block cb+1 is in flight while block
      // cb is reduced; the head weights come four at a time
      float run[4] = {0.f, 0.f, 0.f, 0.f};
      constexpr int NSEG = (IT_N / 2) / HG;  // (query, group) segments of this warp's column half
      float vals[BLK ? NSEG : 1];
      uint32_t rbuf[2][32];
      constexpr int NCB = IT_N / 64;  // 32-column blocks of this warp's half
      __syncwarp();
      tc::tmem_ld32(taddr, rbuf[0]);
#pragma unroll
      for (int cb = 0; cb < NCB; ++cb) {
        uint32_t* r = rbuf[cb & 1];
        tc::tmem_ld_wait();
        tc::reg_dep32(r);
        if (cb + 1 < NCB) {
          __syncwarp();  // converged for the .sync.aligned load
          tc::tmem_ld32(taddr + (cb + 1) * 32, rbuf[(cb + 1) & 1]);
        }
        float4 wv;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if ((j & 3) == 0) wv = W4[cb * 8 + (j >> 2)];
          if ((j & 1) == 0) {  // columns j, j+1: one packed FMA into the partial sums (j & 3), (j & 3) + 1
            const float w0 = (j & 3) == 0 ? wv.x : wv.z, w1 = (j & 3) == 0 ? wv.y : wv.w;
            fma2(run[j & 3], run[(j & 3) + 1], w0, w1, fmaxf(__uint_as_float(r[j]), 0.f),
                 fmaxf(__uint_as_float(r[j + 1]), 0.f));
          }
          const int col = ch * (IT_N / 2) + cb * 32 + j;  // accumulator column = (query, head)
          const bool seg_done = (HG <= 32) ? ((j + 1) % HG == 0) : (j == 31 && ((cb + 1) * 32) % HG == 0);
          if (seg_done) {
            const float tot = (run[0] + run[1]) + (run[2] + run[3]);
            const int sg = col / HG;
            const int qq = sg / a.groups, gg = sg % a.groups;
            if constexpr (BLK) {
              vals[(cb * 32 + j) / HG] = (qq < qn && s <= p_first + qq) ? tot * a.score_scale + 0.f : -INFINITY;
            } else {
              if (qq < qn && s <= p_first + qq)
                a.out[((int64_t)(q0 + qq) * a.groups + gg) * a.width + s] = tot * a.score_scale + 0.f;
            }
            run[0] = run[1] = run[2] = run[3] = 0.f;
          }
        }
      }
      if constexpr (BLK) {
        const bool ok = a.bs == 16 ? block_max_epilogue<NSEG, 16>(vals, a, lane, warp, qd, ch, acc, aph, w.kt, q0,
                                                                   qn, p_first, xbuf, xbar, abort_flag)
                                   : block_max_epilogue<NSEG, 32>(vals, a, lane, warp, qd, ch, acc, aph, w.kt, q0,
                                                                   qn, p_first, xbuf, xbar, abort_flag);
        if (!ok) {
          *abort_flag = 1;
          break;
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&acce[acc]);
        if (w.last) tc::mbar_arrive(&wsempty[wb]);
      }
      advance(w, it);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && tid == 0) raise_flag(a.flags, TSA_FLAG_TIMEOUT);
  if (*abort_flag && warp == 8 && lane == 0) {
    // after an abort a q_I block or a key tile may still be landing: wait
    // (bounded by time only) for the last loads issued before the CTA exits
    volatile int keep_waiting = 0;
    if (b_last_tr >= 0) (void)tc::mbar_wait(bfull, b_last_tr & 1, &keep_waiting);
    for (int g = a_issued > IT_STAGES ? a_issued - IT_STAGES : 0; g < a_issued; ++g)
      (void)tc::mbar_wait(&full[g % IT_STAGES], (g / IT_STAGES) & 1, &keep_waiting);
  }
  if (warp == 5) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

// 2-D bf16 tensor map over a row-major [rows, cols] array, 128-byte swizzle.
cudaError_t make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                              uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool indexer_tc_supported(int H_I, int d_I, int groups, int bs) {
  if (bs != 1 && bs != 16 && bs != 32 && bs != 64 && bs != 128) return false;
  if (d_I != 64 && d_I != 128) return false;
  if (H_I < 2 || H_I > IT_N || (IT_N % H_I) != 0) return false;
  const int hg = H_I / groups;
  return hg >= 2 && hg <= 128 && (hg & (hg - 1)) == 0 && hg * groups == H_I;
}

template <int DI, int HG, bool BLK>
static cudaError_t launch_tc_t(const IndexerArgs& a, cudaStream_t stream) {
  CUtensorMap tq, tk;
  cudaError_t e = make_tmap_bf16_2d(&tq, a.q, (uint64_t)a.T_total * a.H_I, DI, IT_N, 64);
  if (e != cudaSuccess) return e;
  e = make_tmap_bf16_2d(&tk, a.k, (uint64_t)a.T_total, DI, IT_M, 64);
  if (e != cudaSuccess) return e;
  constexpr int smem = ItLayout<DI>::SMEM;
  e = cudaFuncSetAttribute(indexer_tc_kernel<DI, HG, BLK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // the whole shared-memory carveout, so that a top-k CTA fits beside this one
  e = cudaFuncSetAttribute(indexer_tc_kernel<DI, HG, BLK>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  // total (query block, key tile) pairs of the launch; one persistent CTA per SM
  const int QB = IT_N / a.H_I;
  const int nqb = (a.nq + QB - 1) / QB;
  int64_t total = 0;
  for (int qb = 0; qb < nqb; ++qb) {
    const int qn = std::min(QB, a.nq - qb * QB);
    total += (a.p_begin + qb * QB + qn - 1) / IT_M + 1;
  }
  if (total > 0x7fffffffLL) return cudaErrorInvalidValue;
  // SM count of the current device, read per launch (devices may differ)
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int grid = static_cast<int>(std::min<int64_t>(total, sms));
  indexer_tc_kernel<DI, HG, BLK><<<grid, IT_THREADS, smem, stream>>>(tq, tk, a, static_cast<int>(total));
  note_launch();
  return cudaGetLastError();
}

template <int DI, bool BLK>
static cudaError_t launch_tc_d(const IndexerArgs& a, cudaStream_t stream) {
  switch (a.H_I / a.groups) {
    case 2: return launch_tc_t<DI, 2, BLK>(a, stream);
    case 4: return launch_tc_t<DI, 4, BLK>(a, stream);
    case 8: return launch_tc_t<DI, 8, BLK>(a, stream);
    case 16: return launch_tc_t<DI, 16, BLK>(a, stream);
    case 32: return launch_tc_t<DI, 32, BLK>(a, stream);
    case 64: return launch_tc_t<DI, 64, BLK>(a, stream);
    default: return launch_tc_t<DI, 128, BLK>(a, stream);
  }
}

cudaError_t launch_indexer_tc(const IndexerArgs& a, cudaStream_t stream) {
  if (a.nq <= 0) return cudaSuccess;
  if (a.bs > 1) return a.d_I == 128 ? launch_tc_d<128, true>(a, stream) : launch_tc_d<64, true>(a, stream);
  return a.d_I == 128 ? launch_tc_d<128, false>(a, stream) : launch_tc_d<64, false>(a, stream);
}

}  // namespace tsa
