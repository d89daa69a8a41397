// Block Sparse-GQA backward, key-centric.
//
// Megatron-LM issue #7060 "Add trainable QSA sparse attention with a TileLang
// backend" ("Describe the solution you'd like": Sparse-GQA backward over exact
// block top-k selections, BSHD and packed THD).
//
// The gradient of one selected block (block_size keys of one kv group) is a sum
// over the queries that selected it.  A query-centric backward scatters a
// [block_size x d] dK and dV tile per (query, group, block) into global memory
// (64 KB of fp32 reductions per triple at block 64, d 128).  Here the
// selections are inverted once per call (count, scan, fill: for every (block,
// group) the list of queries that selected it, in any order), and one CTA takes
// a chunk of up to GK_CHUNK queries of one (block, group): K and V of the block
// stay in shared memory, the queries' q and dO rows stream through in batches
// of 64 (query, head) rows, dK and dV accumulate in registers and are reduced
// once per chunk, and only dQ (d floats per (query, head) and block) is
// reduced per triple.  The accumulation order of dQ, dK and dV is not fixed.
//
// Per batch (mma.sync m16n8k16, bf16 in, fp32 accumulate), with r = (query,
// head) rows and keys of the block:
//   S^T = K Q^T, dP^T = V dO^T                       [keys x r]
//   P^T = exp(scale S^T - lse_r) on causal keys (key position <= the query's)
//   dS^T = scale P^T (dP^T - Delta_r)
//   dV += P^T dO, dK += dS^T Q                       [keys x d]
//   dQ_r += dS K                                     [r x d]  (fp32 reductions)
#include <algorithm>

#include "kernels.cuh"

namespace tsa {

namespace {
constexpr int GK_THREADS = 256;
constexpr int GK_ROWS = 64;    // (query, head) rows per batch
constexpr int GK_CHUNK = 512;  // queries per CTA at most (longer lists are split over CTAs)

__device__ __forceinline__ int block_seq(const GqaKvArgs& a, int gb) {
  int lo = 0, hi = a.st.num_seqs - 1;  // last sequence whose first block is <= gb
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.blk_base[mid] <= gb) lo = mid; else hi = mid - 1;
  }
  return lo;
}
}  // namespace

// Selection entries (t, g, j) -> (global block, group) counts, or list fill.
template <bool FILL>
__global__ void gqa_inv_kernel(const __grid_constant__ GqaKvArgs a) {
  const int64_t total = static_cast<int64_t>(a.T) * a.Hkv * a.nsel;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = __ldg(a.blk + e);
    if (b < 0) continue;
    const int t = static_cast<int>(e / (static_cast<int64_t>(a.Hkv) * a.nsel));
    const int g = static_cast<int>((e / a.nsel) % a.Hkv);
    const int s = seq_of(a.st, t);
    const int p = t - a.st.cu[s];
    if (static_cast<int64_t>(b) * a.bs > p) continue;  // not a causal block of this query
    const int idx = (a.blk_base[s] + b) * a.Hkv + g;
    if (!FILL) {
      atomicAdd(a.cnt + idx, 1);
    } else {
      const int pos = atomicAdd(a.cur + idx, 1);
      a.list[a.off[idx] + pos] = t;
    }
  }
}

// Exclusive scans of the counts (list offsets) and of the per-list chunk
// counts; clears the fill cursors.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) gqa_inv_scan_kernel(const __grid_constant__ GqaKvArgs a, int nB) {
  __shared__ int warp_tot[2][32];
  __shared__ int carry[2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < 2) carry[threadIdx.x] = 0;
  __syncthreads();
  for (int base = 0; base < nB; base += 1024) {
    const int i = base + threadIdx.x;
    const int c = i < nB ? a.cnt[i] : 0;
    const int ch = (c + GK_CHUNK - 1) / GK_CHUNK;
    if (i < nB) a.cur[i] = 0;
    int x = c, y = ch;  // inclusive warp scans
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

template <int BS, int DH>
__global__ void __launch_bounds__(GK_THREADS, 2) gqa_bwd_kv_kernel(const __grid_constant__ GqaKvArgs a) {
  constexpr int RS = DH + 8;           // bf16 row stride of K, V, Q, dO tiles
  constexpr int PS = GK_ROWS + 8;      // bf16 row stride of P^T, dS^T
  constexpr int RT = BS / 16;          // 16-key row tiles
  constexpr int NWC = 8 / RT;          // warps per row tile
  constexpr int CA = GK_ROWS / NWC;    // (query, head) columns per warp in S^T
  constexpr int NTA = CA / 8;
  constexpr int DCOLS = DH / NWC;      // d columns per warp in dK, dV
  constexpr int NTB = DCOLS / 8;
  constexpr int NTC = DH / 16;         // d n-tiles per warp in dQ (two warps per 16-row tile)
  constexpr int CPR = DH / 8;          // 16-byte chunks per row
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [BS][RS]
  __nv_bfloat16* Vs = Ks + BS * RS;
  __nv_bfloat16* Qs = Vs + BS * RS;                                 // [GK_ROWS][RS]
  __nv_bfloat16* dOs = Qs + GK_ROWS * RS;
  __nv_bfloat16* PT = dOs + GK_ROWS * RS;                           // [BS][PS]
  __nv_bfloat16* dST = PT + BS * PS;
  float* lse2s = reinterpret_cast<float*>(dST + BS * PS);           // [GK_ROWS]
  float* dls = lse2s + GK_ROWS;
  int* qpos = reinterpret_cast<int*>(dls + GK_ROWS);                // local position of the row's query, -1 = none
  int* qtok = qpos + GK_ROWS;                                       // token of the row's query

  const int nB = a.nblk * a.Hkv;
  const int c = blockIdx.x;
  if (c >= a.choff[nB]) return;  // uniform
  int lo = 0, hi = nB - 1;       // the list holding chunk c: choff[idx] <= c < choff[idx + 1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.choff[mid] <= c) lo = mid; else hi = mid - 1;
  }
  const int idx = lo;
  const int gb = idx / a.Hkv, g = idx % a.Hkv;
  const int sq = block_seq(a, gb);
  const int b = gb - a.blk_base[sq];
  const int s0 = a.st.cu[sq];
  const int n = a.st.cu[sq + 1] - s0;
  const int kbase = b * BS;  // local position of the block's first key
  const int qbeg = a.off[idx] + (c - a.choff[idx]) * GK_CHUNK;
  const int qend = min(a.off[idx + 1], qbeg + GK_CHUNK);
  const int G = a.G, QB = GK_ROWS / G;  // queries per batch
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, c4 = lane & 3;

  // K and V of the block (rows past the sequence are zero)
  for (int i = tid; i < BS * CPR; i += GK_THREADS) {
    const int r = i / CPR, ch = i % CPR;
    const bool ok = kbase + r < n;
    const int64_t row = ((int64_t)(s0 + (ok ? kbase + r : 0)) * a.Hkv + g) * DH + ch * 8;
    cp_async16(smem_u32(Ks + r * RS + ch * 8), a.k + row, ok ? 16u : 0u);
    cp_async16(smem_u32(Vs + r * RS + ch * 8), a.v + row, ok ? 16u : 0u);
  }
  cp_async_commit();

  const int ra = warp % RT, ca = warp / RT;  // S^T tile: keys 16 ra .., columns CA ca ..
  float accK[NTB][4], accV[NTB][4];
#pragma unroll
  for (int i = 0; i < NTB; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) accK[i][e] = accV[i][e] = 0.f;

  for (int q0 = qbeg; q0 < qend; q0 += QB) {
    // rows of this batch: r = query qi * G + head hh
    if (tid < GK_ROWS) {
      const int qi = tid / G, hh = tid % G;
      const bool ok = qi < QB && q0 + qi < qend;
      const int t = ok ? a.list[q0 + qi] : -1;
      const int hq = g * G + hh;
      qtok[tid] = t;
      qpos[tid] = ok ? t - s0 : -1;
      lse2s[tid] = ok ? a.lse_in[(int64_t)t * a.Hq + hq] * kLog2e : 0.f;
      dls[tid] = ok ? a.dlt[(int64_t)t * a.Hq + hq] : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < GK_ROWS * CPR; i += GK_THREADS) {
      const int r = i / CPR, ch = i % CPR;
      const int t = qtok[r];
      const bool ok = t >= 0;
      const int64_t off = ((int64_t)(ok ? t : 0) * a.Hq + g * G + r % G) * DH + ch * 8;
      cp_async16(smem_u32(Qs + r * RS + ch * 8), a.q + off, ok ? 16u : 0u);
      cp_async16(smem_u32(dOs + r * RS + ch * 8), a.dout + off, ok ? 16u : 0u);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    // ---- S^T = K Q^T and dP^T = V dO^T for keys 16 ra .. +15, rows CA ca .. +CA-1
    {
      float s[NTA][4], dp[NTA][4];
#pragma unroll
      for (int i = 0; i < NTA; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[i][e] = dp[i][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < DH / 16; ks += 2) {
        uint32_t a0, a1, a2, a3, a4, a5, a6, a7, e0, e1, e2, e3, e4, e5, e6, e7;
        const int krow = ra * 16 + (lane & 15);
        ldsm_x4(smem_u32(Ks + krow * RS + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
        ldsm_x4(smem_u32(Ks + krow * RS + (ks + 1) * 16 + (lane >> 4) * 8), a4, a5, a6, a7);
        ldsm_x4(smem_u32(Vs + krow * RS + ks * 16 + (lane >> 4) * 8), e0, e1, e2, e3);
        ldsm_x4(smem_u32(Vs + krow * RS + (ks + 1) * 16 + (lane >> 4) * 8), e4, e5, e6, e7);
#pragma unroll
        for (int nt = 0; nt < NTA; ++nt) {
          uint32_t b0, b1, b2, b3;
          const int qrow = ca * CA + nt * 8 + (lane & 7);
          ldsm_x4(smem_u32(Qs + qrow * RS + ks * 16 + (lane >> 3) * 8), b0, b1, b2, b3);
          mma_bf16(s[nt], a0, a1, a2, a3, b0, b1);
          mma_bf16(s[nt], a4, a5, a6, a7, b2, b3);
          ldsm_x4(smem_u32(dOs + qrow * RS + ks * 16 + (lane >> 3) * 8), b0, b1, b2, b3);
          mma_bf16(dp[nt], e0, e1, e2, e3, b0, b1);
          mma_bf16(dp[nt], e4, e5, e6, e7, b2, b3);
        }
      }
      // P^T and dS^T (rows = keys, columns = (query, head) rows), causal keys only
#pragma unroll
      for (int nt = 0; nt < NTA; ++nt) {
        const int col = ca * CA + nt * 8 + 2 * c4;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int key = ra * 16 + gq + 8 * hr;
          const int kp = kbase + key;
          float P[2], dS[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int r = col + e;
            const bool v = kp < n && kp <= qpos[r];
            P[e] = v ? exp2f(s[nt][2 * hr + e] * a.scale_log2 - lse2s[r]) : 0.f;
            dS[e] = a.scale * P[e] * (dp[nt][2 * hr + e] - dls[r]);
          }
          *reinterpret_cast<uint32_t*>(PT + key * PS + col) = pack_bf16(P[0], P[1]);
          *reinterpret_cast<uint32_t*>(dST + key * PS + col) = pack_bf16(dS[0], dS[1]);
        }
      }
    }
    __syncthreads();

    // ---- dV += P^T dO, dK += dS^T Q: keys 16 rb .., d columns DCOLS cb ..
    {
      const int rb = warp % RT, cb = warp / RT;
#pragma unroll
      for (int kq = 0; kq < GK_ROWS / 16; ++kq) {
        uint32_t p0, p1, p2, p3, d0, d1, d2, d3;
        ldsm_x4(smem_u32(PT + (rb * 16 + (lane & 15)) * PS + kq * 16 + (lane >> 4) * 8), p0, p1, p2, p3);
        ldsm_x4(smem_u32(dST + (rb * 16 + (lane & 15)) * PS + kq * 16 + (lane >> 4) * 8), d0, d1, d2, d3);
#pragma unroll
        for (int nt = 0; nt < NTB; nt += 2) {
          uint32_t b0, b1, b2, b3;
          const int r = kq * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int ch = cb * DCOLS + nt * 8 + (lane >> 4) * 8;
          ldsm_x4_t(smem_u32(dOs + r * RS + ch), b0, b1, b2, b3);
          mma_bf16(accV[nt], p0, p1, p2, p3, b0, b1);
          mma_bf16(accV[nt + 1], p0, p1, p2, p3, b2, b3);
          ldsm_x4_t(smem_u32(Qs + r * RS + ch), b0, b1, b2, b3);
          mma_bf16(accK[nt], d0, d1, d2, d3, b0, b1);
          mma_bf16(accK[nt + 1], d0, d1, d2, d3, b2, b3);
        }
      }
    }

    // ---- dQ = dS K for rows 16 rc .., d columns DH/2 cc ..; reduced into the fp32 workspace
    {
      const int rc = warp & 3, cc = warp >> 2;
      float dq[NTC][4];
#pragma unroll
      for (int i = 0; i < NTC; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) dq[i][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < BS / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        const int krow = kk * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int mcol = rc * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4_t(smem_u32(dST + krow * PS + mcol), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NTC; nt += 2) {
          uint32_t b0, b1, b2, b3;
          const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int ch = cc * (DH / 2) + nt * 8 + (lane >> 4) * 8;
          ldsm_x4_t(smem_u32(Ks + key * RS + ch), b0, b1, b2, b3);
          mma_bf16(dq[nt], a0, a1, a2, a3, b0, b1);
          mma_bf16(dq[nt + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      const int r0 = rc * 16 + gq, r1 = r0 + 8;
      const int t0 = qtok[r0], t1 = qtok[r1];
      float* row0 = t0 >= 0 ? a.dq_acc + ((int64_t)t0 * a.Hq + g * G + r0 % G) * DH : nullptr;
      float* row1 = t1 >= 0 ? a.dq_acc + ((int64_t)t1 * a.Hq + g * G + r1 % G) * DH : nullptr;
#pragma unroll
      for (int nt = 0; nt < NTC; ++nt) {
        const int ch = cc * (DH / 2) + nt * 8;
        red_frag_v4(row0 ? row0 + ch : nullptr, row1 ? row1 + ch : nullptr, dq[nt], c4);
      }
    }
    __syncthreads();  // the next batch overwrites the row tiles and P^T / dS^T
  }
  cp_async_wait<0>();

  // ---- this chunk's dK, dV of the block's keys (fp32 reductions: other chunks of the list add theirs)
  {
    const int rb = warp % RT, cb = warp / RT;
    const int k0 = rb * 16 + gq, k1 = k0 + 8;
    const bool v0 = kbase + k0 < n, v1 = kbase + k1 < n;
    const int64_t o0 = ((int64_t)(s0 + kbase + k0) * a.Hkv + g) * DH;
    const int64_t o1 = ((int64_t)(s0 + kbase + k1) * a.Hkv + g) * DH;
#pragma unroll
    for (int nt = 0; nt < NTB; ++nt) {
      const int ch = cb * DCOLS + nt * 8;
      red_frag_v4(v0 ? a.dk_acc + o0 + ch : nullptr, v1 ? a.dk_acc + o1 + ch : nullptr, accK[nt], c4);
      red_frag_v4(v0 ? a.dv_acc + o0 + ch : nullptr, v1 ? a.dv_acc + o1 + ch : nullptr, accV[nt], c4);
    }
  }
}

template <int BS, int DH>
static cudaError_t launch_kv_t(const GqaKvArgs& a, int64_t grid, cudaStream_t stream) {
  constexpr int RS = DH + 8, PS = GK_ROWS + 8;
  const size_t smem = sizeof(__nv_bfloat16) * (2 * BS * RS + 2 * GK_ROWS * RS + 2 * BS * PS) + 16 * GK_ROWS;
  cudaError_t e = cudaFuncSetAttribute(gqa_bwd_kv_kernel<BS, DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  gqa_bwd_kv_kernel<BS, DH><<<static_cast<unsigned>(grid), GK_THREADS, smem, stream>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_gqa_bwd_kv(const GqaKvArgs& a, int d, cudaStream_t stream) {
  const int nB = a.nblk * a.Hkv;
  const int64_t entries = static_cast<int64_t>(a.T) * a.Hkv * a.nsel;
  if (entries <= 0 || nB <= 0) return cudaSuccess;
  cudaError_t e;
  const unsigned ig = static_cast<unsigned>(std::min<int64_t>((entries + 255) / 256, 4096));
  if ((e = cudaMemsetAsync(a.cnt, 0, sizeof(int) * nB, stream)) != cudaSuccess) return e;
  gqa_inv_kernel<false><<<ig, 256, 0, stream>>>(a);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gqa_inv_scan_kernel<<<1, 1024, 0, stream>>>(a, nB);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gqa_inv_kernel<true><<<ig, 256, 0, stream>>>(a);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // chunks: at most one partial chunk per list plus entries / GK_CHUNK full ones
  const int64_t grid = nB + (entries + GK_CHUNK - 1) / GK_CHUNK;
  if (a.bs == 64 && d == 128) return launch_kv_t<64, 128>(a, grid, stream);
  if (a.bs == 64 && d == 64) return launch_kv_t<64, 64>(a, grid, stream);
  if (a.bs == 32 && d == 128) return launch_kv_t<32, 128>(a, grid, stream);
  return launch_kv_t<32, 64>(a, grid, stream);
}

}  // namespace tsa
