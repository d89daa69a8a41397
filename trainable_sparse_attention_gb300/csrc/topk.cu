// Deterministic exact top-k over fp32 score rows.
//
// Order: score descending, then index ascending -- the lexicographic
// (score, block_id) key of Megatron-LM issue #7060 "Add trainable QSA sparse
// attention with a TileLang backend" ("Describe the solution you'd like"),
// needed because ReLU indexer scores tie at exactly zero.  -inf entries are
// masked ("cleaned") logits and are never selected; missing slots are -1.
//
// Design (one CTA per row, no global atomics, no data-dependent ordering):
//  * every score maps to an order-preserving 32-bit key u (-0.0 folded to +0.0);
//    the composite 64-bit key (u << 32 | ~index) is unique per row, so the
//    result is a pure function of the row;
//  * rows of <= 4096 entries: bitonic sort of all composite keys in shared memory;
//  * longer rows: three histogram passes (11+11+10 bits) find the k-th largest
//    u = tau; one ordered pass then keeps every u > tau and the lowest-index
//    (k - count(u > tau)) entries with u == tau, ranked by a block prefix sum
//    in index order; the k survivors are bitonic-sorted.
#include "kernels.cuh"

namespace tsa {

constexpr int TK_THREADS = 512;
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int TK_SMALL = 4096;  // rows with at most this many entries are fully sorted
constexpr int TK_MAXK = 4096;   // largest supported k
constexpr int TK_BINS = 2048;
constexpr int TK_PER = 8;       // consecutive entries per thread in the sweeps over long rows


__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t b = __float_as_uint(s);
  if ((b & 0x7fffffffu) == 0u) b = 0u;  // -0.0 == +0.0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ uint64_t comp_key(uint32_t u, uint32_t i) {
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint64_t>(~i);
}

// Bitonic sort of s[0..P) into descending order (P a power of two).
__device__ void bitonic_desc(uint64_t* s, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (P >> 1); i += blockDim.x) {
        int pos = 2 * i - (i & (stride - 1));
        int par = pos + stride;
        bool desc = (pos & size) == 0;
        uint64_t a = s[pos], b = s[par];
        if ((a < b) == desc) { s[pos] = b; s[par] = a; }
      }
      __syncthreads();
    }
  }
}

// Suffix search: find the bin b with count(bins > b) < k <= count(bins >= b).
// Writes (bin, above) to sh[0], sh[1] or bin = -1 if all bins hold < k; total to sh[2].
__device__ void find_bin(const uint32_t* hist, int nbins, uint32_t k, uint32_t* warp_tot, int* sh) {
  const int per = nbins / TK_THREADS;  // 4 or 2
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t v = 0;
  for (int j = 0; j < per; ++j) v += hist[threadIdx.x * per + j];
  uint32_t x = v;  // inclusive suffix sum inside the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) warp_tot[warp] = x;
  if (threadIdx.x == 0) sh[0] = -1;
  __syncthreads();
  uint32_t above = x - v;
  for (int w = warp + 1; w < TK_WARPS; ++w) above += warp_tot[w];
  if (threadIdx.x == 0) {
    uint32_t tot = 0;
    for (int w = 0; w < TK_WARPS; ++w) tot += warp_tot[w];
    sh[2] = static_cast<int>(tot);
  }
  uint32_t cum = above;
  for (int j = per - 1; j >= 0; --j) {
    int b = threadIdx.x * per + j;
    uint32_t c = hist[b];
    if (cum < k && cum + c >= k) { sh[0] = b; sh[1] = static_cast<int>(cum); }
    cum += c;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(TK_THREADS) topk_rows_kernel(TopkRows a) {
  extern __shared__ uint64_t keys[];  // TK_MAXK (>= TK_SMALL) composite keys
  __shared__ uint32_t hist[TK_BINS];
  __shared__ uint32_t warp_tot[2][TK_WARPS];
  __shared__ int sh[4];

  const int64_t r = blockIdx.x;
  const float* row = a.scores + r * a.ld;
  int32_t* out = a.out + r * a.out_ld;
  int64_t n = a.width;
  if (a.mode != 0) {
    int64_t p = a.p0 + r / a.groups;
    int64_t c = (a.mode == 1) ? p + 1 : p / a.bs + 1;
    n = c < n ? c : n;
  }
  const int k = a.k;
  const float NEG_INF = __int_as_float(0xff800000);

  if (n <= TK_SMALL) {
    int P = 1;
    while (P < n) P <<= 1;
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
      uint64_t key = 0;
      if (i < n) {
        float s = row[i];
        if (s != NEG_INF) key = comp_key(order_key(s), static_cast<uint32_t>(i));
      }
      keys[i] = key;
    }
    __syncthreads();
    bitonic_desc(keys, P);
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
      uint64_t key = (j < P) ? keys[j] : 0ull;
      out[j] = key ? static_cast<int32_t>(~static_cast<uint32_t>(key & 0xffffffffull)) : -1;
    }
    return;
  }

  // ---- radix select of the k-th largest u (three passes over the row).  Each
  // thread takes TK_PER consecutive entries per sweep, so their loads are in
  // flight together.
  const int shifts[3] = {21, 10, 0};
  const int nbits[3] = {11, 11, 10};
  uint32_t prefix = 0, above_total = 0, kk = static_cast<uint32_t>(k);
  bool take_all = false;
  for (int pass = 0; pass < 3; ++pass) {
    const int nb = 1 << nbits[pass];
    for (int i = threadIdx.x; i < TK_BINS; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int sh_pref = shifts[pass] + nbits[pass];  // bits above this pass
    for (int64_t base = 0; base < n; base += TK_PER * TK_THREADS) {
      const int64_t i0 = base + static_cast<int64_t>(threadIdx.x) * TK_PER;
      float v[TK_PER];
#pragma unroll
      for (int e = 0; e < TK_PER; ++e) v[e] = (i0 + e < n) ? row[i0 + e] : NEG_INF;
#pragma unroll
      for (int e = 0; e < TK_PER; ++e) {
        if (v[e] == NEG_INF) continue;
        const uint32_t u = order_key(v[e]);
        if (pass == 0 || (u >> sh_pref) == prefix) atomicAdd(&hist[(u >> shifts[pass]) & (nb - 1)], 1u);
      }
    }
    __syncthreads();
    find_bin(hist, nb == TK_BINS ? TK_BINS : nb, kk, warp_tot[0], sh);
    int bin = sh[0];
    if (bin < 0) {  // fewer than k candidates in total (only possible on the first pass)
      take_all = true;
      break;
    }
    above_total += static_cast<uint32_t>(sh[1]);
    kk -= static_cast<uint32_t>(sh[1]);
    prefix = (prefix << nbits[pass]) | static_cast<uint32_t>(bin);
    __syncthreads();
  }
  const uint32_t tau = take_all ? 0u : prefix;
  const uint32_t c_gt = take_all ? 0u : above_total;
  const uint32_t need = take_all ? 0u : kk;  // how many u == tau to keep (lowest indices)

  // ---- ordered selection pass: thread t holds entries [base + TK_PER t, +TK_PER),
  // so thread order is index order; one block-wide exclusive scan of the
  // per-thread counts ranks every kept entry.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t base_gt = 0, base_eq = 0;
  for (int64_t base = 0; base < n; base += TK_PER * TK_THREADS) {
    const int64_t i0 = base + static_cast<int64_t>(threadIdx.x) * TK_PER;
    uint32_t uu[TK_PER];
    uint32_t mgt = 0, meq = 0;
#pragma unroll
    for (int e = 0; e < TK_PER; ++e) {
      const float s = (i0 + e < n) ? row[i0 + e] : NEG_INF;
      const bool cand = s != NEG_INF;
      const uint32_t u = cand ? order_key(s) : 0u;
      uu[e] = u;
      if (cand && u > tau) mgt |= 1u << e;
      if (cand && !take_all && u == tau) meq |= 1u << e;
    }
    // inclusive warp scans of the two counts, packed 16 + 16 bits (each <= 32 * TK_PER)
    const uint32_t mine = (static_cast<uint32_t>(__popc(mgt)) << 16) | static_cast<uint32_t>(__popc(meq));
    uint32_t x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[0][warp] = x;
    __syncthreads();
    uint32_t off = x - mine, tot = 0;
    for (int w = 0; w < TK_WARPS; ++w) {
      const uint32_t wt = warp_tot[0][w];
      if (w < warp) off += wt;
      tot += wt;
    }
    uint32_t og = base_gt + (off >> 16), oe = base_eq + (off & 0xffffu);
#pragma unroll
    for (int e = 0; e < TK_PER; ++e) {
      if ((mgt >> e) & 1u) keys[og++] = comp_key(uu[e], static_cast<uint32_t>(i0 + e));
      if ((meq >> e) & 1u) {
        if (oe < need) keys[c_gt + oe] = comp_key(uu[e], static_cast<uint32_t>(i0 + e));
        ++oe;
      }
    }
    base_gt += tot >> 16;
    base_eq += tot & 0xffffu;
    __syncthreads();
  }
  const int nsel = take_all ? static_cast<int>(base_gt) : k;
  int P = 1;
  while (P < nsel) P <<= 1;
  for (int i = nsel + threadIdx.x; i < P; i += blockDim.x) keys[i] = 0ull;
  __syncthreads();
  bitonic_desc(keys, P);
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    uint64_t key = (j < nsel) ? keys[j] : 0ull;
    out[j] = key ? static_cast<int32_t>(~static_cast<uint32_t>(key & 0xffffffffull)) : -1;
  }
}

cudaError_t launch_topk_rows(const TopkRows& a, int64_t rows, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  size_t smem = sizeof(uint64_t) * TK_MAXK;
  topk_rows_kernel<<<static_cast<unsigned>(rows), TK_THREADS, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace tsa
