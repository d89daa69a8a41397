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
//    result is a pure function of the row, whatever order the keys are
//    gathered in;
//  * rows of <= 4096 entries: sort of all composite keys in shared memory;
//  * longer rows: a 13-bit histogram of u (one sweep over the row) finds the
//    bin b1 holding the k-th largest entry, with c_gt entries above it.  When
//    the c_gt + count(b1) keys of the bins >= b1 fit the 4096-key buffer (the
//    usual case: a 13-bit bin spans 1/16 of an octave), a second sweep
//    gathers exactly those keys and the sort of the buffer puts the k largest
//    first.  Otherwise (heavy exact ties at the threshold) two more histogram
//    sweeps (10 + 9 bits) find the k-th largest u = tau, and an ordered sweep
//    keeps every u > tau and the lowest-index (k - count(u > tau)) entries
//    with u == tau, ranked by a block prefix sum in index order;
//  * the usual path for long rows gathers about 1.25 k candidates above a
//    threshold guessed from a sample and orders them without a sort: buckets
//    of the candidates' u range, a scan of the bucket counts, and each key's
//    rank inside its bucket (a bucket holding more than TK_BUCKET_MAX keys --
//    exact ties in u, or a dense spot under an outlier -- sends the row to the
//    sort instead);
//  * the sort is bitonic: strides below 32 elements exchange registers between
//    lanes, strides inside one warp's chunk exchange a thread's own registers,
//    and only the longer strides go through shared memory with a block barrier.
#include "kernels.cuh"

namespace tsa {

constexpr int TK_THREADS = 512;
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int TK_SMALL = 4096;  // rows with at most this many entries are fully sorted
constexpr int TK_MAXK = 4096;   // largest supported k and capacity of the key buffer
constexpr int TK_BITS1 = 13;    // first histogram digit
constexpr int TK_BINS = 1 << TK_BITS1;
constexpr int TK_SH1 = 32 - TK_BITS1;
constexpr int TK_PER = 8;       // consecutive entries per thread in the sweeps over long rows
constexpr int TK_SMEM = TK_MAXK * 8 + TK_BINS * 4;
constexpr int TK_NB = 2048;          // buckets of the final ranking (4 per thread)
constexpr int TK_BUCKET_MAX = 128;   // a fuller bucket (ties in u, a dense spot) sends the row to the sort
static_assert(TK_NB == 4 * TK_THREADS, "bucket scan: four buckets per thread");
static_assert(TK_NB * 4 + TK_MAXK * 2 <= TK_MAXK * 8, "bucket scratch fits the key buffer");


__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t b = __float_as_uint(s);
  if ((b & 0x7fffffffu) == 0u) b = 0u;  // -0.0 == +0.0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ uint64_t comp_key(uint32_t u, uint32_t i) {
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint64_t>(~i);
}

// Bitonic sort of s[0..P) into descending order, shared memory only (small P).
__device__ void bitonic_desc_smem(uint64_t* s, int P) {
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

// The compare-exchange steps of one bitonic merge of block length `size` whose
// strides are at most `top` (< 32 E), on registers: thread (warp w, lane l)
// holds positions w 32E + 32e + l, e < E.  Strides below 32 pair lanes
// (l ^ stride), longer strides pair a thread's own registers (e ^ stride/32).
template <int E>
__device__ __forceinline__ void bitonic_reg_steps(uint64_t (&v)[E], int wbase, int size, int top) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int st = 16 * E; st >= 1; st >>= 1) {
    if (st > top) continue;
    if (st >= 32) {
      const int se = st >> 5;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (e & se) continue;
        const bool desc = ((wbase + 32 * e + lane) & size) == 0;
        const uint64_t x = v[e], y = v[e + se];
        const bool sw = (x < y) == desc;
        v[e] = sw ? y : x;
        v[e + se] = sw ? x : y;
      }
    } else {
      const bool lower = (lane & st) == 0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, v[e], st);
        const bool desc = ((wbase + 32 * e + lane) & size) == 0;
        const bool keep_max = lower == desc;
        v[e] = (v[e] > o) == keep_max ? v[e] : o;
      }
    }
  }
}

// Bitonic sort of s[0..P) into descending order, P = 512 E.
template <int E>
__device__ void bitonic_desc_reg(uint64_t* s) {
  constexpr int P = TK_THREADS * E;
  constexpr int W = 32 * E;  // one warp's chunk
  const int lane = threadIdx.x & 31;
  const int wbase = (threadIdx.x >> 5) * W;
  uint64_t v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = s[wbase + 32 * e + lane];
  for (int size = 2; size <= W; size <<= 1) bitonic_reg_steps<E>(v, wbase, size, size >> 1);
  for (int size = 2 * W; size <= P; size <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) s[wbase + 32 * e + lane] = v[e];
    __syncthreads();
    for (int stride = size >> 1; stride >= W; stride >>= 1) {
      for (int i = threadIdx.x; i < (P >> 1); i += TK_THREADS) {
        const int pos = 2 * i - (i & (stride - 1));
        const int par = pos + stride;
        const bool desc = (pos & size) == 0;
        const uint64_t a = s[pos], b = s[par];
        if ((a < b) == desc) { s[pos] = b; s[par] = a; }
      }
      __syncthreads();
    }
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = s[wbase + 32 * e + lane];
    bitonic_reg_steps<E>(v, wbase, size, W >> 1);
  }
  __syncthreads();  // every thread has read s before it is overwritten
#pragma unroll
  for (int e = 0; e < E; ++e) s[wbase + 32 * e + lane] = v[e];
  __syncthreads();
}

// Bitonic merge of the bitonic sequence s[0..P) into descending order, P = 512 E.
template <int E>
__device__ void bitonic_merge_reg(uint64_t* s) {
  constexpr int P = TK_THREADS * E;
  constexpr int W = 32 * E;
  for (int stride = P >> 1; stride >= W; stride >>= 1) {
    for (int i = threadIdx.x; i < (P >> 1); i += TK_THREADS) {
      const int pos = 2 * i - (i & (stride - 1));
      const int par = pos + stride;
      const uint64_t a = s[pos], b = s[par];
      if (a < b) { s[pos] = b; s[par] = a; }
    }
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int wbase = (threadIdx.x >> 5) * W;
  uint64_t v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = s[wbase + 32 * e + lane];
  bitonic_reg_steps<E>(v, wbase, 2 * P, W >> 1);  // block length 2P: every pair descending
#pragma unroll
  for (int e = 0; e < E; ++e) s[wbase + 32 * e + lane] = v[e];
  __syncthreads();
}

// Merge of a bitonic s[0..P) into descending order, P a power of two <= TK_MAXK.
__device__ void merge_desc(uint64_t* s, int P) {
  if (P >= 4096) bitonic_merge_reg<8>(s);
  else if (P == 2048) bitonic_merge_reg<4>(s);
  else if (P == 1024) bitonic_merge_reg<2>(s);
  else if (P == 512) bitonic_merge_reg<1>(s);
  else {
    for (int stride = P >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (P >> 1); i += blockDim.x) {
        const int pos = 2 * i - (i & (stride - 1));
        const int par = pos + stride;
        const uint64_t a = s[pos], b = s[par];
        if (a < b) { s[pos] = b; s[par] = a; }
      }
      __syncthreads();
    }
  }
}

// Sort s[0..P) descending, P a power of two <= TK_MAXK.
__device__ void sort_desc(uint64_t* s, int P) {
  if (P >= 4096) bitonic_desc_reg<8>(s);
  else if (P == 2048) bitonic_desc_reg<4>(s);
  else if (P == 1024) bitonic_desc_reg<2>(s);
  else if (P == 512) bitonic_desc_reg<1>(s);
  else bitonic_desc_smem(s, P);
}

// Suffix search: find the bin b with count(bins > b) < k <= count(bins >= b).
// Writes (bin, above) to sh[0], sh[1] or bin = -1 if all bins hold < k; total to sh[2].
// Warp w owns the contiguous bins [w R, (w+1) R), R = nbins / 16 >= 32: the
// warp totals locate the owning warp, which then scans its bins from the top
// in chunks of 32 (lane l reads bin c + l: no bank conflicts).
__device__ void find_bin(const uint32_t* hist, int nbins, uint32_t k, uint32_t* warp_tot, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = nbins / TK_WARPS;
  const int b0 = warp * R;
  uint32_t s = 0;
  for (int i = lane; i < R; i += 32) s += hist[b0 + i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) warp_tot[warp] = s;
  if (threadIdx.x == 0) sh[0] = -1;
  __syncthreads();
  uint32_t above = 0, tot = 0;
  for (int w = 0; w < TK_WARPS; ++w) {
    const uint32_t t = warp_tot[w];
    tot += t;
    if (w > warp) above += t;
  }
  if (threadIdx.x == 0) sh[2] = static_cast<int>(tot);
  if (above < k && above + s >= k) {  // warp-uniform: this warp's bins hold the k-th entry
    uint32_t cum = above;
    for (int c = R - 32; c >= 0; c -= 32) {
      const uint32_t h = hist[b0 + c + lane];
      uint32_t x = h;  // inclusive suffix sum over lanes lane..31 of the chunk
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x += y;
      }
      const uint32_t ab = cum + x - h;  // entries in bins above bin b0 + c + lane
      const bool hit = ab < k && ab + h >= k;
      if (__ballot_sync(0xffffffffu, hit)) {
        if (hit) { sh[0] = b0 + c + lane; sh[1] = static_cast<int>(ab); }
        break;
      }
      cum += __shfl_sync(0xffffffffu, x, 0);
    }
  }
  __syncthreads();
}

// TK_PER consecutive entries of a row starting at i0 (-inf past the end).
__device__ __forceinline__ void load_run(const float* row, int64_t i0, int64_t n, bool vec, float (&v)[TK_PER]) {
  const float NEG_INF = __int_as_float(0xff800000);
  if (vec && i0 + TK_PER <= n) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(row + i0));
    const float4 y = __ldg(reinterpret_cast<const float4*>(row + i0 + 4));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
  } else {
#pragma unroll
    for (int e = 0; e < TK_PER; ++e) v[e] = (i0 + e < n) ? __ldg(row + i0 + e) : NEG_INF;
  }
}

// Runs over a row: thread t takes the TK_PER entries at base + TK_PER t of
// each run of TK_PER x TK_THREADS; the next run's loads are issued before f
// processes the current one.  f(v, i0) is called by every thread for every
// run (block-uniform trip count, so f may hold block barriers).
// for_runs_from takes the first run already loaded (into v).
template <class F>
__device__ __forceinline__ void for_runs_from(const float* row, int64_t n, bool vec, float (&v)[TK_PER], F f) {
  const int64_t me = static_cast<int64_t>(threadIdx.x) * TK_PER;
  const int64_t step = static_cast<int64_t>(TK_PER) * TK_THREADS;
  for (int64_t base = 0; base < n; base += step) {
    float nv[TK_PER];
    const bool more = base + step < n;
    if (more) load_run(row, base + step + me, n, vec, nv);
    f(v, base + me);
    if (more) {
#pragma unroll
      for (int e = 0; e < TK_PER; ++e) v[e] = nv[e];
    }
  }
}
template <class F>
__device__ __forceinline__ void for_runs(const float* row, int64_t n, bool vec, F f) {
  float v[TK_PER];
  load_run(row, static_cast<int64_t>(threadIdx.x) * TK_PER, n, vec, v);
  for_runs_from(row, n, vec, v, f);
}

// Appends the keys of the run entries flagged in msk (thread-local bits) to
// keys[], at slots reserved with one warp scan and one shared-counter atomic
// per warp; slots past the buffer are counted but not written.
__device__ __forceinline__ void append_keys(const float (&v)[TK_PER], int64_t i0, uint32_t msk, uint64_t* keys,
                                            uint32_t* counter) {
  const int lane = threadIdx.x & 31;
  if (__ballot_sync(0xffffffffu, msk != 0u) == 0u) return;
  const uint32_t mine = static_cast<uint32_t>(__popc(msk));
  uint32_t x = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  const uint32_t wtot = __shfl_sync(0xffffffffu, x, 31);
  uint32_t b = 0;
  if (lane == 0) b = atomicAdd(counter, wtot);
  uint32_t o = __shfl_sync(0xffffffffu, b, 0) + x - mine;
  while (msk) {
    const int e = __ffs(msk) - 1;
    msk &= msk - 1u;
    float s = v[0];
#pragma unroll
    for (int j = 1; j < TK_PER; ++j) s = (e == j) ? v[j] : s;
    if (o < static_cast<uint32_t>(TK_MAXK)) keys[o] = comp_key(order_key(s), static_cast<uint32_t>(i0 + e));
    ++o;
  }
}

// Writes the first k keys of the descending key list s[0..m) as indices, -1 past m.
__device__ __forceinline__ void emit(const uint64_t* s, int m, int k, int32_t* out) {
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    const uint64_t key = (j < m) ? s[j] : 0ull;
    out[j] = key ? static_cast<int32_t>(~static_cast<uint32_t>(key & 0xffffffffull)) : -1;
  }
}

// The score of a composite key (inverse of order_key on its upper half).
__device__ __forceinline__ float key_score(uint64_t key) {
  const uint32_t u = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// Orders the m keys of keys[0..m) and writes the row's first k.  When m is
// between Pk = 2^ceil(log2 k) and 2 Pk, the first Pk keys (A) and the other
// m - Pk (B, zero-padded to PB) are sorted on their own; A[i] = max(A[i],
// B[Pk - 1 - i]) then holds the Pk largest of both as a bitonic sequence (B
// read backwards, zeros past PB), and one merge orders them.  Otherwise all m
// keys are sorted, zero-padded to a power of two.
__device__ __forceinline__ void finish_row(uint64_t* keys, int m, int k, int32_t* out) {
  int Pk = 1;
  while (Pk < k) Pk <<= 1;
  if (Pk >= 512 && m > Pk && m - Pk <= Pk) {
    int PB = 1;
    while (PB < m - Pk) PB <<= 1;
    for (int i = m + threadIdx.x; i < Pk + PB; i += TK_THREADS) keys[i] = 0ull;
    __syncthreads();
    sort_desc(keys, Pk);
    sort_desc(keys + Pk, PB);
    for (int t = threadIdx.x; t < PB; t += TK_THREADS) {
      const int i = Pk - PB + t;
      const uint64_t a = keys[i], b = keys[Pk + PB - 1 - t];
      keys[i] = a > b ? a : b;
    }
    __syncthreads();
    merge_desc(keys, Pk);
    emit(keys, Pk, k, out);
    return;
  }
  int P = 1;
  while (P < m) P <<= 1;
  for (int i = m + threadIdx.x; i < P; i += TK_THREADS) keys[i] = 0ull;
  __syncthreads();
  sort_desc(keys, P);
  emit(keys, m, k, out);
}

// Writes the first k of the m keys packed[0..m) in descending order as
// indices (m >= k), without a sort: every key falls in one of TK_NB buckets
// by its u (the range [u_lo, u_hi] of the keys scaled to the buckets, higher
// u in lower buckets), a scan of the bucket counts gives each bucket's place
// in the output, and a key's rank inside its bucket is the number of keys of
// the bucket above it.  The keys are unique, so the ranks are a permutation
// and the result equals the sorted order.  Returns false (block-uniform,
// nothing written) when a bucket holds more than TK_BUCKET_MAX keys; packed
// is left unchanged either way.  Scratch: cnt[TK_NB] and pos[m].
__device__ bool rank_by_buckets(const uint64_t* packed, int m, int k, uint32_t u_lo, uint32_t u_hi, uint32_t* cnt,
                                uint16_t* pos, uint32_t* warp_tot, int* sh, int32_t* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t range = u_hi - u_lo;
  int sft = 0;
  while ((range >> sft) >= static_cast<uint32_t>(TK_NB)) ++sft;
  auto bucket = [&](uint64_t key) {
    return TK_NB - 1 - static_cast<int>((static_cast<uint32_t>(key >> 32) - u_lo) >> sft);
  };
  for (int i = threadIdx.x; i < TK_NB; i += TK_THREADS) cnt[i] = 0;
  if (threadIdx.x == 0) sh[3] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < m; i += TK_THREADS) atomicAdd(&cnt[bucket(packed[i])], 1u);
  __syncthreads();
  // exclusive scan of the counts (buckets 4t .. 4t+3 on thread t) and their maximum
  uint32_t c[4], tsum = 0, tmax = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    c[e] = cnt[4 * threadIdx.x + e];
    tsum += c[e];
    tmax = c[e] > tmax ? c[e] : tmax;
  }
  uint32_t x = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t y = __shfl_xor_sync(0xffffffffu, tmax, o);
    tmax = y > tmax ? y : tmax;
  }
  if (lane == 31) warp_tot[warp] = x;
  if (lane == 0) atomicMax(&sh[3], static_cast<int>(tmax));
  __syncthreads();
  if (sh[3] > TK_BUCKET_MAX) return false;
  uint32_t off = x - tsum;
  for (int w = 0; w < warp; ++w) off += warp_tot[w];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    cnt[4 * threadIdx.x + e] = off;
    off += c[e];
  }
  __syncthreads();
  // place every key in its bucket's range (any order inside a bucket); cnt[b]
  // then holds the end of bucket b, the start of bucket b + 1
  for (int i = threadIdx.x; i < m; i += TK_THREADS) pos[atomicAdd(&cnt[bucket(packed[i])], 1u)] = static_cast<uint16_t>(i);
  __syncthreads();
  for (int i = threadIdx.x; i < m; i += TK_THREADS) {
    const uint64_t key = packed[i];
    const int b = bucket(key);
    const uint32_t st = b > 0 ? cnt[b - 1] : 0u, en = cnt[b];
    if (st >= static_cast<uint32_t>(k)) continue;
    uint32_t r = st;
    for (uint32_t j = st; j < en; ++j) r += packed[pos[j]] > key ? 1u : 0u;
    if (r < static_cast<uint32_t>(k)) out[r] = static_cast<int32_t>(~static_cast<uint32_t>(key & 0xffffffffull));
  }
  return true;
}

// The lower edge of first-digit bin b as a score (inverse of order_key).
__device__ __forceinline__ float bin_floor(int b) {
  const uint32_t u = static_cast<uint32_t>(b) << TK_SH1;
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// One CTA per row.  Rows of n > 4096 entries:
//  * sample: TK_THREADS runs of TK_PER entries spread evenly over the row give
//    a first-digit histogram; the bin where its count from the top reaches
//    1.25 k (scaled to the sample) gives a score threshold g;
//  * guided sweep: every candidate >= g is gathered; if that is between k and
//    TK_MAXK keys, the k largest are among them and the sort finishes the row;
//  * otherwise the exact path: sweep 1 (first-digit histogram), then either
//    sweep 2 (gather the bins >= b1) or, under heavy ties at the threshold,
//    the three-digit search and the ordered selection sweep.
// The guess only decides which exact path runs: the result never depends on it.
__global__ void __launch_bounds__(TK_THREADS, 3) topk_rows_kernel(TopkRows a) {
  extern __shared__ uint64_t keys[];                              // TK_MAXK composite keys
  uint32_t* hist = reinterpret_cast<uint32_t*>(keys + TK_MAXK);   // TK_BINS counters
  __shared__ uint32_t warp_tot[TK_WARPS];
  __shared__ int sh[4];
  __shared__ uint32_t slots[2];
  const float NEG_INF = __int_as_float(0xff800000);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int k = a.k;

  const int64_t r = blockIdx.x;
  const float* row = a.scores + r * a.ld;
  int32_t* out = a.out + r * a.out_ld;
  int64_t n = a.width;
  if (a.mode != 0) {
    const int64_t p = a.p0 + r / a.groups;
    const int64_t c = (a.mode == 1) ? p + 1 : p / a.bs + 1;
    n = c < n ? c : n;
  }

  if (n <= TK_SMALL) {
    int P = 1;
    while (P < n) P <<= 1;
    for (int i = threadIdx.x; i < P; i += TK_THREADS) {
      uint64_t key = 0;
      if (i < n) {
        const float s = row[i];
        if (s != NEG_INF) key = comp_key(order_key(s), static_cast<uint32_t>(i));
      }
      keys[i] = key;
    }
    __syncthreads();
    sort_desc(keys, P);
    emit(keys, P, k, out);
    return;
  }

  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;

  // ---- sample: thread t counts the TK_PER entries at about t n / TK_THREADS.
  // Its loads and those of the guided sweep's first run are issued together,
  // and the histogram is cleared while they are in flight.
  float v0[TK_PER];
  {
    const int64_t i0 = ((static_cast<int64_t>(threadIdx.x) * n / TK_THREADS) & ~static_cast<int64_t>(TK_PER - 1));
    float v[TK_PER];
    load_run(row, i0, n, vec, v);
    load_run(row, static_cast<int64_t>(threadIdx.x) * TK_PER, n, vec, v0);
    for (int i = threadIdx.x; i < TK_BINS; i += TK_THREADS) hist[i] = 0;
    if (threadIdx.x < 2) slots[threadIdx.x] = 0;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < TK_PER; ++e)
      if (v[e] != NEG_INF) atomicAdd(&hist[order_key(v[e]) >> TK_SH1], 1u);
  }
  __syncthreads();
  const int64_t sample = static_cast<int64_t>(TK_PER) * TK_THREADS;
  const int64_t target = static_cast<int64_t>(k) + (k >> 2);
  const uint32_t tq = static_cast<uint32_t>((target * sample + n - 1) / n);  // the target rank in the sample
  find_bin(hist, TK_BINS, tq, warp_tot, sh);
  const int gbin = sh[0];

  if (gbin >= 0) {
    // ---- guided sweep: gather every candidate >= g (float order; -0.0 ==
    // +0.0).  g interpolates inside the sample's bin, assuming its entries
    // spread evenly over the bin's score range.  Warp w appends to its own
    // region of WCAP keys: per run, each thread marks its hits in a bit mask,
    // one warp prefix sum of the hit counts places them, and the warp's count
    // stays in a register (no atomics; the order of the keys inside the region
    // does not matter: the ranking and the sort depend only on the keys).
    float g = bin_floor(gbin);
    if (gbin + 1 < TK_BINS) {
      const float top = bin_floor(gbin + 1);
      const float f = static_cast<float>(tq - static_cast<uint32_t>(sh[1])) / static_cast<float>(hist[gbin]);
      g = top - f * (top - g);
    }
    constexpr int WCAP = TK_MAXK / TK_WARPS;
    uint64_t* wk = keys + warp * WCAP;
    uint32_t wcnt = 0;  // warp-uniform
    for_runs_from(row, n, vec, v0, [&](const float (&v)[TK_PER], int64_t i0) {
      uint32_t msk = 0;
#pragma unroll
      for (int e = 0; e < TK_PER; ++e) msk |= (v[e] >= g && v[e] != NEG_INF) ? (1u << e) : 0u;
      if (__any_sync(0xffffffffu, msk != 0u)) {
        const uint32_t mine = static_cast<uint32_t>(__popc(msk));
        uint32_t x = mine;  // inclusive scan of the hit counts over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        uint32_t pos = wcnt + x - mine;
        while (msk) {
          const int e = __ffs(msk) - 1;
          msk &= msk - 1u;
          float sv = v[0];
#pragma unroll
          for (int j = 1; j < TK_PER; ++j) sv = (e == j) ? v[j] : sv;
          if (pos < static_cast<uint32_t>(WCAP)) wk[pos] = comp_key(order_key(sv), static_cast<uint32_t>(i0 + e));
          ++pos;
        }
        wcnt += __shfl_sync(0xffffffffu, x, 31);
      }
    });
    if (lane == 0) warp_tot[warp] = wcnt;
    __syncthreads();
    uint32_t cnt = 0, before = 0;
    bool over = false;
    for (int w = 0; w < TK_WARPS; ++w) {
      const uint32_t t = warp_tot[w];
      if (w < warp) before += t;
      cnt += t;
      over = over || t > static_cast<uint32_t>(WCAP);
    }
    if (!over && cnt >= static_cast<uint32_t>(k)) {
      // the k largest are among the gathered keys: pack the regions into the
      // (now free) histogram area, with the range of their u, and rank them
      // there by buckets (the sort when a bucket is too full)
      uint64_t* packed = reinterpret_cast<uint64_t*>(hist);
      if (threadIdx.x == 0) {
        slots[0] = 0xffffffffu;
        slots[1] = 0u;
      }
      __syncthreads();
      uint32_t ulo = 0xffffffffu, uhi = 0u;
      for (uint32_t i = lane; i < wcnt; i += 32) {
        const uint64_t key = wk[i];
        packed[before + i] = key;
        const uint32_t u = static_cast<uint32_t>(key >> 32);
        ulo = u < ulo ? u : ulo;
        uhi = u > uhi ? u : uhi;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint32_t a = __shfl_xor_sync(0xffffffffu, ulo, o), b = __shfl_xor_sync(0xffffffffu, uhi, o);
        ulo = a < ulo ? a : ulo;
        uhi = b > uhi ? b : uhi;
      }
      if (lane == 0) {
        atomicMin(&slots[0], ulo);
        atomicMax(&slots[1], uhi);
      }
      __syncthreads();  // packed and the range are complete; the key buffer is free
      const uint32_t u_lo = slots[0], u_hi = slots[1];
      if (!rank_by_buckets(packed, static_cast<int>(cnt), k, u_lo, u_hi, reinterpret_cast<uint32_t*>(keys),
                           reinterpret_cast<uint16_t*>(reinterpret_cast<uint32_t*>(keys) + TK_NB), warp_tot, sh,
                           out))
        finish_row(packed, static_cast<int>(cnt), k, out);
      return;
    }
    __syncthreads();  // every thread has read warp_tot
  }

  // ---- sweep 1: histogram of the first digit (top TK_BITS1 bits of u)
  for (int i = threadIdx.x; i < TK_BINS; i += TK_THREADS) hist[i] = 0;
  if (threadIdx.x < 2) slots[threadIdx.x] = 0;
  __syncthreads();
  for_runs(row, n, vec, [&](const float (&v)[TK_PER], int64_t) {
#pragma unroll
    for (int e = 0; e < TK_PER; ++e)
      if (v[e] != NEG_INF) atomicAdd(&hist[order_key(v[e]) >> TK_SH1], 1u);
  });
  __syncthreads();
  find_bin(hist, TK_BINS, static_cast<uint32_t>(k), warp_tot, sh);
  const int bin1 = sh[0];
  const bool take_all = bin1 < 0;  // fewer than k candidates: every one is kept
  const uint32_t c_gt1 = take_all ? 0u : static_cast<uint32_t>(sh[1]);
  const uint32_t cnt_b1 = take_all ? static_cast<uint32_t>(sh[2]) : hist[bin1];

  if (c_gt1 + cnt_b1 <= static_cast<uint32_t>(TK_MAXK)) {
    // ---- sweep 2: the keys of the bins above b1 go to [0, c_gt1), those of
    // bin b1 to [c_gt1, c_gt1 + cnt_b1), in any order
    for_runs(row, n, vec, [&](const float (&v)[TK_PER], int64_t i0) {
      uint32_t mgt = 0, meq = 0;
#pragma unroll
      for (int e = 0; e < TK_PER; ++e) {
        if (v[e] == NEG_INF) continue;
        const int d = static_cast<int>(order_key(v[e]) >> TK_SH1);
        if (take_all || d > bin1) mgt |= 1u << e;
        else if (d == bin1) meq |= 1u << e;
      }
      append_keys(v, i0, mgt, keys, &slots[0]);
      append_keys(v, i0, meq, keys + c_gt1, &slots[1]);
    });
    __syncthreads();
    finish_row(keys, static_cast<int>(c_gt1 + cnt_b1), k, out);
    return;
  }

  // ---- heavy ties at the threshold: two more histogram sweeps (10 + 9 bits)
  // inside bin b1 find tau, the k-th largest u
  const int shifts[2] = {9, 0};
  const int nbits[2] = {10, 9};
  uint32_t prefix = static_cast<uint32_t>(bin1), above_total = c_gt1, kk = static_cast<uint32_t>(k) - c_gt1;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int nb = 1 << nbits[pass];
    for (int i = threadIdx.x; i < nb; i += TK_THREADS) hist[i] = 0;
    __syncthreads();
    const int sh_pref = shifts[pass] + nbits[pass];  // bits above this digit
    for_runs(row, n, vec, [&](const float (&v)[TK_PER], int64_t) {
#pragma unroll
      for (int e = 0; e < TK_PER; ++e) {
        if (v[e] == NEG_INF) continue;
        const uint32_t u = order_key(v[e]);
        if ((u >> sh_pref) == prefix) atomicAdd(&hist[(u >> shifts[pass]) & (nb - 1)], 1u);
      }
    });
    __syncthreads();
    find_bin(hist, nb, kk, warp_tot, sh);
    const int bin = sh[0];  // >= 0: bin b1 holds at least kk entries
    above_total += static_cast<uint32_t>(sh[1]);
    kk -= static_cast<uint32_t>(sh[1]);
    prefix = (prefix << nbits[pass]) | static_cast<uint32_t>(bin);
    __syncthreads();
  }
  const uint32_t tau = prefix;
  const uint32_t c_gt = above_total;
  const uint32_t need = kk;  // how many u == tau to keep (lowest indices)

  // ---- ordered selection sweep: thread order is index order; one
  // block-wide exclusive scan of the per-thread counts ranks every kept entry
  uint32_t base_gt = 0, base_eq = 0;
  for_runs(row, n, vec, [&](const float (&v)[TK_PER], int64_t i0) {
    uint32_t uu[TK_PER];
    uint32_t mgt = 0, meq = 0;
#pragma unroll
    for (int e = 0; e < TK_PER; ++e) {
      const bool cand = v[e] != NEG_INF;
      const uint32_t u = cand ? order_key(v[e]) : 0u;
      uu[e] = u;
      if (cand && u > tau) mgt |= 1u << e;
      if (cand && u == tau) meq |= 1u << e;
    }
    // inclusive warp scans of the two counts, packed 16 + 16 bits (each <= 32 * TK_PER)
    const uint32_t mine = (static_cast<uint32_t>(__popc(mgt)) << 16) | static_cast<uint32_t>(__popc(meq));
    uint32_t x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    uint32_t off = x - mine, tot = 0;
    for (int w = 0; w < TK_WARPS; ++w) {
      const uint32_t wt = warp_tot[w];
      if (w < warp) off += wt;
      tot += wt;
    }
    uint32_t og = base_gt + (off >> 16), oe = base_eq + (off & 0xffffu);
#pragma unroll
    for (int e = 0; e < TK_PER; ++e) {
      if (((mgt >> e) & 1u) && og < c_gt) keys[og++] = comp_key(uu[e], static_cast<uint32_t>(i0 + e));
      if ((meq >> e) & 1u) {
        if (oe < need) keys[c_gt + oe] = comp_key(uu[e], static_cast<uint32_t>(i0 + e));
        ++oe;
      }
    }
    base_gt += tot >> 16;
    base_eq += tot & 0xffffu;
    __syncthreads();
  });
  finish_row(keys, k, k, out);
}

// Launches whose rows hold at most 256 entries (the block scores of the QSA
// selection, short sequences): one warp per row, its 32 E keys in registers (E
// per lane) ordered by the warp-level bitonic network (lane shuffles and
// in-register exchanges, no block barrier).  Keys are the same composite keys
// as above, so the order is the same.
template <int E>
__global__ void __launch_bounds__(256) topk_warp_rows_kernel(TopkRows a, int64_t rows) {
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;  // warp-uniform
  const int lane = threadIdx.x & 31;
  const float NEG_INF = __int_as_float(0xff800000);
  const float* row = a.scores + r * a.ld;
  int32_t* out = a.out + r * a.out_ld;
  int64_t n = a.width;
  if (a.mode != 0) {
    const int64_t p = a.p0 + r / a.groups;
    const int64_t c = (a.mode == 1) ? p + 1 : p / a.bs + 1;
    n = c < n ? c : n;
  }
  uint64_t v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = 32 * e + lane;
    uint64_t key = 0;
    if (i < n) {
      const float sc = row[i];
      if (sc != NEG_INF) key = comp_key(order_key(sc), static_cast<uint32_t>(i));
    }
    v[e] = key;
  }
  for (int size = 2; size <= 32 * E; size <<= 1) bitonic_reg_steps<E>(v, 0, size, size >> 1);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = 32 * e + lane;
    if (j < a.k) out[j] = v[e] ? static_cast<int32_t>(~static_cast<uint32_t>(v[e] & 0xffffffffull)) : -1;
  }
  for (int j = 32 * E + lane; j < a.k; j += 32) out[j] = -1;
}

cudaError_t launch_topk_rows(const TopkRows& a, int64_t rows, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (a.width <= 256) {
    const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
    auto kern = a.width <= 32 ? topk_warp_rows_kernel<1>
                : a.width <= 64 ? topk_warp_rows_kernel<2>
                : a.width <= 128 ? topk_warp_rows_kernel<4> : topk_warp_rows_kernel<8>;
    kern<<<grid, 256, 0, stream>>>(a, rows);
    note_launch();
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TK_SMEM);
  if (e != cudaSuccess) return e;
  // the whole shared-memory carveout: the rows of one chunk run beside the
  // indexer's persistent CTAs of the next
  e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  topk_rows_kernel<<<static_cast<unsigned>(rows), TK_THREADS, TK_SMEM, stream>>>(a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tsa
