// Ranking order of finished top-k rows (DSA_FLAG_SORT_BY_SCORE): score
// descending, index ascending, the order of the repeated-varlen-ends rows in
// PR #8403's review ("Preservation and acceptance").  A pass over the rows
// the fused kernel wrote, so the fused kernel itself is the same in either
// order.  One 256-thread CTA per row (grid-stride), E units a thread.  The
// row's rankable prefix (valid entries with a finite score; KPool tail
// tokens, scored +INF, stay last) arrives in ascending index order.  In KPool
// mode the unit is a pool (its P consecutive tokens share one score and move
// together), so rows of up to 4096 pools rank at pool granularity.
//
// Bucket rank (the common case): every unit is put in one of U buckets by a
// monotone map of its score, so a unit's final position is the number of
// units in higher buckets plus the number of units of its own bucket that
// rank before it (higher score, or equal score and lower index), counted by
// comparing it with each member.  The map is linear near zero and
// logarithmic further out: f(v) = sign(v) * (bits(c + |v|) - bits(c)), with
// bits() the IEEE pattern of a positive float and c = (max - min) / 64, then
// scaled to the bucket range by a fixed-point multiply; every step is a
// rounded float add, an integer difference or a multiply by a positive
// constant, each monotone, so the map never reorders two scores.  One pass
// over shared memory: count (shared atomics give each unit a slot in its
// bucket), scan, scatter into bucket order, then place: each thread takes
// staged positions, so the lanes of a warp hold neighbouring buckets (their
// member loads broadcast and their loop counts agree), counts the members of
// the position's bucket that rank before it, and writes the unit to its final
// place (single entries straight into the output row, whose writes then fall
// on neighbouring addresses).
//
// Radix rank (the fallback, for rows whose largest bucket holds more than
// kBucketCap units: many tied scores, or a distribution the map does not
// spread): a stable block radix sort on the order-preserving 32-bit score key,
// least significant 4-bit digit first, skipping the digits on which every
// unit agrees; a stable sort of the index-ordered prefix on the score alone
// gives the ranking.  Per digit: each thread counts its units in its own
// column of a digit-major counter table, one block scan turns the counts into
// destinations, and the units are scattered through shared memory (slot
// index padded by one per 32, conflict-free).
//
// Indices are below 65536 in every mode, and the fused kernel writes
// canonical scores (-0 as +0), so the round trip through the key is exact.
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_params.h"

namespace dsa {
namespace {

constexpr int kRankMaxUnits = 4096;   // index_topk <= 4096 (KPool: pools) carry a finite score
constexpr int kRankThreads = 256;
constexpr int kRankWarps = kRankThreads / 32;
constexpr int kDigits = 16;           // 4-bit digits of the radix fallback
constexpr int kBucketCap = 64;        // larger bucket: the row takes the radix fallback
constexpr int kBucketsPerUnit = 1;   // buckets per rankable unit

__device__ __forceinline__ int padded(int g) { return g + (g >> 5); }

__device__ __forceinline__ uint32_t score_key(float v) {
  uint32_t b = __float_as_uint(v);
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// the monotone bucket map's first stage: sign(v) * (bits(c + |v|) - bits(c))
// (two's complement, so differences of coordinates are taken as uint32)
__device__ __forceinline__ uint32_t bucket_coord(float v, float c, uint32_t bits_c) {
  const uint32_t h = __float_as_uint(__fadd_rn(c, fabsf(v))) - bits_c;   // < 2^31
  return v >= 0.f ? h : 0u - h;
}

// Units of the radix fallback (slot index padded by one per 32).
template <int U>
struct RadixSmem {
  uint32_t key[U + U / 32];
  uint16_t idx[U + U / 32];
  uint32_t cnt[kDigits * kRankThreads + kDigits * kRankThreads / 32];   // digit-major, padded
};

template <int U>
struct BucketSmem {
  static constexpr int kBuckets = U * kBucketsPerUnit;
  uint64_t stage[U];   // units grouped by bucket: key << 32 | ~index (larger ranks first)
  uint64_t fin[U];     // units in ranking order (KPool pools; single entries go straight to the row)
  uint32_t cnt[kBuckets + kBuckets / 32];   // bucket counters, then start | count << 13 (padded)
  uint16_t bkt[U];     // bucket of each staged unit
};

template <int U>
union RankSmem {
  BucketSmem<U> b;
  RadixSmem<U> r;
};

// Sorts units 0 .. n-1 of sm (padded slots; units n .. U-1 hold key 0, index
// 0xFFFF) by key descending, stably.  Thread t holds units tE .. tE+E-1.
// `red` holds 2 * kRankWarps words.
template <int E>
__device__ __forceinline__ void radix_rank(RadixSmem<kRankThreads * E>& sm, uint32_t* red, int n, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t key[E], idx[E];
  uint32_t vor = 0u, vand = 0xFFFFFFFFu;   // over the real units only
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int g = tid * E + e;
    key[e] = sm.key[padded(g)];
    idx[e] = sm.idx[padded(g)];
    if (g < n) {
      vor |= key[e];
      vand &= key[e];
    }
  }
  vor = __reduce_or_sync(0xffffffffu, vor);
  vand = __reduce_and_sync(0xffffffffu, vand);
  if (lane == 0) {
    red[warp] = vor;
    red[kRankWarps + warp] = vand;
  }
  __syncthreads();
  uint32_t all_or = 0u, all_and = 0xFFFFFFFFu;
#pragma unroll
  for (int w = 0; w < kRankWarps; ++w) {
    all_or |= red[w];
    all_and &= red[kRankWarps + w];
  }
  const uint32_t vary = all_or ^ all_and;
  __syncthreads();   // red is reused by the scans
#pragma unroll 1
  for (int shift = 0; shift < 32; shift += 4) {
    if (((vary >> shift) & 0xFu) == 0u) continue;   // every unit has the same digit: order kept
    // 1. count: digit' = 15 - digit (descending keys), rank among this thread's earlier units
#pragma unroll
    for (int d = 0; d < kDigits; ++d) sm.cnt[padded(d * kRankThreads + tid)] = 0u;
    uint32_t dg[E], rk[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      dg[e] = 15u - ((key[e] >> shift) & 0xFu);
      const int c = padded((int)dg[e] * kRankThreads + tid);
      rk[e] = sm.cnt[c];
      sm.cnt[c] = rk[e] + 1u;
    }
    __syncthreads();
    // 2. exclusive scan of the counters in digit-major order; thread t owns
    //    linear positions 16t .. 16t+15
    uint32_t v[kDigits], tot = 0u;
#pragma unroll
    for (int i = 0; i < kDigits; ++i) {
      v[i] = sm.cnt[padded(kDigits * tid + i)];
      tot += v[i];
    }
    uint32_t incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    uint32_t base = incl - tot;
    for (int w = 0; w < warp; ++w) base += red[w];
#pragma unroll
    for (int i = 0; i < kDigits; ++i) {
      sm.cnt[padded(kDigits * tid + i)] = base;
      base += v[i];
    }
    __syncthreads();
    // 3. scatter to the destinations, then reload in thread order
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int dst = (int)(sm.cnt[padded((int)dg[e] * kRankThreads + tid)] + rk[e]);
      sm.key[padded(dst)] = key[e];
      sm.idx[padded(dst)] = (uint16_t)idx[e];
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) {
      key[e] = sm.key[padded(tid * E + e)];
      idx[e] = sm.idx[padded(tid * E + e)];
    }
    __syncthreads();   // every reload (and every read of cnt) before the next digit's writes
  }
}

// The bucket rank of one row (n > 1 units, not all one score).  Returns
// false, having moved nothing, when a bucket holds more than kBucketCap units.
// FULL: every one of the U units is rankable (n == U), so no unit needs the
// n bound.
template <int E, bool SINGLE, bool FULL>
__device__ __forceinline__ bool bucket_rank(RankSmem<kRankThreads * E>& sm, uint32_t (&red)[4][kRankWarps],
                                            const int32_t (&li)[E], const float (&ls)[E], int n, int group,
                                            uint32_t kmin, uint32_t kmax, int32_t* ri, float* rs, int tid) {
  constexpr int U = kRankThreads * E;
  constexpr int EB = E * kBucketsPerUnit;
  constexpr int NB = U * kBucketsPerUnit;
  const int lane = tid & 31, warp = tid >> 5;
  // the bucket map, the same in every thread; a multiplier at or below
  // NB * 2^32 / (range + 1) keeps every bucket below NB (float estimate
  // scaled down by more than its rounding error)
  const float vmin = key_score(kmin), vmax = key_score(kmax);
  const float c = __fmul_rn(__fsub_rn(vmax, vmin), 1.0f / 64.0f);
  const uint32_t bits_c = __float_as_uint(c);
  const uint32_t lo = bucket_coord(vmin, c, bits_c);
  const uint32_t range = bucket_coord(vmax, c, bits_c) - lo;
  const uint32_t mul =
      range < (uint32_t)NB
          ? 0u
          : __float2uint_rz(__fdiv_rn((float)NB * 4294967296.0f * (1.0f - 1.0f / 1048576.0f),
                                      __fadd_ru(__uint2float_ru(range), 1.0f)));
  // per unit: its bucket | slot in the bucket << 16
  uint32_t bs[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int u = e * kRankThreads + tid;
    if (FULL || u < n) {
      const uint32_t x = bucket_coord(ls[e], c, bits_c) - lo;   // -0 and +0 alike
      const uint32_t b = mul == 0u ? x : __umulhi(x, mul);
      bs[e] = b | (atomicAdd(&sm.b.cnt[padded((int)b)], 1u) << 16);
    }
  }
  __syncthreads();
  // bucket starts in ranking order: start[b] = n - (counts of buckets 0..b);
  // thread t owns buckets t*EB .. t*EB+EB-1 (padded slots: conflict-free)
  uint32_t tot = 0u, cmax = 0u;
#pragma unroll
  for (int i = 0; i < EB; ++i) {
    const uint32_t cv = sm.b.cnt[padded(tid * EB + i)];
    tot += cv;
    cmax = max(cmax, cv);
  }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  cmax = __reduce_max_sync(0xffffffffu, cmax);
  if (lane == 31) red[3][warp] = incl;
  if (lane == 0) red[0][warp] = cmax;   // red[0] was last read before the previous barrier
  __syncthreads();
  uint32_t before = incl - tot, big = 0u;
#pragma unroll
  for (int w = 0; w < kRankWarps; ++w) {
    if (w < warp) before += red[3][w];
    big = max(big, red[0][w]);
  }
  if (big > (uint32_t)kBucketCap) return false;   // the radix fallback ranks this row
#pragma unroll
  for (int i = 0; i < EB; ++i) {   // the counts again (unchanged since they were summed)
    const uint32_t cv = sm.b.cnt[padded(tid * EB + i)];
    before += cv;
    sm.b.cnt[padded(tid * EB + i)] = ((uint32_t)n - before) | (cv << 13);
  }
  __syncthreads();
  // scatter into bucket order (count <= kBucketCap < 2^7, start < 2^13)
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int u = e * kRankThreads + tid;
    if (FULL || u < n) {
      const uint32_t bv = sm.b.cnt[padded((int)(bs[e] & 0xFFFFu))];
      const uint32_t slot = bs[e] >> 16;
      const uint32_t at = (bv & 0x1FFFu) + slot;
      sm.b.stage[at] = ((uint64_t)score_key(ls[e]) << 32) | (uint32_t)~(uint32_t)li[e];
      sm.b.bkt[at] = (uint16_t)(bs[e] & 0xFFFFu);
    }
  }
  __syncthreads();
  // final position: the bucket's start plus the members that rank before the
  // unit, taken over staged positions (a warp's lanes hold neighbouring buckets)
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int p = e * kRankThreads + tid;
    if (FULL || p < n) {
      const uint64_t pk = sm.b.stage[p];
      const uint32_t bv = sm.b.cnt[padded((int)sm.b.bkt[p])];
      const uint32_t st = bv & 0x1FFFu, m = (bv >> 13) & 0x7Fu;
      uint32_t pos = st;
      if (m > 1u)
        for (uint32_t j = 0; j < m; ++j) pos += sm.b.stage[st + j] > pk ? 1u : 0u;
      if (SINGLE) {   // the row's loads were all taken before the first barrier
        ri[pos] = (int32_t)~(uint32_t)pk;
        rs[pos] = key_score((uint32_t)(pk >> 32));
      } else {
        sm.b.fin[pos] = pk;
      }
    }
  }
  __syncthreads();   // every read of the counters and the stage before they are reused
  if (!SINGLE) {
    for (int g = tid; g < n * group; g += kRankThreads) {
      const int u = g / group;
      const uint64_t v = sm.b.fin[u];
      ri[g] = (int32_t)~(uint32_t)v + (g - u * group);
      rs[g] = key_score((uint32_t)(v >> 32));
    }
  }
  // the counters are zero again for the next row (read for the last time above)
#pragma unroll
  for (int i = 0; i < EB; ++i) sm.b.cnt[padded(tid * EB + i)] = 0u;
  return true;
}

// One row per CTA iteration.  A unit is `group` consecutive entries with one
// score: a single entry (group 1, SINGLE), or one KPool pool whose tokens are
// consecutive (group = pool size); units move as a whole, so a pool's tokens
// stay together and ascending.  Units are striped: unit u = e * 256 + thread.
template <int E, bool SINGLE>
__global__ void __launch_bounds__(kRankThreads, E <= 8 ? 4 : 2)
    rank_rows_kernel(int32_t* idx, float* score, int64_t rows, int width, int group) {
  constexpr int U = kRankThreads * E;
  constexpr int EB = E * kBucketsPerUnit;   // buckets a thread owns in the scan
  extern __shared__ __align__(16) unsigned char rank_smem_raw[];
  RankSmem<U>& sm = *reinterpret_cast<RankSmem<U>*>(rank_smem_raw);
  __shared__ uint32_t red[4][kRankWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (SINGLE) group = 1;
  const int nu_max = min((width + group - 1) / group, U);
#pragma unroll
  for (int i = 0; i < EB; ++i) sm.b.cnt[padded(tid * EB + i)] = 0u;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    int32_t* ri = idx + r * width;
    float* rs = score + r * width;
    // the rankable units are a prefix of the row: valid (index >= 0) with a finite score;
    // every load of the row is issued before any is used
    int32_t li[E];
    float ls[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int u = e * kRankThreads + tid;
      const size_t off = SINGLE ? (size_t)u : (size_t)u * group;
      li[e] = u < nu_max ? ri[off] : -1;
      ls[e] = u < nu_max ? rs[off] : 0.f;
    }
    uint32_t last = 0u, kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint32_t key = score_key(ls[e]);
      if (li[e] >= 0 && ls[e] != __int_as_float(0x7f800000)) {
        last = (uint32_t)(e * kRankThreads + tid) + 1u;
        kmin = min(kmin, key);
        kmax = max(kmax, key);
      }
    }
    last = __reduce_max_sync(0xffffffffu, last);
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0) {
      red[0][warp] = last;
      red[1][warp] = kmin;
      red[2][warp] = kmax;
    }
    __syncthreads();
    int n = 0;
    kmin = 0xFFFFFFFFu;
    kmax = 0u;
#pragma unroll
    for (int w = 0; w < kRankWarps; ++w) {
      n = max(n, (int)red[0][w]);
      kmin = min(kmin, red[1][w]);
      kmax = max(kmax, red[2][w]);
    }
    // one unit, or one score for all: the index order is the ranking
    if (n <= 1 || kmin == kmax) {
      __syncthreads();   // every read of red before the next row writes it
      continue;
    }
    const bool ranked = n == U ? bucket_rank<E, SINGLE, true>(sm, red, li, ls, n, group, kmin, kmax, ri, rs, tid)
                               : bucket_rank<E, SINGLE, false>(sm, red, li, ls, n, group, kmin, kmax, ri, rs, tid);
    if (!ranked) {
      // radix fallback over the same smem (the counters were read before the last barrier)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int g = e * kRankThreads + tid;
        const bool real = g < n;
        sm.r.key[padded(g)] = real ? score_key(ls[e]) : 0u;
        sm.r.idx[padded(g)] = real ? (uint16_t)li[e] : (uint16_t)0xFFFFu;
      }
      __syncthreads();
      radix_rank<E>(sm.r, &red[0][0], n, tid);
      for (int g = tid; g < n * group; g += kRankThreads) {
        const int u = g / group;
        ri[g] = (int32_t)sm.r.idx[padded(u)] + (g - u * group);
        rs[g] = key_score(sm.r.key[padded(u)]);
      }
      __syncthreads();   // every read of the units before the counters (same smem) are cleared
#pragma unroll
      for (int i = 0; i < EB; ++i) sm.b.cnt[padded(tid * EB + i)] = 0u;
    }
  }
}

template <int E, bool SINGLE>
cudaError_t launch_es(int32_t* idx, float* score, int64_t rows, int width, int group, int sm_count,
                      cudaStream_t stream) {
  constexpr int U = kRankThreads * E;
  const size_t smem = sizeof(RankSmem<U>);
  cudaError_t e = cudaFuncSetAttribute(rank_rows_kernel<E, SINGLE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rank_rows_kernel<E, SINGLE>, kRankThreads, smem);
  if (e != cudaSuccess) return e;
  int64_t grid = (int64_t)sm_count * (per_sm > 0 ? per_sm : 1);
  if (grid > rows) grid = rows;
  rank_rows_kernel<E, SINGLE><<<(unsigned)grid, kRankThreads, smem, stream>>>(idx, score, rows, width, group);
  return cudaGetLastError();
}

template <int E>
cudaError_t launch_e(int32_t* idx, float* score, int64_t rows, int width, int group, int sm_count,
                     cudaStream_t stream) {
  return group == 1 ? launch_es<E, true>(idx, score, rows, width, group, sm_count, stream)
                    : launch_es<E, false>(idx, score, rows, width, group, sm_count, stream);
}

}  // namespace

cudaError_t launch_rank_rows(int32_t* idx, float* score, int64_t rows, int width, int group, int sm_count,
                             cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  // at most kRankMaxUnits units are rankable (the API keeps at most 4096 keys or
  // pools per row); a KPool tail beyond them is never ranked and stays in place
  int units = (width + group - 1) / group;
  if (units > kRankMaxUnits) units = kRankMaxUnits;
  if (units <= 256) return launch_e<1>(idx, score, rows, width, group, sm_count, stream);
  if (units <= 512) return launch_e<2>(idx, score, rows, width, group, sm_count, stream);
  if (units <= 1024) return launch_e<4>(idx, score, rows, width, group, sm_count, stream);
  if (units <= 2048) return launch_e<8>(idx, score, rows, width, group, sm_count, stream);
  return launch_e<16>(idx, score, rows, width, group, sm_count, stream);
}

}  // namespace dsa
