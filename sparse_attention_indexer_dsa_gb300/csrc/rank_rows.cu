// Ranking order of finished top-k rows (DSA_FLAG_SORT_BY_SCORE): score
// descending, index ascending, the order of the repeated-varlen-ends rows in
// PR #8403's review ("Preservation and acceptance").  A pass over the rows
// the fused kernel wrote, so the fused kernel itself is the same in either
// order.  One CTA of 128 threads per row of up to 2048 units, 256 threads up
// to 4096 (grid-stride).  The row's rankable
// prefix (valid entries with a finite score; KPool tail tokens, scored +INF,
// stay last) arrives in ascending index order, so a stable sort on the
// order-preserving 32-bit score key alone gives the ranking: a block radix
// sort, least significant 4-bit digit first, E units a thread, skipping the
// digits on which every unit agrees.  In KPool mode the unit is a pool (its
// P consecutive tokens share one score and move together), so rows of up to
// 4096 pools rank at pool granularity.  Per digit: each thread counts its
// units in its own column of a digit-major counter table, one block scan
// turns the counts into destinations, and the units
// are scattered through shared memory (slot index padded by one per 32,
// conflict-free).  Indices are below 65536 in every mode, and the fused
// kernel writes canonical scores (-0 as +0), so the round trip through the
// key is exact.
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_params.h"

namespace dsa {
namespace {

constexpr int kRankMaxUnits = 4096;   // index_topk <= 4096 (KPool: pools) carry a finite score
constexpr int kDigits = 16;           // 4-bit digits

__device__ __forceinline__ int padded(int g) { return g + (g >> 5); }

__device__ __forceinline__ uint32_t score_key(float v) {
  uint32_t b = __float_as_uint(v);
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// NT threads rank up to 16 * NT units (128 threads up to 2048, 256 up to 4096:
// the smaller block keeps more rows in flight per SM).
template <int NT>
struct RankSmem {
  static constexpr int kUnits = 16 * NT;
  uint32_t key[kUnits + kUnits / 32];
  uint16_t idx[kUnits + kUnits / 32];
  uint32_t cnt[kDigits * NT + kDigits * NT / 32];   // digit-major, padded
  uint32_t red[2 * (NT / 32)];
  int n;
};

// Sorts units 0 .. n-1 of sm (padded slots; units n .. 256E-1 hold key 0,
// index 0xFFFF) by key descending, stably.  Thread t holds units tE .. tE+E-1.
template <int NT, int E>
__device__ __forceinline__ void rank_sort(RankSmem<NT>& sm, int n, int tid) {
  constexpr int kRankThreads = NT, kRankWarps = NT / 32;
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
    sm.red[warp] = vor;
    sm.red[kRankWarps + warp] = vand;
  }
  __syncthreads();
  uint32_t all_or = 0u, all_and = 0xFFFFFFFFu;
#pragma unroll
  for (int w = 0; w < kRankWarps; ++w) {
    all_or |= sm.red[w];
    all_and &= sm.red[kRankWarps + w];
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
    if (lane == 31) sm.red[warp] = incl;
    __syncthreads();
    uint32_t base = incl - tot;
    for (int w = 0; w < warp; ++w) base += sm.red[w];
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

// One row per CTA iteration.  A unit is `group` consecutive entries with one
// score: a single entry (group 1), or one KPool pool whose tokens are
// consecutive (group = pool size); units move as a whole, so a pool's tokens
// stay together and ascending.
template <int NT, int E>
__global__ void __launch_bounds__(NT) rank_rows_kernel(int32_t* idx, float* score, int64_t rows, int width,
                                                       int group) {
  constexpr int kRankThreads = NT;
  __shared__ RankSmem<NT> sm;
  const int tid = threadIdx.x;
  const int nu_max = min((width + group - 1) / group, RankSmem<NT>::kUnits);
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    int32_t* ri = idx + r * width;
    float* rs = score + r * width;
    if (tid == 0) sm.n = 0;
    __syncthreads();
    // the rankable units are a prefix of the row: valid (index >= 0) with a finite score;
    // every load of the row is issued before any is used
    int32_t li[E];
    float ls[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int u = e * kRankThreads + tid;
      li[e] = u < nu_max ? ri[(size_t)u * group] : -1;
      ls[e] = u < nu_max ? rs[(size_t)u * group] : 0.f;
    }
    int last = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int u = e * kRankThreads + tid;
      if (li[e] >= 0 && ls[e] != __int_as_float(0x7f800000)) last = u + 1;
    }
    if (last > 0) atomicMax(&sm.n, last);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int g = e * kRankThreads + tid;
      sm.key[padded(g)] = li[e] >= 0 ? score_key(ls[e]) : 0u;
      sm.idx[padded(g)] = li[e] >= 0 ? (uint16_t)li[e] : (uint16_t)0xFFFFu;
    }
    __syncthreads();
    const int n = sm.n;
    if (n > 1) {
      // units n .. 256E-1 (padding, +INF tail) sort after every real unit
      for (int g = n + tid; g < E * kRankThreads; g += kRankThreads) {
        sm.key[padded(g)] = 0u;
        sm.idx[padded(g)] = (uint16_t)0xFFFFu;
      }
      __syncthreads();
      rank_sort<NT, E>(sm, n, tid);
      for (int g = tid; g < n * group; g += kRankThreads) {
        const int u = g / group;
        ri[g] = (int32_t)sm.idx[padded(u)] + (g - u * group);
        rs[g] = key_score(sm.key[padded(u)]);
      }
    }
    __syncthreads();   // n and the slots are reused by the next row
  }
}

template <int NT, int E>
cudaError_t launch_e(int32_t* idx, float* score, int64_t rows, int width, int group, int sm_count,
                     cudaStream_t stream) {
  int64_t grid = (int64_t)sm_count * 8;
  if (grid > rows) grid = rows;
  rank_rows_kernel<NT, E><<<(unsigned)grid, NT, 0, stream>>>(idx, score, rows, width, group);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rank_rows(int32_t* idx, float* score, int64_t rows, int width, int group, int sm_count,
                             cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  // at most kRankMaxUnits units are rankable (the API keeps at most 4096 keys or
  // pools per row); a KPool tail beyond them is never ranked and stays in place
  int units = (width + group - 1) / group;
  if (units > kRankMaxUnits) units = kRankMaxUnits;
  if (units <= 128) return launch_e<128, 1>(idx, score, rows, width, group, sm_count, stream);
  if (units <= 256) return launch_e<128, 2>(idx, score, rows, width, group, sm_count, stream);
  if (units <= 512) return launch_e<128, 4>(idx, score, rows, width, group, sm_count, stream);
  if (units <= 1024) return launch_e<128, 8>(idx, score, rows, width, group, sm_count, stream);
  if (units <= 2048) return launch_e<128, 16>(idx, score, rows, width, group, sm_count, stream);
  return launch_e<256, 16>(idx, score, rows, width, group, sm_count, stream);
}

}  // namespace dsa
