// Ranking order of finished top-k rows (DSA_FLAG_SORT_BY_SCORE): score
// descending, index ascending, the order of the repeated-varlen-ends rows in
// PR #8403's review ("Preservation and acceptance").  A pass over the rows
// the fused kernel wrote, so the fused kernel itself is the same in either
// order.  One CTA of 128 threads per row (grid-stride).  The row's rankable
// prefix (valid entries with a finite score; KPool tail tokens, scored +INF,
// stay last) arrives in ascending index order, so a stable sort on the
// order-preserving 32-bit score key alone gives the ranking: a block radix
// sort, least significant 4-bit digit first, E entries a thread, skipping
// the digits on which every entry agrees.  Per digit: each thread counts its
// entries in its own column of a digit-major counter table, one block scan
// turns the counts into destinations, and the entries are scattered through
// shared memory (slot index padded by one per 32, conflict-free).  Indices
// are below 65536 in every mode, and the fused kernel writes canonical scores
// (-0 as +0), so the round trip through the key is exact.
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_params.h"

namespace dsa {
namespace {

constexpr int kRankThreads = 128;
constexpr int kRankMaxSlots = 2048;   // index_topk <= 2048 entries carry a finite score
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

struct RankSmem {
  uint32_t key[kRankMaxSlots + kRankMaxSlots / 32];
  uint16_t idx[kRankMaxSlots + kRankMaxSlots / 32];
  uint32_t cnt[kDigits * kRankThreads + kDigits * kRankThreads / 32];   // digit-major, padded
  uint32_t red[8];
  int n;
};

// Sorts entries 0 .. n-1 of sm (padded slots; entries n .. 128E-1 hold key 0,
// index 0xFFFF) by key descending, stably.  Thread t holds entries tE .. tE+E-1.
template <int E>
__device__ __forceinline__ void rank_sort(RankSmem& sm, int n, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t key[E], idx[E];
  uint32_t vor = 0u, vand = 0xFFFFFFFFu;   // over the real entries only
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
    sm.red[4 + warp] = vand;
  }
  __syncthreads();
  const uint32_t vary = (sm.red[0] | sm.red[1] | sm.red[2] | sm.red[3]) ^
                        (sm.red[4] & sm.red[5] & sm.red[6] & sm.red[7]);
  __syncthreads();   // red is reused by the scans
#pragma unroll 1
  for (int shift = 0; shift < 32; shift += 4) {
    if (((vary >> shift) & 0xFu) == 0u) continue;   // every entry has the same digit: order kept
    // 1. count: digit' = 15 - digit (descending keys), rank among this thread's earlier entries
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

__global__ void __launch_bounds__(kRankThreads) rank_rows_kernel(int32_t* idx, float* score, int64_t rows,
                                                                  int width) {
  __shared__ RankSmem sm;
  const int tid = threadIdx.x;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    int32_t* ri = idx + r * width;
    float* rs = score + r * width;
    if (tid == 0) sm.n = 0;
    __syncthreads();
    // the rankable entries are a prefix of the row: valid (index >= 0) with a finite score
    int last = 0;
    for (int g = tid; g < width; g += kRankThreads)
      if (ri[g] >= 0 && rs[g] != __int_as_float(0x7f800000)) last = g + 1;
    if (last > 0) atomicMax(&sm.n, last);
    __syncthreads();
    const int n = sm.n < kRankMaxSlots ? sm.n : kRankMaxSlots;
    if (n > 1) {
      int np = kRankThreads;
      while (np < n) np <<= 1;
      for (int g = tid; g < np; g += kRankThreads) {
        sm.key[padded(g)] = g < n ? score_key(rs[g]) : 0u;
        sm.idx[padded(g)] = g < n ? (uint16_t)ri[g] : (uint16_t)0xFFFFu;
      }
      __syncthreads();
      switch (np / kRankThreads) {
        case 1: rank_sort<1>(sm, n, tid); break;
        case 2: rank_sort<2>(sm, n, tid); break;
        case 4: rank_sort<4>(sm, n, tid); break;
        case 8: rank_sort<8>(sm, n, tid); break;
        default: rank_sort<16>(sm, n, tid); break;
      }
      for (int g = tid; g < n; g += kRankThreads) {
        ri[g] = (int32_t)sm.idx[padded(g)];
        rs[g] = key_score(sm.key[padded(g)]);
      }
    }
    __syncthreads();   // n and the slots are reused by the next row
  }
}

}  // namespace

cudaError_t launch_rank_rows(int32_t* idx, float* score, int64_t rows, int width, int sm_count,
                             cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  int64_t grid = (int64_t)sm_count * 8;
  if (grid > rows) grid = rows;
  rank_rows_kernel<<<(unsigned)grid, kRankThreads, 0, stream>>>(idx, score, rows, width);
  return cudaGetLastError();
}

}  // namespace dsa
