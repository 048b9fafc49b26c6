// Ranking order of finished top-k rows (DSA_FLAG_SORT_BY_SCORE): score
// descending, index ascending, the order of the repeated-varlen-ends rows in
// PR #8403's review ("Preservation and acceptance").  A pass over the rows
// the fused kernel wrote, so the fused kernel itself is the same in either
// order.  One CTA of 128 threads per row (grid-stride): the row's rankable
// prefix (valid entries with a finite score; KPool tail tokens, scored +INF,
// stay last) is packed as (order-preserving score key << 16) | (0xFFFF -
// index), sorted by a bitonic network held in registers (E consecutive slots
// a thread; pairs closer than E slots in registers, closer than 32 E by warp
// shuffles, the rest through shared memory), and written back.  Indices are
// below 65536 in every mode, and the fused kernel writes canonical scores
// (-0 as +0), so the round trip through the key is exact.  Bandwidth-bound:
// each row is read and written once.
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_params.h"

namespace dsa {
namespace {

constexpr int kRankThreads = 128;
constexpr int kRankMaxSlots = 2048;   // index_topk <= 2048 entries carry a finite score

__device__ __forceinline__ int padded(int g) { return g + (g >> 5); }   // conflict-free strided slots

__device__ __forceinline__ uint32_t score_key(float v) {
  uint32_t b = __float_as_uint(v);
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// One network stage between slots J apart inside a thread (J < E).
template <int J, int E>
__device__ __forceinline__ void stage_in_thread(uint64_t (&c)[E], int tid, int k2) {
  if constexpr (J < E) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if ((e & J) == 0) {
        const bool best_first = ((tid * E + e) & k2) == 0;
        const uint64_t a = c[e], b = c[e | J];
        c[e] = best_first ? umax64(a, b) : umin64(a, b);
        c[e | J] = best_first ? umin64(a, b) : umax64(a, b);
      }
    }
  }
}

// Sorts the NP = 128 E packed entries at padded slots of sm descending, in
// place.  The stage loops stay rolled (a fully unrolled network overflows the
// instruction cache); only the per-slot loops unroll.
template <int E>
__device__ __forceinline__ void rank_sort(uint64_t* sm, int tid) {
  constexpr int NP = kRankThreads * E;
  uint64_t c[E];
#pragma unroll
  for (int e = 0; e < E; ++e) c[e] = sm[padded(tid * E + e)];
  __syncthreads();
#pragma unroll 1
  for (int k2 = 2; k2 <= NP; k2 <<= 1) {
#pragma unroll 1
    for (int j = k2 >> 1; j > 0; j >>= 1) {
      if (j < E) {                                  // both slots in this thread
        switch (j) {
          case 1: stage_in_thread<1, E>(c, tid, k2); break;
          case 2: stage_in_thread<2, E>(c, tid, k2); break;
          case 4: stage_in_thread<4, E>(c, tid, k2); break;
          default: stage_in_thread<8, E>(c, tid, k2); break;
        }
        continue;
      }
      const int m = j / E;                          // partner thread: tid ^ m
      const bool lower = (tid & m) == 0;
      if (j < 32 * E) {                             // same warp
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)c[e], m);
          const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(c[e] >> 32), m);
          const uint64_t o = ((uint64_t)hi << 32) | lo;
          const bool best_first = (((tid * E + e) & ~j) & k2) == 0;
          c[e] = (lower == best_first) ? umax64(c[e], o) : umin64(c[e], o);
        }
      } else {                                      // another warp
#pragma unroll
        for (int e = 0; e < E; ++e) sm[padded(tid * E + e)] = c[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint64_t o = sm[padded((tid * E + e) ^ j)];
          const bool best_first = (((tid * E + e) & ~j) & k2) == 0;
          c[e] = (lower == best_first) ? umax64(c[e], o) : umin64(c[e], o);
        }
        __syncthreads();
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) sm[padded(tid * E + e)] = c[e];
  __syncthreads();
}

__global__ void __launch_bounds__(kRankThreads, 4) rank_rows_kernel(int32_t* idx, float* score, int64_t rows,
                                                                  int width) {
  __shared__ uint64_t sm[kRankMaxSlots + kRankMaxSlots / 32];
  __shared__ int s_n;
  const int tid = threadIdx.x;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    int32_t* ri = idx + r * width;
    float* rs = score + r * width;
    if (tid == 0) s_n = 0;
    __syncthreads();
    // the rankable entries are a prefix of the row: valid (index >= 0) with a finite score
    int last = 0;
    for (int g = tid; g < width; g += kRankThreads)
      if (ri[g] >= 0 && rs[g] != __int_as_float(0x7f800000)) last = g + 1;
    if (last > 0) atomicMax(&s_n, last);
    __syncthreads();
    const int n = s_n < kRankMaxSlots ? s_n : kRankMaxSlots;
    if (n > 1) {
      int np = kRankThreads;
      while (np < n) np <<= 1;
      for (int g = tid; g < np; g += kRankThreads)
        sm[padded(g)] = g < n ? ((uint64_t)score_key(rs[g]) << 16) | (uint64_t)(0xFFFFu - (uint32_t)ri[g]) : 0ull;
      __syncthreads();
      switch (np / kRankThreads) {
        case 1: rank_sort<1>(sm, tid); break;
        case 2: rank_sort<2>(sm, tid); break;
        case 4: rank_sort<4>(sm, tid); break;
        case 8: rank_sort<8>(sm, tid); break;
        default: rank_sort<16>(sm, tid); break;
      }
      for (int g = tid; g < n; g += kRankThreads) {
        const uint64_t v = sm[padded(g)];
        ri[g] = (int32_t)(0xFFFFu - (uint32_t)(v & 0xFFFFu));
        rs[g] = key_score((uint32_t)(v >> 16));
      }
    }
    __syncthreads();   // s_n and sm are reused by the next row
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
