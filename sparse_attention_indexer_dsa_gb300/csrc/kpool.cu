// KPool key compression for sm_103a (Megatron-LM PR #7522 "KPool (pooled-key)
// DSA indexer support", "Changes"): in each document, every complete group of
// P consecutive keys becomes sum_i softmax_i(gate_i + bias_i) * k_i (softmax
// over the P slots in FP32, BF16 gate, FP32 per-slot bias), stored as BF16.
// Pooling restarts at document boundaries; a trailing incomplete group is not
// pooled.  HBM-bound: one warp per pool, 128-bit loads (FP32 keys), the pool's
// P rows requested together.
#include <cuda_bf16.h>

#include "dsa_device.cuh"
#include "dsa_params.h"

namespace dsa {

// cu_pools[d] = sum over earlier documents of floor(L / P); one block.
__global__ void __launch_bounds__(1024) kpool_cu_kernel(const int32_t* __restrict__ cu, int num_seqs,
                                                       int P, int32_t* __restrict__ cu_pools) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x;
  int carry = 0;
  for (int base = 0; base < num_seqs; base += 1024) {
    const int d = base + tid;
    const int v = d < num_seqs ? (cu[d + 1] - cu[d]) / P : 0;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if ((tid & 31) >= o) x += y;
    }
    if ((tid & 31) == 31) warp_tot[tid >> 5] = x;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < (tid >> 5); ++w) before += warp_tot[w];
    if (d < num_seqs) cu_pools[d] = carry + before + x - v;
    int tot = 0;
    for (int w = 0; w < 32; ++w) tot += warp_tot[w];
    __syncthreads();
    carry += tot;
  }
  if (tid == 0) cu_pools[num_seqs] = carry;
}

// Loads one key row slice (VEC values of lane `lane`) as FP32.
template <int VEC>
__device__ __forceinline__ void load_key(const void* k, int k_bf16, size_t row, float (&x)[VEC]) {
  if (k_bf16) {
    const uint16_t* kp = reinterpret_cast<const uint16_t*>(k) + row;
    if constexpr (VEC == 4) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(kp));
      x[0] = __uint_as_float(u.x << 16);
      x[1] = __uint_as_float(u.x & 0xFFFF0000u);
      x[2] = __uint_as_float(u.y << 16);
      x[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
      const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(kp));
      x[0] = __uint_as_float(u << 16);
      x[1] = __uint_as_float(u & 0xFFFF0000u);
    }
  } else {
    const float* kp = reinterpret_cast<const float*>(k) + row;
    if constexpr (VEC == 4) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(kp));
      x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    } else {
      const float2 f = __ldg(reinterpret_cast<const float2*>(kp));
      x[0] = f.x; x[1] = f.y;
    }
  }
}

// One warp per pool; the pool's P key rows are all requested before the gate
// softmax is formed, so P loads per lane are in flight at once.  Eight
// resident blocks per SM (32 registers) for P <= 4 keep enough bytes in
// flight (measured 79 % of the copy bandwidth against 74 % at four); P = 8
// holds twice the rows and stays at four.
template <int VEC, int P>
__global__ void __launch_bounds__(256, P <= 4 ? 8 : 4) kpool_compress_kernel(
    const void* __restrict__ k, int k_bf16, const uint16_t* __restrict__ gate,
    const float* __restrict__ bias, const int32_t* __restrict__ cu,
    const int32_t* __restrict__ cu_pools, int num_seqs, int max_pools,
    uint16_t* __restrict__ out) {
  constexpr int D = VEC * 32;
  const int lane = threadIdx.x & 31;
  const int total = cu_pools[num_seqs];
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int pi = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pi < total && pi < max_pools;
       pi += nwarps) {
    int lo = 0, hi = num_seqs - 1;   // document of pool pi
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu_pools[mid] <= pi) lo = mid; else hi = mid - 1;
    }
    const int tok0 = cu[lo] + (pi - cu_pools[lo]) * P;
    float x[P][VEC];
#pragma unroll
    for (int i = 0; i < P; ++i) load_key<VEC>(k, k_bf16, (size_t)(tok0 + i) * D + lane * VEC, x[i]);
    float logit[P];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < P; ++i) {
      logit[i] = __uint_as_float((uint32_t)__ldg(gate + tok0 + i) << 16) + __ldg(bias + i);
      mx = fmaxf(mx, logit[i]);
    }
    float den = 0.f;
#pragma unroll
    for (int i = 0; i < P; ++i) {
      logit[i] = expf(logit[i] - mx);
      den += logit[i];
    }
    float acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const float wgt = logit[i] / den;
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] = fmaf(wgt, x[i][e], acc[e]);
    }
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out) + (size_t)pi * D + lane * VEC;
#pragma unroll
    for (int e = 0; e < VEC; e += 2) *reinterpret_cast<__nv_bfloat162*>(o + e) = __floats2bfloat162_rn(acc[e], acc[e + 1]);
  }
}

template <int VEC, int P>
static void launch_kpool_p(const void* k, int k_bf16, const uint16_t* gate, const float* bias, const int32_t* cu,
                           int num_seqs, int max_pools, uint16_t* out, const int32_t* cu_pools, int blocks,
                           cudaStream_t stream) {
  kpool_compress_kernel<VEC, P><<<blocks, 256, 0, stream>>>(k, k_bf16, gate, bias, cu, cu_pools, num_seqs,
                                                            max_pools, out);
}

template <int VEC>
static void launch_kpool_v(const void* k, int k_bf16, const uint16_t* gate, const float* bias, const int32_t* cu,
                           int num_seqs, int max_pools, int P, uint16_t* out, const int32_t* cu_pools, int blocks,
                           cudaStream_t stream) {
  if (P == 2) launch_kpool_p<VEC, 2>(k, k_bf16, gate, bias, cu, num_seqs, max_pools, out, cu_pools, blocks, stream);
  else if (P == 4) launch_kpool_p<VEC, 4>(k, k_bf16, gate, bias, cu, num_seqs, max_pools, out, cu_pools, blocks, stream);
  else launch_kpool_p<VEC, 8>(k, k_bf16, gate, bias, cu, num_seqs, max_pools, out, cu_pools, blocks, stream);
}

cudaError_t launch_kpool(const void* k, int k_bf16, const uint16_t* gate, const float* bias,
                         const int32_t* cu, int num_seqs, int total_tokens, int D, int P,
                         uint16_t* out, int32_t* cu_pools, int sm_count, cudaStream_t stream) {
  kpool_cu_kernel<<<1, 1024, 0, stream>>>(cu, num_seqs, P, cu_pools);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int max_pools = total_tokens / P;
  if (max_pools == 0) return cudaSuccess;
  int blocks = (max_pools + 7) / 8;
  if (blocks > sm_count * 8) blocks = sm_count * 8;
  if (D == 128)
    launch_kpool_v<4>(k, k_bf16, gate, bias, cu, num_seqs, max_pools, P, out, cu_pools, blocks, stream);
  else
    launch_kpool_v<2>(k, k_bf16, gate, bias, cu, num_seqs, max_pools, P, out, cu_pools, blocks, stream);
  return cudaGetLastError();
}

}  // namespace dsa
