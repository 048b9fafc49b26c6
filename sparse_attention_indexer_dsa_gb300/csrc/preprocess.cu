// Query/key preprocessing and MXFP8 / per-vector FP8 quantisation for sm_103a
// (HBM-bound).
//
// * preprocess_kernel: key LayerNorm -> RoPE -> BF16 or MXFP8, one block per
//   token (its H query rows + its key row), one warp per row, 128-bit loads,
//   warp-shuffle reductions.  Megatron-LM PR #8403 "cuDNN DSA indexer
//   precision options": "What does this PR do?" (dsa_indexer_rope_fp32 keeps
//   the key LayerNorm -> RoPE chain in FP32) and "Motivation" (the default
//   path materialises BF16 between the LayerNorm and RoPE); review finding 2
//   (BF16 scoring rounds FP32 carriers to BF16).  PR #7522 "Changes": NoPE
//   (rope_dim = 0).  PR #5992 "Key changes": MXFP8 scoring operands.
// * quantize_mxfp8_kernel: stand-alone FP32/BF16 -> E4M3 + UE8M0 per 32
//   elements (PR #5992 "Key changes", BF16 -> MXFP8 quantisation).
//
// MXFP8 block rule (DSA_MX_SCALE_NOSAT): the UE8M0 exponent is the smallest e
// with amax <= 448 * 2^e, found from the exponent and mantissa bits of amax
// (448 = 1.75 * 2^8); the payload is RNE(x * 2^-e) to E4M3 with saturation
// (hardware cvt.rn.satfinite).  DSA_MX_SCALE_FLOOR: e = floor(log2 amax) - 8.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "dsa_device.cuh"
#include "dsa_params.h"

namespace dsa {


__device__ __forceinline__ float bf16_rne(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// UE8M0 exponent of a 32-element block from its max magnitude (see header).
__device__ __forceinline__ int mx_exponent(float amax, int rule) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (b == 0) return -127;
  int E;
  bool above;    // mantissa of amax (normalised) > 1.75
  const uint32_t eb = b >> 23, mant = b & 0x7FFFFFu;
  if (eb == 0) {   // subnormal: amax = mant * 2^-149
    const int pbit = 31 - __clz(mant);
    E = pbit - 149;
    above = (uint64_t)mant * 4u > (uint64_t)7u << pbit;
  } else {
    E = (int)eb - 127;
    above = mant > 0x600000u;
  }
  int e = rule == 1 ? E - 8 : (above ? E - 7 : E - 8);
  e = e < -127 ? -127 : (e > 127 ? 127 : e);
  return e;
}

// 2^-e as a float for e in [-127, 127]
__device__ __forceinline__ float exp2_neg(int e) {
  const int be = 127 - e;
  return be >= 1 ? __uint_as_float((uint32_t)be << 23) : __uint_as_float(0x00400000u);
}

// Quantise one block of 4*GL elements spread over GL consecutive lanes (4
// values per lane): GL = 8 is an MXFP8 block of 32, GL = 32 a whole 128-element
// row of per-vector FP8.  Returns the lane's 4 payload bytes; *scale_byte is
// the block's UE8M0.
template <int GL>
__device__ __forceinline__ uint32_t quant_lane4(const float v[4], int rule, int* scale_byte) {
  float amax;
  if constexpr (GL == 32) {
    // whole-warp block: magnitudes compare as unsigned integers, one warp
    // reduction (measured faster than five shuffle steps; for 8-lane blocks a
    // reduction with a partial mask is slower than three shuffles)
    uint32_t am = max(max(__float_as_uint(v[0]) & 0x7FFFFFFFu, __float_as_uint(v[1]) & 0x7FFFFFFFu),
                      max(__float_as_uint(v[2]) & 0x7FFFFFFFu, __float_as_uint(v[3]) & 0x7FFFFFFFu));
    amax = __uint_as_float(__reduce_max_sync(0xffffffffu, am));
  } else {
    amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 1; o < GL; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  }
  const int e = mx_exponent(amax, rule);
  const float mul = exp2_neg(e);
  const __nv_fp8x2_storage_t lo =
      __nv_cvt_float2_to_fp8x2(make_float2(v[0] * mul, v[1] * mul), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi =
      __nv_cvt_float2_to_fp8x2(make_float2(v[2] * mul, v[3] * mul), __NV_SATFINITE, __NV_E4M3);
  *scale_byte = e + 127;
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

template <int VEC>
__device__ __forceinline__ void load_row(const void* base, int in_bf16, size_t row, int D, int lane,
                                         float (&x)[VEC]) {
  if (in_bf16) {
    const __nv_bfloat16* p = reinterpret_cast<const __nv_bfloat16*>(base) + row * D + lane * VEC;
    if constexpr (VEC == 4) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
      x[0] = __uint_as_float(u.x << 16);
      x[1] = __uint_as_float(u.x & 0xFFFF0000u);
      x[2] = __uint_as_float(u.y << 16);
      x[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
      const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(p));
      x[0] = __uint_as_float(u << 16);
      x[1] = __uint_as_float(u & 0xFFFF0000u);
    }
  } else {
    const float* p = reinterpret_cast<const float*>(base) + row * D + lane * VEC;
    if constexpr (VEC == 4) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(p));
      x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    } else {
      const float2 f = __ldg(reinterpret_cast<const float2*>(p));
      x[0] = f.x; x[1] = f.y;
    }
  }
}

constexpr int kPreThreads = 256;
constexpr int kPreMinBlocks = 4;   // resident blocks per SM: 64 registers a thread, no spills
constexpr int kPreMaxRows = 9;   // ceil((64 query heads + 1 key) / 8 warps)

// One block per token.  Row r < H is query head r, row H is the key.
template <int D>
__global__ void __launch_bounds__(kPreThreads, kPreMinBlocks) preprocess_kernel(const __grid_constant__ PreParams p) {
  constexpr int VEC = D / 32;
  __shared__ float s_cos[64], s_sin[64];
  __shared__ int s_pos;
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H;
  // issue the row loads first (memory-level parallelism), then the position
  float x[kPreMaxRows][VEC];
#pragma unroll
  for (int j = 0; j < kPreMaxRows; ++j) {
    const int r = warp + 8 * j;
    if (r < H) load_row<VEC>(p.q, p.in_bf16, (size_t)t * H + r, D, lane, x[j]);
    else if (r == H) load_row<VEC>(p.k, p.in_bf16, (size_t)t, D, lane, x[j]);
  }
  if (threadIdx.x == 0) {
    int lo = 0, hi = p.num_seqs - 1;   // last document whose start is <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    s_pos = t - p.cu[lo];
  }
  __syncthreads();
  const int half = p.rope_dim >> 1;
  if ((int)threadIdx.x < half) {
    // angle pos*theta_i in double, Cody-Waite reduction by 2*pi (two-term
    // constant), then single-precision sincos of the reduced angle
    const double ang = (double)s_pos * p.inv_freq[threadIdx.x];
    const double kq = rint(ang * 0.15915494309189535);
    double red = fma(-kq, 6.283185307179586, ang);
    red = fma(-kq, 2.4492935982947064e-16, red);
    float sv, cv;
    sincosf((float)red, &sv, &cv);
    s_cos[threadIdx.x] = cv;
    s_sin[threadIdx.x] = sv;
  }
  __syncthreads();
  const int d0 = lane * VEC;
  // this lane's rotary factors and partner lane, the same for every row of the token
  float rc[VEC], rs[VEC];
  const bool rot = half > 0 && d0 < p.rope_dim;
  const uint32_t rot_mask = __ballot_sync(0xffffffffu, rot);   // the rotary lanes (and their partners)
  const int src_lane = d0 < half ? lane + half / VEC : (d0 < p.rope_dim ? lane - half / VEC : lane);
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    const int d = d0 + e;
    const int i = p.interleaved ? (d >> 1) : (d < half ? d : d - half);
    rc[e] = rot ? s_cos[i] : 1.f;
    rs[e] = rot ? (p.interleaved || d < half ? -s_sin[i] : s_sin[i]) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < kPreMaxRows; ++j) {
    const int r = warp + 8 * j;
    if (r > H) break;
    const bool is_key = r == H;
    float v[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) v[e] = x[j][e];
    if (is_key && p.gamma != nullptr) {   // key LayerNorm: biased variance, two passes
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < VEC; ++e) s += v[e];
      const float mean = warp_sum(s) / (float)D;
      float s2 = 0.f;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        v[e] -= mean;
        s2 += v[e] * v[e];
      }
      const float var = warp_sum(s2) / (float)D;
      const float rstd = 1.0f / sqrtf(var + p.eps);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        v[e] = fmaf(v[e] * rstd, __ldg(p.gamma + d0 + e), __ldg(p.beta + d0 + e));
        if (!p.rope_fp32) v[e] = bf16_rne(v[e]);
      }
    }
    if (rot) {
      // rotate-half: v' = v cos -/+ partner sin (sign folded into rs); the partner
      // value comes from lane +- half/VEC.  Interleaved: pairs (2i, 2i+1) in-lane.
      if (p.interleaved) {
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
          const float a = v[e], b = v[e + 1];
          v[e] = fmaf(a, rc[e], b * rs[e]);          // a cos - b sin
          v[e + 1] = fmaf(b, rc[e + 1], -a * rs[e + 1]);   // b cos + a sin
        }
      } else {
        float pv[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) pv[e] = __shfl_sync(rot_mask, v[e], src_lane);
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[e] = fmaf(v[e], rc[e], pv[e] * rs[e]);
      }
    }
    if (!p.rope_fp32) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) v[e] = bf16_rne(v[e]);
    }
    const size_t orow = is_key ? (size_t)t : (size_t)t * H + r;
    void* out = is_key ? p.k_out : p.q_out;
    if (p.out_mode == 2) {   // FP8, one scale per row (D = 128: 4 values per lane)
      if constexpr (VEC == 4) {
        int sb;
        const uint32_t pay = quant_lane4<32>(v, p.scale_rule, &sb);
        reinterpret_cast<uint32_t*>(out)[orow * (D / 4) + lane] = pay;
        if (lane == 0) (is_key ? p.k_scale : p.q_scale)[orow] = (uint8_t)sb;
      }
    } else if (p.out_mode == 1) {
      if constexpr (VEC == 4) {
        int sb;
        const uint32_t pay = quant_lane4<8>(v, p.scale_rule, &sb);
        reinterpret_cast<uint32_t*>(out)[orow * (D / 4) + lane] = pay;
        // the first lane of each 8-lane block writes the block's scale byte
        if ((lane & 7) == 0) (is_key ? p.k_scale : p.q_scale)[orow * (D / 32) + (lane >> 3)] = (uint8_t)sb;
      }
    } else {
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out) + orow * D + d0;
      if constexpr (VEC == 4) {
        __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&a);
        u.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(o) = u;
      } else {
        *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(v[0], v[1]);
      }
    }
  }
}

// Flat view: the tensor is a sequence of 32-element blocks (rows*cols/32,
// cols % 32 == 0 so no block straddles rows) whose scale bytes are stored in
// the same order.  A warp quantises 4 consecutive blocks, 8 lanes per block.
__global__ void __launch_bounds__(256) quantize_mxfp8_kernel(const void* __restrict__ x, int in_bf16,
                                                            int64_t nblocks, int rule,
                                                            uint8_t* __restrict__ out,
                                                            uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t wg = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       wg * 4 < nblocks; wg += warps) {
    const int64_t blk = wg * 4 + (lane >> 3);
    const bool valid = blk < nblocks;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    const int64_t e0 = blk * 32 + (lane & 7) * 4;
    if (valid) {
      if (in_bf16) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(x) + e0));
        v[0] = __uint_as_float(u.x << 16);
        v[1] = __uint_as_float(u.x & 0xFFFF0000u);
        v[2] = __uint_as_float(u.y << 16);
        v[3] = __uint_as_float(u.y & 0xFFFF0000u);
      } else {
        const float4 f = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + e0));
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
      }
    }
    int sb;
    const uint32_t pay = quant_lane4<8>(v, rule, &sb);
    if (valid) {
      reinterpret_cast<uint32_t*>(out)[e0 >> 2] = pay;
      if ((lane & 7) == 0) scales[blk] = (uint8_t)sb;
    }
  }
}

// Per-vector FP8: one warp per 128-element row, 4 elements per lane.
__global__ void __launch_bounds__(256) quantize_fp8_rows_kernel(const void* __restrict__ x, int in_bf16,
                                                               int64_t rows, int rule,
                                                               uint8_t* __restrict__ out,
                                                               uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    float v[4];
    load_row<4>(x, in_bf16, (size_t)r, 128, lane, v);
    int sb;
    const uint32_t pay = quant_lane4<32>(v, rule, &sb);
    reinterpret_cast<uint32_t*>(out)[r * 32 + lane] = pay;
    if (lane == 0) scales[r] = (uint8_t)sb;
  }
}

cudaError_t launch_quantize_fp8_rows(const void* x, int in_bf16, int64_t rows, int rule, uint8_t* out,
                                     uint8_t* scales, int sm_count, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = (int64_t)sm_count * 16;
  if (blocks > cap) blocks = cap;
  quantize_fp8_rows_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, in_bf16, rows, rule, out, scales);
  return cudaGetLastError();
}

cudaError_t launch_preprocess(const PreParams& p, int D, cudaStream_t stream) {
  if (p.total_tokens == 0) return cudaSuccess;
  if (D == 128)
    preprocess_kernel<128><<<p.total_tokens, kPreThreads, 0, stream>>>(p);
  else
    preprocess_kernel<64><<<p.total_tokens, kPreThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quantize_mxfp8(const void* x, int in_bf16, int64_t nblocks, int rule,
                                  uint8_t* out, uint8_t* scales, int sm_count, cudaStream_t stream) {
  if (nblocks == 0) return cudaSuccess;
  const int64_t warps_needed = (nblocks + 3) / 4;
  int64_t blocks = (warps_needed + 7) / 8;
  const int64_t cap = (int64_t)sm_count * 16;
  if (blocks > cap) blocks = cap;
  quantize_mxfp8_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, in_bf16, nblocks, rule, out, scales);
  return cudaGetLastError();
}

}  // namespace dsa
