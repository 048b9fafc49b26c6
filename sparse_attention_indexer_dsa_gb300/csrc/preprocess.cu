// Query/key preprocessing and MXFP8 / per-vector FP8 quantisation for sm_103a
// (HBM-bound).
//
// * preprocess_kernel: key LayerNorm -> RoPE -> BF16, MXFP8 or per-vector
//   FP8, one block per token (its H query rows + its key row), one warp per
//   row, 128-bit loads, warp-shuffle reductions; the output format, RoPE
//   layout and BF16 mid-rounding are template parameters, so a row's code has
//   no branches.  Megatron-LM PR #8403 "cuDNN DSA indexer
//   precision options": "What does this PR do?" (dsa_indexer_rope_fp32 keeps
//   the key LayerNorm -> RoPE chain in FP32) and "Motivation" (the default
//   path materialises BF16 between the LayerNorm and RoPE); review finding 2
//   (BF16 scoring rounds FP32 carriers to BF16).  PR #7522 "Changes": NoPE
//   (rope_dim = 0).  PR #5992 "Key changes": MXFP8 scoring operands.
// * quantize_mxfp8_kernel: stand-alone FP32/BF16 -> E4M3 + UE8M0 per 32
//   elements (PR #5992 "Key changes", BF16 -> MXFP8 quantisation);
//   quantize_fp8_rows_kernel: the same with one UE8M0 scale per 128-element
//   row (PR #8403 "What does this PR do?", the per-vector FP8 path).
//
// MXFP8 block rule (DSA_MX_SCALE_NOSAT): the UE8M0 exponent is the smallest e
// with amax <= 448 * 2^e, found from the exponent and mantissa bits of amax
// (448 = 1.75 * 2^8, see mx_exponent_bits); the payload is RNE(x * 2^-e) to
// E4M3 with saturation (hardware cvt.rn.satfinite).  DSA_MX_SCALE_FLOOR:
// e = floor(log2 amax) - 8.  Non-finite inputs give unspecified codes (the
// checked build's input scan covers the scoring call, not these kernels).
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

// UE8M0 exponent of a block from the bit pattern of its max magnitude
// (sign cleared).  With amax = m * 2^E, m in [1, 2), the smallest e with
// amax <= 448 * 2^e = 1.75 * 2^(e+8) is E - 8, plus one when m > 1.75 (mantissa
// field above 0x600000).  Adding 0x1FFFFF to the bit pattern carries into the
// exponent field exactly in that case, so the NOSAT exponent is
// ((bits + 0x1FFFFF) >> 23) - 135 and the FLOOR exponent (bits >> 23) - 135.
// Zero, subnormal and tiny magnitudes land at or below -127 and clamp there;
// the largest pattern (NaN) gives 121, so no upper clamp is needed.
__device__ __forceinline__ int mx_exponent_bits(uint32_t amax_bits, uint32_t carry) {
  return max((int)((amax_bits + carry) >> 23) - 135, -127);
}

// mantissa carry for the rule: 0 = NOSAT, 1 = FLOOR
__device__ __forceinline__ uint32_t mx_carry(int rule) { return rule == 1 ? 0u : 0x1FFFFFu; }

// 2^-e as a float for e in [-127, 121] (always a normal number)
__device__ __forceinline__ float exp2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// Quantise one block of 4*GL elements spread over GL consecutive lanes (4
// values per lane): GL = 8 is an MXFP8 block of 32, GL = 32 a whole 128-element
// row of per-vector FP8.  Returns the lane's 4 payload bytes; *scale_byte is
// the block's UE8M0.
template <int GL>
__device__ __forceinline__ uint32_t quant_lane4(const float v[4], uint32_t carry, int* scale_byte) {
  // magnitudes compare as unsigned integers
  uint32_t am = max(max(__float_as_uint(v[0]) & 0x7FFFFFFFu, __float_as_uint(v[1]) & 0x7FFFFFFFu),
                    max(__float_as_uint(v[2]) & 0x7FFFFFFFu, __float_as_uint(v[3]) & 0x7FFFFFFFu));
  if constexpr (GL == 32) {
    // whole-warp block: one warp reduction (measured faster than five shuffle
    // steps; for 8-lane blocks a reduction with a partial mask is slower than
    // three shuffles)
    am = __reduce_max_sync(0xffffffffu, am);
  } else {
#pragma unroll
    for (int o = 1; o < GL; o <<= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, o));
  }
  const int e = mx_exponent_bits(am, carry);
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
constexpr int kPreQRows = 8;       // query rows per warp: H <= 64 over 8 warps

enum PreRope { kRopeNone = 0, kRopeHalf = 1, kRopeInterleaved = 2 };

// Loads row `row` of a [rows, D] tensor, VEC = D/32 values per lane.
template <int VEC, bool IN_BF16>
__device__ __forceinline__ void load_lane(const void* base, size_t row, int lane, float (&x)[VEC]) {
  constexpr int D = VEC * 32;
  if constexpr (IN_BF16) {
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

// The issued loads of one token: up to 8 query rows per warp plus the key row
// (held by warp H % 8).
template <int VEC, bool IN_BF16>
__device__ __forceinline__ void load_token(const PreParams& p, int t, int warp, int lane,
                                           float (&xq)[kPreQRows][VEC], float (&xk)[VEC]) {
  const int H = p.H;
#pragma unroll
  for (int j = 0; j < kPreQRows; ++j) {
    const int r = warp + 8 * j;
    if (r < H) load_lane<VEC, IN_BF16>(p.q, (size_t)t * H + r, lane, xq[j]);
  }
  if (warp == (H & 7)) load_lane<VEC, IN_BF16>(p.k, (size_t)t, lane, xk);
}

// RoPE (in-place) for one row; rc/rs are the lane's rotary factors (1 and 0
// on unrotated dims) with the rotate-half sign folded into rs.
template <int VEC, int ROPE>
__device__ __forceinline__ void rope_row(float (&v)[VEC], const float (&rc)[VEC], const float (&rs)[VEC],
                                         bool rot, int src_lane) {
  if constexpr (ROPE == kRopeHalf) {
    // partner value from lane +- half/VEC (itself on unrotated lanes)
    float pv[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) pv[e] = __shfl_sync(0xffffffffu, v[e], src_lane);
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const float r = fmaf(v[e], rc[e], pv[e] * rs[e]);
      v[e] = rot ? r : v[e];
    }
  } else if constexpr (ROPE == kRopeInterleaved) {
    // pairs (2i, 2i+1) in-lane: (a cos - b sin, b cos + a sin)
#pragma unroll
    for (int e = 0; e < VEC; e += 2) {
      const float a = v[e], b = v[e + 1];
      const float ra = fmaf(a, rc[e], b * rs[e]);
      const float rb = fmaf(b, rc[e + 1], -a * rs[e + 1]);
      v[e] = rot ? ra : a;
      v[e + 1] = rot ? rb : b;
    }
  }
}

// Quantises (or rounds) one finished row and stores it.
template <int VEC, int OUT>
__device__ __forceinline__ void store_row(const float (&v)[VEC], void* out, uint8_t* scale, size_t orow,
                                          int lane, uint32_t carry) {
  constexpr int D = VEC * 32;
  if constexpr (OUT == 2) {   // FP8, one scale per row (D = 128: 4 values per lane)
    int sb;
    const uint32_t pay = quant_lane4<32>(v, carry, &sb);
    reinterpret_cast<uint32_t*>(out)[orow * (D / 4) + lane] = pay;
    if (lane == 0) scale[orow] = (uint8_t)sb;
  } else if constexpr (OUT == 1) {   // MXFP8, one scale per 32 elements (8 lanes)
    int sb;
    const uint32_t pay = quant_lane4<8>(v, carry, &sb);
    reinterpret_cast<uint32_t*>(out)[orow * (D / 4) + lane] = pay;
    // the first lane of each 8-lane block writes the block's scale byte
    if ((lane & 7) == 0) scale[orow * (D / 32) + (lane >> 3)] = (uint8_t)sb;
  } else {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out) + orow * D + lane * VEC;
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

// One block per token: warp w handles query heads w, w+8, ... and warp H % 8
// also the key row.  Every choice that is fixed for a call (output format,
// RoPE layout, BF16 rounding between the steps) is a template parameter, so a
// row's code has no branches.
template <int D, int OUT, int ROPE, bool MID_BF16>
__global__ void __launch_bounds__(kPreThreads, kPreMinBlocks) preprocess_kernel(const __grid_constant__ PreParams p) {
  constexpr int VEC = D / 32;
  __shared__ float s_cos[64], s_sin[64];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H;
  // issue the row loads first (memory-level parallelism), then the position
  float xq[kPreQRows][VEC], xk[VEC];
  if (p.in_bf16) load_token<VEC, true>(p, t, warp, lane, xq, xk);
  else load_token<VEC, false>(p, t, warp, lane, xq, xk);
  float rc[VEC], rs[VEC];
  bool rot = false;
  int src_lane = lane;
  if constexpr (ROPE != kRopeNone) {
    const int half = p.rope_dim >> 1;
    if (warp == 0) {
      // position in the document: every lane of warp 0 runs the same search
      int lo = 0, hi = p.num_seqs - 1;   // last document whose start is <= t
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.cu + mid) <= t) lo = mid; else hi = mid - 1;
      }
      const int pos = t - __ldg(p.cu + lo);
      for (int i = lane; i < half; i += 32) {
        // angle pos*theta_i in double, Cody-Waite reduction by 2*pi (two-term
        // constant), then single-precision sincos of the reduced angle
        const double ang = (double)pos * p.inv_freq[i];
        const double kq = rint(ang * 0.15915494309189535);
        double red = fma(-kq, 6.283185307179586, ang);
        red = fma(-kq, 2.4492935982947064e-16, red);
        float sv, cv;
        sincosf((float)red, &sv, &cv);
        s_cos[i] = cv;
        s_sin[i] = sv;
      }
    }
    __syncthreads();
    // this lane's rotary factors and partner lane, the same for every row
    const int d0 = lane * VEC;
    rot = d0 < p.rope_dim;
    if constexpr (ROPE == kRopeHalf)
      src_lane = d0 < half ? lane + half / VEC : (rot ? lane - half / VEC : lane);
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const int d = d0 + e;
      const int i = ROPE == kRopeInterleaved ? (d >> 1) : (d < half ? d : d - half);
      const int ic = rot ? i : 0;
      rc[e] = rot ? s_cos[ic] : 1.f;
      rs[e] = rot ? (ROPE == kRopeInterleaved || d < half ? -s_sin[ic] : s_sin[ic]) : 0.f;
    }
  }
  const uint32_t carry = mx_carry(p.scale_rule);
  uint8_t* q_scale = p.q_scale;
  void* q_out = p.q_out;
#pragma unroll
  for (int j = 0; j < kPreQRows; ++j) {
    const int r = warp + 8 * j;
    if (r >= H) break;
    rope_row<VEC, ROPE>(xq[j], rc, rs, rot, src_lane);
    if constexpr (MID_BF16) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) xq[j][e] = bf16_rne(xq[j][e]);
    }
    store_row<VEC, OUT>(xq[j], q_out, q_scale, (size_t)t * H + r, lane, carry);
  }
  if (warp == (H & 7)) {
    float* v = xk;
    if (p.gamma != nullptr) {   // key LayerNorm: biased variance, two passes
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
        v[e] = fmaf(v[e] * rstd, __ldg(p.gamma + lane * VEC + e), __ldg(p.beta + lane * VEC + e));
        if constexpr (MID_BF16) v[e] = bf16_rne(v[e]);
      }
    }
    rope_row<VEC, ROPE>(xk, rc, rs, rot, src_lane);
    if constexpr (MID_BF16) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) xk[e] = bf16_rne(xk[e]);
    }
    store_row<VEC, OUT>(xk, p.k_out, p.k_scale, (size_t)t, lane, carry);
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
    const uint32_t pay = quant_lane4<8>(v, mx_carry(rule), &sb);
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
    const uint32_t pay = quant_lane4<32>(v, mx_carry(rule), &sb);
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

template <int D, int OUT, int ROPE>
static void launch_pre_mid(const PreParams& p, cudaStream_t stream) {
  if (p.rope_fp32)
    preprocess_kernel<D, OUT, ROPE, false><<<p.total_tokens, kPreThreads, 0, stream>>>(p);
  else
    preprocess_kernel<D, OUT, ROPE, true><<<p.total_tokens, kPreThreads, 0, stream>>>(p);
}

template <int D, int OUT>
static void launch_pre_rope(const PreParams& p, cudaStream_t stream) {
  if (p.rope_dim == 0) launch_pre_mid<D, OUT, kRopeNone>(p, stream);
  else if (p.interleaved) launch_pre_mid<D, OUT, kRopeInterleaved>(p, stream);
  else launch_pre_mid<D, OUT, kRopeHalf>(p, stream);
}

cudaError_t launch_preprocess(const PreParams& p, int D, cudaStream_t stream) {
  if (p.total_tokens == 0) return cudaSuccess;
  if (D == 128) {
    if (p.out_mode == 1) launch_pre_rope<128, 1>(p, stream);
    else if (p.out_mode == 2) launch_pre_rope<128, 2>(p, stream);
    else launch_pre_rope<128, 0>(p, stream);
  } else {
    launch_pre_rope<64, 0>(p, stream);   // 64-wide rows: BF16 output only
  }
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
