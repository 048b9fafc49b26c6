// C ABI of the library (include/dsa_idx.h): host-side validation, workspace
// carving, TMA tensor-map construction and kernel launches.  Never allocates,
// frees or synchronises (except dsa_idx_read_status, an eager helper).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "dsa_idx.h"
#include "dsa_idx_testing.h"
#include "dsa_status_codes.h"
#include "dsa_params.h"


using namespace dsa;

namespace {

thread_local std::string g_last_error;

}  // namespace

namespace dsa {
// Set the message dsa_idx_last_error() returns (for entry points in other files).
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace dsa

namespace {

dsa_status_t fail(dsa_status_t s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
dsa_status_t fail(dsa_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

dsa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device facts, cached per device ordinal.
struct DevInfo {
  int sm_count = 0, major = 0, minor = 0;
};

dsa_status_t device_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev].sm_count == 0) {
    DevInfo d;
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    cache[dev] = d;
  }
  *out = cache[dev];
  if (out->major != 10 || out->minor != 3)
    return fail(DSA_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", out->major, out->minor);
  return DSA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Operand [rows, D] (bf16 or u8), box box_rows x 128 bytes, 128-byte swizzle.
dsa_status_t make_operand_map(CUtensorMap* m, const void* base, int64_t rows, int D, bool fp8,
                              int box_rows = kTileKeys) {
  auto enc = encode_fn();
  if (!enc) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const int elem = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)D * elem};
  cuuint32_t box[2] = {(cuuint32_t)(kChunkBytes / elem), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled(operand) failed: %d", (int)r);
  return DSA_OK;
}

// Scale words: rows of 4 UE8M0 bytes viewed as u32 [rows], box 132 words.
dsa_status_t make_scale_map(CUtensorMap* m, const void* base, int64_t rows) {
  auto enc = encode_fn();
  if (!enc) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[1] = {(cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {4};
  cuuint32_t box[1] = {(cuuint32_t)kSfRawWords};
  cuuint32_t estr[1] = {1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 1, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled(scale) failed: %d", (int)r);
  return DSA_OK;
}

bool heads_ok(int H) { return H == 4 || H == 8 || H == 16 || H == 32 || H == 64; }

// workspace layout: [0,256) header (status, item count); per-document item
// prefix int[num_seqs+1]; per-document key-tile prefix int[num_seqs+1]; work
// items int2[total_tokens + num_seqs]; MXFP8 and FP8: key scales laid out per
// key tile for tcgen05.cp, 512 bytes x (total_tokens/128 + num_seqs + 1).
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
size_t ws_prefix_off() { return 256; }
size_t ws_tiles_off(int num_seqs) { return ws_prefix_off() + round256((size_t)(num_seqs + 1) * 4); }
size_t ws_items_off(int num_seqs) { return ws_tiles_off(num_seqs) + round256((size_t)(num_seqs + 1) * 4); }
size_t ws_ksf_off(int total_tokens, int num_seqs) {
  return ws_items_off(num_seqs) + round256((size_t)8 * ((size_t)total_tokens + num_seqs));
}
int ws_ksf_tiles(int total_tokens, int num_seqs) { return total_tokens / kTileKeys + num_seqs + 1; }
size_t ws_total(int total_tokens, int num_seqs, bool scales) {
  return ws_ksf_off(total_tokens, num_seqs) +
         (scales ? (size_t)kSfTxBytes * ws_ksf_tiles(total_tokens, num_seqs) : 0);
}

unsigned long long g_timeout_ns = 2000000000ull;
int g_fault_inject = 0;

}  // namespace

extern "C" {

#ifdef DSA_CHECKED
int dsa_idx_version(void) { return 200 + 1; }   // 2.0.0, checked build (odd)
#else
int dsa_idx_version(void) { return 200; }       // 2.0.0
#endif

const char* dsa_idx_last_error(void) { return g_last_error.c_str(); }

const char* dsa_idx_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
    case DSA_ERR_BOUNDS: return "DSA_ERR_BOUNDS";
  }
  return "DSA_ERR_UNKNOWN";
}

size_t dsa_idx_workspace_size(int total_tokens, int num_seqs, int max_seqlen, int n_heads,
                              int head_dim, int index_topk, int kpool_size, dsa_precision_t prec) {
  (void)max_seqlen; (void)n_heads; (void)head_dim; (void)index_topk; (void)kpool_size;
  if (total_tokens < 0 || num_seqs < 1) return 0;
  return ws_total(total_tokens, num_seqs, prec == DSA_PREC_MXFP8 || prec == DSA_PREC_FP8);
}

int dsa_idx_output_width(int index_topk, int kpool_size, int flags) {
  if (flags & DSA_FLAG_COMPRESSED_KEYS) return index_topk;
  if (kpool_size > 1 && (flags & DSA_FLAG_KPOOL_TAIL)) return index_topk + kpool_size - 1;
  return index_topk;
}

dsa_status_t dsa_idx_preprocess(const void* q, const void* k, dsa_dtype_t in_dtype,
                                const float* ln_gamma, const float* ln_beta, float ln_eps,
                                const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                                int max_seqlen, int n_heads, int head_dim, int rope_dim,
                                float rope_base, int rope_interleaved, int rope_fp32,
                                dsa_precision_t out_prec, dsa_mx_scale_rule_t scale_rule,
                                void* q_out, uint8_t* q_scale_out, void* k_out,
                                uint8_t* k_scale_out, dsa_stream_t stream) {
  if (!q || !k || !cu_seqlens || !q_out || !k_out) return fail(DSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_out) || !aligned16(k_out))
    return fail(DSA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (in_dtype != DSA_DTYPE_F32 && in_dtype != DSA_DTYPE_BF16) return fail(DSA_ERR_INVALID_ARG, "in_dtype");
  if (num_seqs < 1 || total_tokens < 0 || max_seqlen < 0) return fail(DSA_ERR_INVALID_ARG, "sizes");
  if (head_dim != 64 && head_dim != 128) return fail(DSA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (n_heads < 1 || n_heads > 64) return fail(DSA_ERR_UNSUPPORTED, "n_heads must be 1..64");
  if (rope_dim < 0 || rope_dim > head_dim || rope_dim % 8 != 0)
    return fail(DSA_ERR_INVALID_ARG, "rope_dim must be a multiple of 8 in [0, head_dim]");
  if ((ln_gamma == nullptr) != (ln_beta == nullptr))
    return fail(DSA_ERR_INVALID_ARG, "ln_gamma and ln_beta must both be given or both NULL");
  if (!(ln_eps >= 0.f)) return fail(DSA_ERR_INVALID_ARG, "ln_eps");
  if (rope_dim > 0 && !(rope_base > 0.f)) return fail(DSA_ERR_INVALID_ARG, "rope_base");
  if (out_prec == DSA_PREC_MXFP8) {
    if (head_dim != 128) return fail(DSA_ERR_UNSUPPORTED, "MXFP8 output needs head_dim 128");
    if (!q_scale_out || !k_scale_out || !aligned16(q_scale_out) || !aligned16(k_scale_out))
      return fail(DSA_ERR_INVALID_ARG, "MXFP8 output needs 16-byte aligned scale buffers");
  } else if (out_prec == DSA_PREC_FP8) {
    if (head_dim != 128) return fail(DSA_ERR_UNSUPPORTED, "FP8 output needs head_dim 128");
    if (!q_scale_out || !k_scale_out) return fail(DSA_ERR_INVALID_ARG, "FP8 output needs scale buffers");
  } else if (out_prec != DSA_PREC_BF16) {
    return fail(DSA_ERR_INVALID_ARG, "out_prec");
  }
  if (scale_rule != DSA_MX_SCALE_NOSAT && scale_rule != DSA_MX_SCALE_FLOOR)
    return fail(DSA_ERR_INVALID_ARG, "scale_rule");
  DevInfo di;
  dsa_status_t s = device_info(&di);
  if (s != DSA_OK) return s;
  PreParams p{};
  p.q = q; p.k = k; p.gamma = ln_gamma; p.beta = ln_beta; p.cu = cu_seqlens;
  p.q_out = q_out; p.q_scale = q_scale_out; p.k_out = k_out; p.k_scale = k_scale_out;
  for (int i = 0; i < rope_dim / 2; ++i)
    p.inv_freq[i] = std::pow((double)rope_base, -2.0 * i / (double)rope_dim);
  p.eps = ln_eps;
  p.in_bf16 = in_dtype == DSA_DTYPE_BF16;
  p.num_seqs = num_seqs;
  p.total_tokens = total_tokens;
  p.H = n_heads;
  p.rope_dim = rope_dim;
  p.interleaved = rope_interleaved ? 1 : 0;
  p.rope_fp32 = rope_fp32 ? 1 : 0;
  p.out_mode = out_prec == DSA_PREC_MXFP8 ? 1 : (out_prec == DSA_PREC_FP8 ? 2 : 0);
  p.scale_rule = (int)scale_rule;
  cudaError_t e = launch_preprocess(p, head_dim, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "preprocess launch");
  return DSA_OK;
}

dsa_status_t dsa_idx_quantize_fp8_rows(const void* x, dsa_dtype_t in_dtype, int64_t rows, int cols,
                                       dsa_mx_scale_rule_t scale_rule, uint8_t* x_e4m3, uint8_t* x_ue8m0,
                                       dsa_stream_t stream) {
  if (!x || !x_e4m3 || !x_ue8m0) return fail(DSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(x_e4m3)) return fail(DSA_ERR_INVALID_ARG, "16-byte alignment");
  if (rows < 0 || cols != 128) return fail(DSA_ERR_UNSUPPORTED, "cols must be 128");
  if (in_dtype != DSA_DTYPE_F32 && in_dtype != DSA_DTYPE_BF16) return fail(DSA_ERR_INVALID_ARG, "in_dtype");
  if (scale_rule != DSA_MX_SCALE_NOSAT && scale_rule != DSA_MX_SCALE_FLOOR)
    return fail(DSA_ERR_INVALID_ARG, "scale_rule");
  DevInfo di;
  dsa_status_t s = device_info(&di);
  if (s != DSA_OK) return s;
  cudaError_t e = launch_quantize_fp8_rows(x, in_dtype == DSA_DTYPE_BF16, rows, (int)scale_rule, x_e4m3, x_ue8m0,
                                           di.sm_count, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return DSA_OK;
}

dsa_status_t dsa_idx_quantize_mxfp8(const void* x, dsa_dtype_t in_dtype, int64_t rows, int cols,
                                    dsa_mx_scale_rule_t scale_rule, uint8_t* x_e4m3,
                                    uint8_t* x_ue8m0, dsa_stream_t stream) {
  if (!x || !x_e4m3 || !x_ue8m0) return fail(DSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(x_e4m3)) return fail(DSA_ERR_INVALID_ARG, "16-byte alignment");
  if (rows < 0 || cols <= 0 || cols % 32 != 0) return fail(DSA_ERR_INVALID_ARG, "cols must be a positive multiple of 32");
  if (in_dtype != DSA_DTYPE_F32 && in_dtype != DSA_DTYPE_BF16) return fail(DSA_ERR_INVALID_ARG, "in_dtype");
  if (scale_rule != DSA_MX_SCALE_NOSAT && scale_rule != DSA_MX_SCALE_FLOOR)
    return fail(DSA_ERR_INVALID_ARG, "scale_rule");
  DevInfo di;
  dsa_status_t s = device_info(&di);
  if (s != DSA_OK) return s;
  cudaError_t e = launch_quantize_mxfp8(x, in_dtype == DSA_DTYPE_BF16, rows * (int64_t)(cols / 32),
                                        (int)scale_rule, x_e4m3, x_ue8m0, di.sm_count,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return DSA_OK;
}

dsa_status_t dsa_idx_kpool_compress(const void* k, dsa_dtype_t k_dtype, const uint16_t* gate_bf16,
                                    const float* slot_bias, const int32_t* cu_seqlens, int num_seqs,
                                    int total_tokens, int head_dim, int pool_size,
                                    uint16_t* k_pooled, int32_t* cu_pools, dsa_stream_t stream) {
  if (!k || !gate_bf16 || !slot_bias || !cu_seqlens || !k_pooled || !cu_pools)
    return fail(DSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k) || !aligned16(k_pooled)) return fail(DSA_ERR_INVALID_ARG, "16-byte alignment");
  if (head_dim != 64 && head_dim != 128) return fail(DSA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (pool_size != 2 && pool_size != 4 && pool_size != 8) return fail(DSA_ERR_UNSUPPORTED, "pool_size must be 2, 4 or 8");
  if (num_seqs < 1 || total_tokens < 0) return fail(DSA_ERR_INVALID_ARG, "sizes");
  if (k_dtype != DSA_DTYPE_F32 && k_dtype != DSA_DTYPE_BF16) return fail(DSA_ERR_INVALID_ARG, "k_dtype");
  DevInfo di;
  dsa_status_t s = device_info(&di);
  if (s != DSA_OK) return s;
  cudaError_t e = launch_kpool(k, k_dtype == DSA_DTYPE_BF16, gate_bf16, slot_bias, cu_seqlens, num_seqs,
                               total_tokens, head_dim, pool_size, k_pooled, cu_pools, di.sm_count,
                               reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kpool launch");
  return DSA_OK;
}

namespace {

// The fused call for self-attention documents (cu_k == nullptr: every
// document has as many keys as queries) or for documents whose queries are
// the last tokens of a longer key sequence (cu_k, total_k, max_seqlen_k).
dsa_status_t score_topk_impl(const void* q, const uint8_t* q_scale, const void* k, const uint8_t* k_scale,
                             const void* w, dsa_dtype_t w_dtype, float sm_scale, const int32_t* cu_seqlens,
                             const int32_t* cu_k, int num_seqs, int total_tokens, int total_k,
                             int max_seqlen, int max_seqlen_k, int n_heads, int head_dim, int index_topk,
                             dsa_precision_t prec, int flags, int kpool_size, const int32_t* cu_pools,
                             int32_t* topk_idx, float* topk_score, int32_t* topk_len, void* ws,
                             size_t ws_bytes, dsa_stream_t stream) {
  if (!q || !k || !w || !cu_seqlens || !topk_idx) return fail(DSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k)) return fail(DSA_ERR_INVALID_ARG, "q and k must be 16-byte aligned");
  if (num_seqs < 1 || total_tokens < 0 || max_seqlen < 0 || total_k < 0 || max_seqlen_k < 0)
    return fail(DSA_ERR_INVALID_ARG, "sizes");
  if (max_seqlen > 65536 || max_seqlen_k > 65536) return fail(DSA_ERR_UNSUPPORTED, "max_seqlen above 65536");
  if (cu_k && kpool_size > 1) return fail(DSA_ERR_UNSUPPORTED, "pool mode with separate key lengths");
  if (!heads_ok(n_heads)) return fail(DSA_ERR_UNSUPPORTED, "n_heads must be 4, 8, 16, 32 or 64");
  if (prec != DSA_PREC_BF16 && prec != DSA_PREC_MXFP8 && prec != DSA_PREC_FP8)
    return fail(DSA_ERR_INVALID_ARG, "prec");
  if (prec == DSA_PREC_MXFP8) {
    if (head_dim != 128) return fail(DSA_ERR_UNSUPPORTED, "MXFP8 scoring needs head_dim 128");
    if (!q_scale || !k_scale || !aligned16(q_scale) || !aligned16(k_scale))
      return fail(DSA_ERR_INVALID_ARG, "MXFP8 needs 16-byte aligned q_scale and k_scale");
  } else if (prec == DSA_PREC_FP8) {
    if (head_dim != 128) return fail(DSA_ERR_UNSUPPORTED, "FP8 scoring needs head_dim 128");
    if (!q_scale || !k_scale) return fail(DSA_ERR_INVALID_ARG, "FP8 needs q_scale and k_scale");
  } else if (head_dim != 64 && head_dim != 128) {
    return fail(DSA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  }
  if (w_dtype != DSA_DTYPE_F32 && w_dtype != DSA_DTYPE_BF16) return fail(DSA_ERR_INVALID_ARG, "w_dtype");
  if (flags & ~(DSA_FLAG_DETERMINISTIC | DSA_FLAG_SORT_BY_SCORE | DSA_FLAG_KPOOL_TAIL | DSA_FLAG_COMPRESSED_KEYS))
    return fail(DSA_ERR_INVALID_ARG, "unknown flag bits");
  const bool compressed = (flags & DSA_FLAG_COMPRESSED_KEYS) != 0;
  const bool rank_order = (flags & DSA_FLAG_SORT_BY_SCORE) != 0;
  if (rank_order && !topk_score) return fail(DSA_ERR_INVALID_ARG, "DSA_FLAG_SORT_BY_SCORE needs topk_score");
  if (kpool_size < 1) return fail(DSA_ERR_INVALID_ARG, "kpool_size");
  if (compressed) {
    if (kpool_size < 2 || kpool_size > 64) return fail(DSA_ERR_UNSUPPORTED, "compression ratio must be 2..64");
    if (!cu_pools) return fail(DSA_ERR_INVALID_ARG, "compressed keys need cu_pools");
    if (flags & DSA_FLAG_KPOOL_TAIL) return fail(DSA_ERR_INVALID_ARG, "DSA_FLAG_KPOOL_TAIL applies to KPool only");
  } else if (kpool_size > 1) {
    if (kpool_size != 2 && kpool_size != 4 && kpool_size != 8) return fail(DSA_ERR_UNSUPPORTED, "kpool_size must be 1, 2, 4 or 8");
    if (!cu_pools) return fail(DSA_ERR_INVALID_ARG, "pool mode needs cu_pools");
    if (index_topk % kpool_size != 0) return fail(DSA_ERR_INVALID_ARG, "index_topk must be a multiple of kpool_size");
  }
  const int expand = kpool_size > 1 && !compressed ? kpool_size : 1;   // tokens per selected key in the output
  if (index_topk < 1 || index_topk > kMaxKeep * expand)
    return fail(DSA_ERR_UNSUPPORTED, "index_topk must be in [1, 4096] (KPool: at most 4096 pools)");
  const int keep = index_topk / expand;
  if (keep < 1) return fail(DSA_ERR_INVALID_ARG, "index_topk / kpool_size must be >= 1");
  if (!ws) return fail(DSA_ERR_WORKSPACE, "workspace is NULL");
  const bool mxw = prec == DSA_PREC_MXFP8 || prec == DSA_PREC_FP8;   // key-scale tiles in the workspace
  const int ws_tokens = total_k > total_tokens ? total_k : total_tokens;   // workspace sizing unit
  if (ws_bytes < ws_total(ws_tokens, num_seqs, mxw))
    return fail(DSA_ERR_WORKSPACE, "workspace %zu bytes, need %zu", ws_bytes, ws_total(ws_tokens, num_seqs, mxw));
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(DSA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  ScoreParams p{};
  const int pl_prec = prec == DSA_PREC_MXFP8 ? PREC_MXFP8 : (prec == DSA_PREC_FP8 ? PREC_FP8 : PREC_BF16);
  if (!make_score_plan(pl_prec, head_dim, n_heads, keep, &p.plan))
    return fail(DSA_ERR_UNSUPPORTED, "no kernel configuration fits (n_heads %d, keep %d)", n_heads, keep);
  DevInfo di;
  dsa_status_t s = device_info(&di);
  if (s != DSA_OK) return s;
  const bool fp8 = pl_prec != PREC_BF16;          // one-byte operands
  const bool mx = pl_prec == PREC_MXFP8;          // block scales through TMEM
  const int64_t krows = kpool_size > 1 ? total_tokens / kpool_size : total_k;
  if ((s = make_operand_map(&p.tm_q, q, (int64_t)total_tokens * n_heads, head_dim, fp8, p.plan.ncols)) != DSA_OK)
    return s;
  if ((s = make_operand_map(&p.tm_k, k, krows, head_dim, fp8)) != DSA_OK) return s;
  if (mx) {
    if ((s = make_scale_map(&p.tm_qs, q_scale, (int64_t)total_tokens * n_heads)) != DSA_OK) return s;
    if ((s = make_scale_map(&p.tm_ks, k_scale, krows)) != DSA_OK) return s;
  }
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  int* hdr = reinterpret_cast<int*>(wsb);
  int* doc_prefix = reinterpret_cast<int*>(wsb + ws_prefix_off());
  int* tile_base = reinterpret_cast<int*>(wsb + ws_tiles_off(num_seqs));
  int2* items = reinterpret_cast<int2*>(wsb + ws_items_off(num_seqs));
  uint32_t* ksf_tiles = reinterpret_cast<uint32_t*>(wsb + ws_ksf_off(ws_tokens, num_seqs));
  const int tq = p.plan.nq;
  const int max_items = total_tokens + num_seqs;
  p.w = w;
  p.cu_seqlens = cu_seqlens;
  p.cu_keys = kpool_size > 1 ? cu_pools : (cu_k ? cu_k : cu_seqlens);
  p.cu_seqlens_k = cu_k;
  p.out_idx = topk_idx;
  p.out_score = topk_score;
  p.out_len = topk_len;
  p.out_rows = total_tokens;
  p.items = items;
  p.hdr = hdr;
  p.tile_base = tile_base;
  p.ksf_tiles = fp8 ? ksf_tiles : nullptr;
  p.q_scale_vec = pl_prec == PREC_FP8 ? q_scale : nullptr;
  p.k_rows = krows;
  p.timeout_ns = g_timeout_ns;
  p.sm_scale = sm_scale;
  p.w_bf16 = w_dtype == DSA_DTYPE_BF16;
  p.pool = kpool_size;
  p.expand = expand > 1 ? 1 : 0;
  p.tail = (expand > 1 && (flags & DSA_FLAG_KPOOL_TAIL)) ? 1 : 0;
  p.out_width = dsa_idx_output_width(index_topk, kpool_size, flags);
  p.fault_inject = g_fault_inject;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_build_worklist(cu_seqlens, cu_k, compressed ? cu_pools : nullptr, num_seqs, total_tokens,
                                        total_k, max_seqlen, max_seqlen_k, tq, kpool_size, items, doc_prefix,
                                        tile_base, hdr, max_items, st);
  if (e != cudaSuccess) return cuda_fail(e, "work-list launch");
  if (total_tokens == 0) return DSA_OK;
#ifdef DSA_CHECKED
  {
    const int64_t elem = fp8 ? 1 : 2;
    const int64_t qrows = (int64_t)total_tokens * n_heads;
    const int64_t ns = mx ? head_dim / 32 : 1;   // scale bytes per row (FP8: one)
    e = launch_validate_inputs(q, qrows * head_dim * elem, k, krows * head_dim * elem, fp8 ? 0 : 1,
                               fp8 ? q_scale : nullptr, qrows * ns, fp8 ? k_scale : nullptr, krows * ns, w,
                               (int64_t)total_tokens * n_heads, w_dtype == DSA_DTYPE_BF16, hdr, di.sm_count, st);
    if (e != cudaSuccess) return cuda_fail(e, "input check launch");
  }
#endif
  if (fp8) {   // FP8: each row's one scale byte, replicated over its four 32-element blocks
    e = launch_tiled_kscales(k_scale, krows, mx ? 0 : 1, p.cu_keys, tile_base, num_seqs,
                             ws_ksf_tiles(ws_tokens, num_seqs), ksf_tiles, di.sm_count, st);
    if (e != cudaSuccess) return cuda_fail(e, "key-scale layout launch");
  }
  int grid = di.sm_count;
  const int64_t bound = (int64_t)total_tokens / tq + num_seqs;
  if (bound < grid) grid = (int)bound;
  e = launch_score_topk(p, grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "score_topk launch");
  if (rank_order) {
    e = launch_rank_rows(topk_idx, topk_score, total_tokens, p.out_width, expand, di.sm_count, st);
    if (e != cudaSuccess) return cuda_fail(e, "rank_rows launch");
  }
  return DSA_OK;
}

}  // namespace

dsa_status_t dsa_idx_score_topk(const void* q, const uint8_t* q_scale, const void* k,
                                const uint8_t* k_scale, const void* w, dsa_dtype_t w_dtype,
                                float sm_scale, const int32_t* cu_seqlens, int num_seqs,
                                int total_tokens, int max_seqlen, int n_heads, int head_dim,
                                int index_topk, dsa_precision_t prec, int flags, int kpool_size,
                                const int32_t* cu_pools, int32_t* topk_idx, float* topk_score,
                                int32_t* topk_len, void* ws, size_t ws_bytes, dsa_stream_t stream) {
  return score_topk_impl(q, q_scale, k, k_scale, w, w_dtype, sm_scale, cu_seqlens, nullptr, num_seqs,
                         total_tokens, total_tokens, max_seqlen, max_seqlen, n_heads, head_dim, index_topk,
                         prec, flags, kpool_size, cu_pools, topk_idx, topk_score, topk_len, ws, ws_bytes,
                         stream);
}

dsa_status_t dsa_idx_score_topk_kv(const void* q, const uint8_t* q_scale, const void* k,
                                   const uint8_t* k_scale, const void* w, dsa_dtype_t w_dtype,
                                   float sm_scale, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, int num_seqs, int total_q, int total_k,
                                   int max_seqlen_q, int max_seqlen_k, int n_heads, int head_dim,
                                   int index_topk, dsa_precision_t prec, int flags, int32_t* topk_idx,
                                   float* topk_score, int32_t* topk_len, void* ws, size_t ws_bytes,
                                   dsa_stream_t stream) {
  if (!cu_seqlens_k) return fail(DSA_ERR_INVALID_ARG, "cu_seqlens_k is NULL");
  return score_topk_impl(q, q_scale, k, k_scale, w, w_dtype, sm_scale, cu_seqlens_q, cu_seqlens_k, num_seqs,
                         total_q, total_k, max_seqlen_q, max_seqlen_k, n_heads, head_dim, index_topk, prec,
                         flags, 1, nullptr, topk_idx, topk_score, topk_len, ws, ws_bytes, stream);
}

dsa_status_t dsa_idx_read_status(const void* ws, dsa_stream_t stream, dsa_status_t* out) {
  if (!ws || !out) return fail(DSA_ERR_INVALID_ARG, "null pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int h = 0;
  e = cudaMemcpy(&h, ws, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *out = (dsa_status_t)h;
  return DSA_OK;
}

dsa_status_t dsa_idx_debug_mma_tile(const void* q, const uint8_t* q_scale, int64_t q_rows,
                                    int64_t q_row0, const void* k, const uint8_t* k_scale,
                                    int64_t k_rows, int64_t k_row0, int head_dim, int n_cols,
                                    dsa_precision_t prec, float* acc_out, void* ws, size_t ws_bytes,
                                    dsa_stream_t stream) {
  if (!q || !k || !acc_out || !ws || ws_bytes < 256) return fail(DSA_ERR_INVALID_ARG, "null pointer / workspace");
  if (n_cols < 16 || n_cols > 128 || n_cols % 16 != 0) return fail(DSA_ERR_INVALID_ARG, "n_cols must be 16..128, multiple of 16");
  const bool fp8 = prec == DSA_PREC_MXFP8;
  if (fp8 ? head_dim != 128 : (head_dim != 64 && head_dim != 128)) return fail(DSA_ERR_UNSUPPORTED, "head_dim");
  if (fp8 && (!q_scale || !k_scale)) return fail(DSA_ERR_INVALID_ARG, "scales");
  if (q_row0 < 0 || k_row0 < 0 || q_row0 >= q_rows || k_row0 >= k_rows) return fail(DSA_ERR_INVALID_ARG, "row0");
  DevInfo di;
  dsa_status_t s = device_info(&di);
  if (s != DSA_OK) return s;
  DebugParams p{};
  if ((s = make_operand_map(&p.tm_q, q, q_rows, head_dim, fp8)) != DSA_OK) return s;
  if ((s = make_operand_map(&p.tm_k, k, k_rows, head_dim, fp8)) != DSA_OK) return s;
  if (fp8) {
    if ((s = make_scale_map(&p.tm_qs, q_scale, q_rows)) != DSA_OK) return s;
    if ((s = make_scale_map(&p.tm_ks, k_scale, k_rows)) != DSA_OK) return s;
  }
  p.q_row0 = q_row0;
  p.k_row0 = k_row0;
  p.chunks = head_dim * (fp8 ? 1 : 2) / kChunkBytes;
  p.n_cols = n_cols;
  p.out = acc_out;
  p.status = reinterpret_cast<int*>(ws);
  p.timeout_ns = g_timeout_ns;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e != cudaSuccess) return cuda_fail(e, "memset");
  e = launch_debug_mma_tile(p, fp8 ? PREC_MXFP8 : PREC_BF16, st);
  if (e != cudaSuccess) return cuda_fail(e, "debug launch");
  return DSA_OK;
}

// Test hooks (dsa_idx_testing.h): the bounded-wait limit of the fused kernel,
// and a fault injection that withholds its first key stage so the timeout
// path runs without faulting the GPU.
void dsa_idx_test_set_timeout_ns(unsigned long long ns) { g_timeout_ns = ns; }
void dsa_idx_test_set_fault_inject(int mode) { g_fault_inject = mode; }

}  // extern "C"
