// Kernel parameter blocks and launcher declarations shared by the C ABI
// (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "score_layout.h"

namespace dsa {

struct PreParams {
  const void* q;
  const void* k;
  const float* gamma;
  const float* beta;
  const int32_t* cu;
  void* q_out;
  uint8_t* q_scale;
  void* k_out;
  uint8_t* k_scale;
  double inv_freq[64];
  float eps;
  int in_bf16, num_seqs, total_tokens, H, rope_dim, interleaved, rope_fp32, scale_rule;
  int out_mode;   // 0: BF16, 1: MXFP8 (scale per 32 elements), 2: FP8 (scale per row)
};

struct DebugParams {
  CUtensorMap tm_q, tm_k, tm_qs, tm_ks;
  int64_t q_row0, k_row0;
  int chunks, n_cols;
  float* out;
  int* status;
  unsigned long long timeout_ns;
};

cudaError_t launch_preprocess(const PreParams& p, int D, cudaStream_t stream);
cudaError_t launch_quantize_fp8_rows(const void* x, int in_bf16, int64_t rows, int rule, uint8_t* out,
                                     uint8_t* scales, int sm_count, cudaStream_t stream);
cudaError_t launch_quantize_mxfp8(const void* x, int in_bf16, int64_t nblocks, int rule,
                                  uint8_t* out, uint8_t* scales, int sm_count, cudaStream_t stream);
cudaError_t launch_kpool(const void* k, int k_bf16, const uint16_t* gate, const float* bias,
                         const int32_t* cu, int num_seqs, int total_tokens, int D, int P,
                         uint16_t* out, int32_t* cu_pools, int sm_count, cudaStream_t stream);
cudaError_t launch_build_worklist(const int32_t* cu, const int32_t* cu_k, const int32_t* cu_comp, int num_seqs,
                                  int total_tokens,
                                  int total_k, int max_seqlen, int max_seqlen_k, int tq, int pool,
                                  int2* items, int* doc_prefix, int* tile_base, int* hdr, int max_items,
                                  cudaStream_t stream);
cudaError_t launch_tiled_kscales(const uint8_t* k_scale, int64_t k_rows, int replicate, const int32_t* cu_keys,
                                 const int* tile_base, int num_seqs, int max_tiles, uint32_t* out,
                                 int sm_count, cudaStream_t stream);
cudaError_t launch_score_topk(const ScoreParams& p, int grid, cudaStream_t stream);
// Checked build: NaN / Inf scan of a score + top-k call's inputs (status word).
cudaError_t launch_validate_inputs(const void* q, int64_t q_bytes, const void* k, int64_t k_bytes, int op_bf16,
                                   const uint8_t* qs, int64_t qs_bytes, const uint8_t* ks, int64_t ks_bytes,
                                   const void* w, int64_t w_elems, int w_bf16, int* hdr, int sm_count,
                                   cudaStream_t stream);
cudaError_t launch_debug_mma_tile(const DebugParams& p, int prec, cudaStream_t stream);
// Reorders each finished top-k row into ranking order (score desc, index asc),
// moving units of `group` consecutive entries (1, or the KPool pool size).
cudaError_t launch_rank_rows(int32_t* idx, float* score, int64_t rows, int width, int group, int sm_count,
                             cudaStream_t stream);

}  // namespace dsa
