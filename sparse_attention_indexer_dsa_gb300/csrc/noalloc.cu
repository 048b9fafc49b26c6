// Allocation-free variant of dsa_idx_score_topk.
//
// Some callers cannot hand the library a device workspace: code that runs
// after a "no allocation past start-up" point (latency-critical serving loops,
// real-time pipelines), hosts whose memory is owned by an allocator they may
// not grow, and plugin-style integrations that receive only input and output
// tensors.  For them this entry point keeps the fused kernel's scratch (status
// word, document prefix sums, work list) in one file-scope device array that
// every GPU loading the library holds until the process exits.
//
// The array's name is only a host-side stand-in in host code; its device
// address comes from cudaGetSymbolAddress, looked up the first time this entry
// point runs on a device (with that device current) and kept once the lookup
// has succeeded; a failed lookup is retried by the next call.  Make that first
// call before capturing any stream.  The address stays valid for the life of
// the CUDA context: a device reset is not supported while the library is
// loaded.  All calls share the one array: calls whose work overlaps on the GPU
// (different streams, or the same device from several threads without
// ordering) race on it.  The fused kernel's work-list builder rewrites the
// status word and the item count at the start of every call, and every other
// scratch word is written before it is read, so nothing carries over from the
// previous call.  dsa_idx_score_topk_noalloc_status reads the status word the
// last call left there (a bounded device wait that ran out, or cu_seqlens the
// device found inconsistent).
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "dsa_idx.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct ScratchSlot {
  std::mutex mu;
  void* ptr = nullptr;
};

ScratchSlot g_slots[64];

// Device address of the array on the current device; null (and *err set) if
// the lookup failed.  Only a successful lookup is kept.
void* scratch_address(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  ScratchSlot& slot = g_slots[dev];
  std::lock_guard<std::mutex> lk(slot.mu);
  if (slot.ptr == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    slot.ptr = p;
  }
  return slot.ptr;
}

}  // namespace

namespace dsa {
void set_last_error(const std::string& msg);   // api.cu: the message dsa_idx_last_error() returns
}

extern "C" {

dsa_status_t dsa_idx_score_topk_noalloc(
    const void* q, const uint8_t* q_scale, const void* k, const uint8_t* k_scale, const void* w,
    dsa_dtype_t w_dtype, float sm_scale, const int32_t* cu_seqlens, int num_seqs, int total_tokens,
    int max_seqlen, int n_heads, int head_dim, int index_topk, dsa_precision_t prec, int flags,
    int kpool_size, const int32_t* cu_pools, int32_t* topk_idx, float* topk_score,
    int32_t* topk_len, dsa_stream_t stream) {
  const size_t need = dsa_idx_workspace_size(total_tokens, num_seqs, max_seqlen, n_heads, head_dim,
                                             index_topk, kpool_size, prec);
  if (need == 0) {
    dsa::set_last_error("dsa_idx_score_topk_noalloc: invalid sizes");
    return DSA_ERR_INVALID_ARG;
  }
  if (need > kNoAllocScratchBytes) {
    dsa::set_last_error("dsa_idx_score_topk_noalloc: these sizes need " + std::to_string(need) +
                        " bytes of scratch, above the fixed " + std::to_string(kNoAllocScratchBytes) +
                        "-byte array; use dsa_idx_score_topk with a caller workspace");
    return DSA_ERR_WORKSPACE;
  }
  cudaError_t e = cudaSuccess;
  void* scratch = scratch_address(&e);
  if (scratch == nullptr) {
    dsa::set_last_error(std::string("dsa_idx_score_topk_noalloc: no device address for the scratch array: ") +
                        cudaGetErrorString(e));
    return DSA_ERR_CUDA;
  }
  return dsa_idx_score_topk(q, q_scale, k, k_scale, w, w_dtype, sm_scale, cu_seqlens, num_seqs,
                            total_tokens, max_seqlen, n_heads, head_dim, index_topk, prec, flags,
                            kpool_size, cu_pools, topk_idx, topk_score, topk_len, scratch,
                            kNoAllocScratchBytes, stream);
}

dsa_status_t dsa_idx_score_topk_noalloc_status(dsa_stream_t stream, dsa_status_t* out) {
  if (out == nullptr) {
    dsa::set_last_error("dsa_idx_score_topk_noalloc_status: out is NULL");
    return DSA_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaSuccess;
  void* scratch = scratch_address(&e);
  if (scratch == nullptr) {
    dsa::set_last_error(std::string("dsa_idx_score_topk_noalloc_status: no device address for the scratch array: ") +
                        cudaGetErrorString(e));
    return DSA_ERR_CUDA;
  }
  return dsa_idx_read_status(scratch, stream, out);
}

}  // extern "C"
