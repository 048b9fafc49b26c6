// Fused DSA lightning-indexer score + streaming top-k for sm_103a.
//
// What it computes (Megatron-LM PR #8403 "cuDNN DSA indexer precision
// options", review findings 1-3; PR #5992 "[DeepSeek-V4] Add compact BF16 and
// MXFP8 DSA indexer support", "Key changes"; PR #7522 "KPool (pooled-key) DSA
// indexer support", "Changes"):
//   I[t,s] = sm_scale * sum_j w[t,j] * ReLU(q[t,j] . k[s])  for visible s,
//   then the `keep` best s per query t, ties to the lower index.
//
// Structure (one persistent CTA per SM; 448 threads for the 8-bit formats,
// 576 for BF16):
//   * A work item is nq consecutive queries of one document (one query per
//     epilogue warpgroup at 64 heads).  Its nq*H q rows stay in shared memory
//     as one UMMA B operand of N = nq*H columns.  Items are built and sorted
//     longest-first on the device and dealt to CTAs in snake order.
//   * Warp 0 streams the item's visible keys in tiles of 128 rows through a
//     ring of shared-memory stages with TMA (128-byte swizzle); for MXFP8 each
//     stage also brings the tile's key scales, laid out for tcgen05.cp.
//   * Warp 1 issues one tcgen05.mma chain per key tile (M = 128 keys, N = nq*H,
//     K = head_dim) into a double-buffered TMEM accumulator: kind::f16 (BF16),
//     block-scaled kind::mxf8f6f4 (MXFP8; FP8 with one scale per row uses it
//     too, the key row's scale repeated over its blocks and the query row's
//     folded into the head weights).
//   * Warps 2.. are the epilogue warpgroups (3, or 4 for BF16), one query
//     each.  They read the accumulator with tcgen05.ld (16x256b fragments at 64
//     heads, so each lane needs only 16 head weights), apply ReLU, the head
//     weights and the causal mask, and offer each key's score to the query's
//     candidate buffer in shared memory: keys above the running threshold are
//     appended in index order, and a sampled or radix shrink keeps the buffer
//     small and raises the threshold; a final exact radix select keeps exactly
//     `keep` entries.  Scores never reach HBM.
//   * Every wait is bounded (status word + abort flag, no trap); see
//     dsa_device.cuh.
#include <cuda_bf16.h>

#include "dsa_device.cuh"
#include "dsa_params.h"

namespace dsa {

// Optional per-phase cycle counters (compile with -DDSA_PHASE_TIMERS; off in
// the product build).  Each role accumulates clock64() deltas in registers
// and adds them to g_phase_cycles once, at exit.
#ifdef DSA_PHASE_TIMERS
__device__ unsigned long long g_phase_cycles[64];
#define PT_DECL unsigned long long pt_acc[8] = {0, 0, 0, 0, 0, 0, 0, 0}; long long pt_t0 = clock64();
#define PT_MARK() (pt_t0 = clock64())
#define PT_ADD(i) do { const long long pt_t1 = clock64(); pt_acc[i] += (unsigned long long)(pt_t1 - pt_t0); pt_t0 = pt_t1; } while (0)
#define PT_FLUSH(base, rec) do { if (rec) for (int i_ = 0; i_ < 8; ++i_) atomicAdd(&g_phase_cycles[(base) + i_], pt_acc[i_]); } while (0)
#else
#define PT_DECL
#define PT_MARK() ((void)0)
#define PT_ADD(i) ((void)0)
#define PT_FLUSH(base, rec) ((void)0)
#endif
// Optional event timeline of CTA 0 (compile with -DDSA_TRACE): clock64() of
// event `ev` for tile number `t` (t < 256).
#ifdef DSA_TRACE
__device__ long long g_trace[16][256];
#define TRACE(ev, t, cond) do { if ((cond) && blockIdx.x == 0 && (t) < 256) g_trace[ev][t] = clock64(); } while (0)
#else
#define TRACE(ev, t, cond) ((void)0)
#endif

// Checked build (-DDSA_CHECKED): a write's bounds condition is verified on the
// device; a failure records DSA_ERR_BOUNDS in the status word and the write is
// skipped.  In the normal build the conditions hold by construction and cost
// nothing.
#ifdef DSA_CHECKED
__device__ __forceinline__ bool in_bounds(bool ok, int* status) {
  if (!ok) set_status(status, DSA_DEV_ERR_BOUNDS);
  return ok;
}
#define DSA_IN_BOUNDS(cond, status) in_bounds((cond), (status))
#define DSA_CHK_PARAM , int* status
#define DSA_CHK_ARG , status
#else
#define DSA_IN_BOUNDS(cond, status) true
#define DSA_CHK_PARAM
#define DSA_CHK_ARG
#endif

// ----------------------------------------------------------------------------
// Work list: items (document, first query) sorted by descending tile count so
// the persistent CTAs take the longest items first.  One block.
// ----------------------------------------------------------------------------
constexpr int kWLThreads = 1024;
constexpr int kWLMaxBins = 1025;

// With cu_k (keys per document outnumbering its queries), document d's queries
// are its last cu[d+1]-cu[d] tokens: query i sits at position off_d + i,
// off_d = (cu_k[d+1]-cu_k[d]) - (cu[d+1]-cu[d]), and sees keys 0 .. off_d + i.
__global__ void __launch_bounds__(kWLThreads) build_worklist_kernel(
    const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_k, const int32_t* __restrict__ cu_comp,
    int num_seqs, int total_tokens,
    int total_k, int max_seqlen, int max_seqlen_k, int tq, int pool, int2* __restrict__ items,
    int* __restrict__ doc_prefix, int* __restrict__ tile_base, int* __restrict__ hdr, int max_items) {
  __shared__ int hist[kWLMaxBins];
  __shared__ int s_bad;
  __shared__ int s_total;
  const int tid = threadIdx.x;
  if (tid == 0) {
    hdr[0] = 0;
    hdr[1] = 0;
    s_bad = 0;
  }
  for (int b = tid; b < kWLMaxBins; b += kWLThreads) hist[b] = 0;
  __syncthreads();
  // validate cu_seqlens (and cu_seqlens_k: at least as many keys as queries per document)
  for (int d = tid; d < num_seqs; d += kWLThreads) {
    const int a = cu[d], b = cu[d + 1];
    if (b < a || b - a > max_seqlen) s_bad = 1;
    if (cu_k) {
      const int ak = cu_k[d], bk = cu_k[d + 1];
      if (bk < ak || bk - ak > max_seqlen_k || bk - ak < b - a) s_bad = 1;
    }
  }
  if (tid == 0 && (cu[0] != 0 || cu[num_seqs] != total_tokens)) s_bad = 1;
  if (tid == 0 && cu_k && (cu_k[0] != 0 || cu_k[num_seqs] != total_k)) s_bad = 1;
  // caller-provided compressed keys: room for every complete group, within total_tokens / pool rows
  if (cu_comp) {
    for (int d = tid; d < num_seqs; d += kWLThreads)
      if (cu_comp[d + 1] - cu_comp[d] < (cu[d + 1] - cu[d]) / pool) s_bad = 1;
    if (tid == 0 && (cu_comp[0] < 0 || cu_comp[num_seqs] > total_tokens / pool)) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) set_status(hdr, DSA_DEV_ERR_INVALID_ARG);
    return;
  }
  // per-document item counts -> exclusive prefix (serial chunks of kWLThreads)
  int carry = 0;
  __shared__ int warp_tot[32];
  for (int base = 0; base < num_seqs; base += kWLThreads) {
    const int d = base + tid;
    int v = 0;
    if (d < num_seqs) v = (cu[d + 1] - cu[d] + tq - 1) / tq;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if ((tid & 31) >= o) x += y;
    }
    if ((tid & 31) == 31) warp_tot[tid >> 5] = x;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < (tid >> 5); ++w) before += warp_tot[w];
    if (d < num_seqs) doc_prefix[d] = carry + before + x - v;
    int chunk_total = 0;
    for (int w = 0; w < 32; ++w) chunk_total += warp_tot[w];
    __syncthreads();
    carry += chunk_total;
  }
  if (tid == 0) {
    doc_prefix[num_seqs] = carry;
    s_total = carry;
  }
  __syncthreads();
  // key tiles of every document -> exclusive prefix (where its laid-out key scales start)
  carry = 0;
  for (int base = 0; base < num_seqs; base += kWLThreads) {
    const int d = base + tid;
    int v = 0;
    if (d < num_seqs) {
      const int S = cu_k ? cu_k[d + 1] - cu_k[d] : cu[d + 1] - cu[d];   // keys of the document
      v = ((pool > 1 ? S / pool : S) + kTileKeys - 1) / kTileKeys;
    }
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if ((tid & 31) >= o) x += y;
    }
    if ((tid & 31) == 31) warp_tot[tid >> 5] = x;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < (tid >> 5); ++w) before += warp_tot[w];
    if (d < num_seqs) tile_base[d] = carry + before + x - v;
    int chunk_total = 0;
    for (int w = 0; w < 32; ++w) chunk_total += warp_tot[w];
    __syncthreads();
    carry += chunk_total;
  }
  if (tid == 0) tile_base[num_seqs] = carry;
  __syncthreads();
  const int total = s_total < max_items ? s_total : max_items;
  __threadfence_block();
  auto doc_of = [&](int i) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (doc_prefix[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  auto tiles_of = [&](int d, int blk) {
    const int L = cu[d + 1] - cu[d];
    const int off = cu_k ? (cu_k[d + 1] - cu_k[d]) - L : 0;
    int t_end = (blk + 1) * tq;
    if (t_end > L) t_end = L;
    const int nk = pool > 1 ? t_end / pool : off + t_end;
    int nt = (nk + kTileKeys - 1) / kTileKeys;
    return nt < kWLMaxBins - 1 ? nt : kWLMaxBins - 1;
  };
  for (int i = tid; i < total; i += kWLThreads) {
    const int d = doc_of(i);
    atomicAdd(&hist[tiles_of(d, i - doc_prefix[d])], 1);
  }
  __syncthreads();
  if (tid == 0) {   // exclusive scan in descending tile order (small: <= 1025 bins)
    int run = 0;
    for (int b = kWLMaxBins - 1; b >= 0; --b) {
      const int h = hist[b];
      hist[b] = run;
      run += h;
    }
  }
  __syncthreads();
  for (int i = tid; i < total; i += kWLThreads) {
    const int d = doc_of(i);
    const int blk = i - doc_prefix[d];
    const int pos = atomicAdd(&hist[tiles_of(d, blk)], 1);
    items[pos] = make_int2(d, blk * tq);
  }
  if (tid == 0) hdr[1] = total;
}

// Checked build: a pass over the inputs of a score + top-k call.  A NaN or
// Inf in a BF16 operand (exponent bits all ones), an E4M3 NaN code (0x7F /
// 0xFF), a UE8M0 NaN scale (0xFF) or a non-finite head weight records
// DSA_ERR_INVALID_ARG in the status word and clears the item count, so the
// fused kernel that follows writes nothing.  Operands are scanned in 16-byte
// words (their sizes are multiples of 16 bytes), scales byte by byte.
__global__ void __launch_bounds__(256) validate_inputs_kernel(
    const uint8_t* __restrict__ q, int64_t q_bytes, const uint8_t* __restrict__ k, int64_t k_bytes, int op_bf16,
    const uint8_t* __restrict__ qs, int64_t qs_bytes, const uint8_t* __restrict__ ks, int64_t ks_bytes,
    const void* __restrict__ w, int64_t w_elems, int w_bf16, int* __restrict__ hdr) {
  bool bad = false;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nth = (int64_t)gridDim.x * blockDim.x;
  auto words = [&](const uint8_t* base, int64_t bytes) {
    for (int64_t i = tid * 16; i < bytes; i += nth * 16) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + i));
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (op_bf16) {
          bad |= (u[j] & 0x7F80u) == 0x7F80u || (u[j] & 0x7F800000u) == 0x7F800000u;
        } else {
#pragma unroll
          for (int b = 0; b < 4; ++b) bad |= ((u[j] >> (8 * b)) & 0x7Fu) == 0x7Fu;
        }
      }
    }
  };
  auto scale_bytes = [&](const uint8_t* base, int64_t bytes) {
    for (int64_t i = tid; i < bytes; i += nth) bad |= base[i] == 0xFFu;
  };
  words(q, q_bytes);
  words(k, k_bytes);
  if (qs) scale_bytes(qs, qs_bytes);
  if (ks) scale_bytes(ks, ks_bytes);
  for (int64_t i = tid; i < w_elems; i += nth) {
    const uint32_t b = w_bf16 ? (uint32_t)reinterpret_cast<const uint16_t*>(w)[i] << 16
                              : reinterpret_cast<const uint32_t*>(w)[i];
    bad |= (b & 0x7F800000u) == 0x7F800000u;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) {
    set_status(hdr, DSA_DEV_ERR_INVALID_ARG);
    atomicExch(hdr + 1, 0);
  }
}

// MXFP8 key scales, laid out once per call in the tcgen05.cp source form: for
// key tile t of document d (512 bytes at tile_base[d] + t), 16-byte row l holds
// the 32-bit scale words of the tile's key rows l, l+32, l+64, l+96 (rows past
// the end of the key tensor get 0).  One thread per (tile, row).
__global__ void __launch_bounds__(128) build_tiled_kscales_kernel(
    const uint8_t* __restrict__ kscale, int64_t k_rows, int replicate, const int32_t* __restrict__ cu_keys,
    const int* __restrict__ tile_base, int num_seqs, int max_tiles, uint32_t* __restrict__ out) {
  const int total = tile_base[num_seqs];
  const int r = threadIdx.x;
  for (int g = blockIdx.x; g < total && g < max_tiles; g += gridDim.x) {
    int lo = 0, hi = num_seqs - 1;   // document whose tiles contain g
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_base[mid] <= g) lo = mid; else hi = mid - 1;
    }
    const int64_t row = (int64_t)cu_keys[lo] + (int64_t)(g - tile_base[lo]) * kTileKeys + r;
    uint32_t word = 0u;   // the row's four block scales (FP8: its one scale, four times)
    if (row < k_rows)
      word = replicate ? (uint32_t)__ldg(kscale + row) * 0x01010101u
                       : __ldg(reinterpret_cast<const uint32_t*>(kscale) + row);
    out[(size_t)g * 128 + (r & 31) * 4 + (r >> 5)] = word;
  }
}

// ----------------------------------------------------------------------------
// helpers of the fused kernel
// ----------------------------------------------------------------------------
struct Item {
  int doc, t0, L, off, qrow0, krow0, ntiles, ktile0;   // off: position of the document's first query
};

__device__ __forceinline__ int item_index(int r, int nitems) {
  const int g = gridDim.x;
  const int c = (r & 1) ? (g - 1 - (int)blockIdx.x) : (int)blockIdx.x;
  const int i = r * g + c;
  return i < nitems ? i : -1;
}

__device__ __forceinline__ Item load_item(const ScoreParams& p, int i) {
  const int2 it = p.items[i];
  Item m;
  m.doc = it.x;
  m.t0 = it.y;
  const int a = p.cu_seqlens[m.doc];
  m.L = p.cu_seqlens[m.doc + 1] - a;
  m.qrow0 = (a + m.t0) * p.plan.n_heads;
  m.krow0 = p.cu_keys[m.doc];
  m.off = p.cu_seqlens_k ? (p.cu_seqlens_k[m.doc + 1] - p.cu_seqlens_k[m.doc]) - m.L : 0;
  int t_end = m.t0 + p.plan.nq;
  if (t_end > m.L) t_end = m.L;
  const int nk = p.pool > 1 ? t_end / p.pool : m.off + t_end;
  m.ntiles = (nk + kTileKeys - 1) / kTileKeys;
  m.ktile0 = p.ksf_tiles ? p.tile_base[m.doc] : 0;
  return m;
}

// Bounded wait used while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity, kWaitHintNs)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

// Scale words for tcgen05.cp: raw[off + r] is the 32-bit scale word of row r
// (4 UE8M0 bytes = the row's 4 K-blocks of 32).  Output row l (16 bytes) holds
// rows l, l+32, l+64, l+96: the 32x128-bit source the warpx4 copy replicates
// into every TMEM lane quarter.  Whole warp.
__device__ __forceinline__ void transpose_scales(const uint32_t* raw, int off, uint32_t* tx,
                                                 uint32_t lane) {
  uint4 v;
  v.x = raw[off + lane];
  v.y = raw[off + lane + 32];
  v.z = raw[off + lane + 64];
  v.w = raw[off + lane + 96];
  reinterpret_cast<uint4*>(tx)[lane] = v;
}

__device__ __forceinline__ uint64_t sf_src_desc(uint32_t saddr) {
  return smem_desc(saddr, 0, 128, 0);   // 8-row x 16-byte core matrices, no swizzle
}

__device__ __forceinline__ int warp_incl_scan(int x, uint32_t lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if ((int)lane >= o) x += y;
  }
  return x;
}

// misc scratch (ints) per epilogue warpgroup
enum {
  MS_WTOT = 0,          // [4] scan warp totals
  MS_DIGIT = 4,
  MS_ABOVE = 5,
  MS_BIN = 6,
  MS_GT = 8,            // [4]
  MS_EQ = 12,           // [4]
  MS_MIN = 16,          // [4]
  MS_MAX = 20,          // [4]
  MS_RCNT = 24,         // [2][8] per-warp counts of a compaction round
  MS_BCNT = 48,         // [2][kBatch][kMaxQpw][4] per-warp append counts of a batch
  MS_CAND = MS_BCNT + 2 * kBatch * kMaxQpw * 4,   // [2] the two sampled thresholds
  MS_CNT4 = MS_CAND + 4,                           // [2][4] per-warp counts above them
  MS_SORT = MS_CNT4 + 12,                          // [128] sample keys (sort exchange)
};
static_assert(MS_SORT + 128 <= kMiscInts, "per-warpgroup scratch ints");

// Compactions move PER entries per thread per round (one warpgroup barrier
// per 128 * PER entries): 8 where the block has 128 registers a thread, 4
// where it has 96.
template <int PREC>
__host__ __device__ constexpr int compact_per() { return score_threads(PREC) <= 448 ? 8 : 4; }

// Shrink the n candidates of one query (n > keep).  The buffer holds
// orderable score keys in index order.  Radix select on key - kmin, 8-bit
// digits from the highest bit in which the buffer's keys differ:
//  * exact: keeps exactly `keep` entries, the largest keys with ties to the
//    earlier position (= lower index); returns the keep-th key, so a later
//    candidate must be strictly larger.
//  * approximate (exact == false): stops at the first digit level where
//    keeping the whole boundary bin leaves at most cap_after entries; keeps
//    every entry in or above that bin (never fewer than `keep`) and returns
//    the bin's lower edge minus one, a threshold no larger than the true
//    keep-th key, so no member of the final top-k is ever rejected.
// Histogram passes re-read the keys from shared memory; the stable in-place
// compaction runs in rounds of 128 * PER entries (writes of a round land below the
// next round's inputs).  *count_out receives the number kept.  All 128
// threads of the warpgroup.
template <int PER>
__device__ __noinline__ uint32_t wg_select(uint32_t* keys, uint16_t* idx, int n, int keep,
                                           bool exact, int cap_after, int wq, uint32_t lane,
                                           int* hist, int* ms, int bar_id, int* count_out DSA_CHK_PARAM) {
  const int tid = wq * 32 + (int)lane;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  int e0 = tid;
  for (; e0 + 384 < n; e0 += 512) {
    const uint32_t k0 = keys[e0], k1 = keys[e0 + 128], k2 = keys[e0 + 256], k3 = keys[e0 + 384];
    kmin = min(kmin, min(min(k0, k1), min(k2, k3)));
    kmax = max(kmax, max(max(k0, k1), max(k2, k3)));
  }
  for (; e0 < n; e0 += 128) {
    const uint32_t k = keys[e0];
    kmin = min(kmin, k);
    kmax = max(kmax, k);
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    ms[MS_MIN + wq] = (int)kmin;
    ms[MS_MAX + wq] = (int)kmax;
  }
  named_bar_sync(bar_id, 128);
  kmin = min(min((uint32_t)ms[MS_MIN + 0], (uint32_t)ms[MS_MIN + 1]),
             min((uint32_t)ms[MS_MIN + 2], (uint32_t)ms[MS_MIN + 3]));
  kmax = max(max((uint32_t)ms[MS_MAX + 0], (uint32_t)ms[MS_MAX + 1]),
             max((uint32_t)ms[MS_MAX + 2], (uint32_t)ms[MS_MAX + 3]));
  const uint32_t range = kmax - kmin;
  const int nbits = range == 0 ? 0 : 32 - __clz(range);
  int shift = nbits > 8 ? nbits - 8 : 0;
  uint32_t prefix = 0, pmask = 0;   // in key - kmin space
  int kk = keep;                    // rank still to place inside the current bin
  int keep_eq = keep;               // entries of the final bin to keep
  bool resolved = false;            // prefix is the exact keep-th key
  for (;;) {
    for (int b = tid; b < 256; b += 128) hist[b] = 0;
    named_bar_sync(bar_id, 128);
    int e = tid;
    for (; e + 384 < n; e += 512) {
      uint32_t rel[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) rel[u] = keys[e + 128 * u] - kmin;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if ((rel[u] & pmask) == prefix) atomicAdd(&hist[(rel[u] >> shift) & 0xFFu], 1);
    }
    for (; e < n; e += 128) {
      const uint32_t rel = keys[e] - kmin;
      if ((rel & pmask) == prefix) atomicAdd(&hist[(rel >> shift) & 0xFFu], 1);
    }
    named_bar_sync(bar_id, 128);
    const int hi_bin = 255 - 2 * tid;
    const int h_hi = hist[hi_bin], h_lo = hist[hi_bin - 1];
    const int loc = h_hi + h_lo;
    const int incl = warp_incl_scan(loc, lane);
    if (lane == 31) ms[MS_WTOT + wq] = incl;
    named_bar_sync(bar_id, 128);
    int before = 0;
    for (int w = 0; w < wq; ++w) before += ms[MS_WTOT + w];
    const int excl = before + incl - loc;
    if (excl < kk && excl + h_hi >= kk) {
      ms[MS_DIGIT] = hi_bin;
      ms[MS_ABOVE] = excl;
      ms[MS_BIN] = h_hi;
    } else if (excl + h_hi < kk && excl + loc >= kk) {
      ms[MS_DIGIT] = hi_bin - 1;
      ms[MS_ABOVE] = excl + h_hi;
      ms[MS_BIN] = h_lo;
    }
    named_bar_sync(bar_id, 128);
    const int d = ms[MS_DIGIT];
    kk -= ms[MS_ABOVE];
    const int bin = ms[MS_BIN];
    prefix |= (uint32_t)d << shift;
    pmask |= 0xFFu << shift;
    if (bin == kk) {                       // the whole bin is kept
      keep_eq = bin;
      resolved = shift == 0;
      break;
    }
    if (shift == 0) {                      // prefix is the exact keep-th key
      keep_eq = kk;
      resolved = true;
      break;
    }
    if (!exact && keep - kk + bin <= cap_after) {
      keep_eq = bin;
      break;
    }
    shift = shift > 8 ? shift - 8 : 0;
  }
  // stable compaction in rounds of 128 * PER: keep (rel & pmask) > prefix,
  // and the first keep_eq (in buffer order) with == prefix
  const uint32_t lt = (1u << lane) - 1u;
  const uint32_t keys_s = smem_u32(keys), idx_s = smem_u32(idx);
  int out = 0, eq_seen = 0;
  for (int r0 = 0, rnd = 0; r0 < n; r0 += (128 * PER), ++rnd) {
    uint32_t rk[PER];
    uint16_t ri[PER];
    uint32_t bg[PER], be[PER];
    int gt = 0, eq = 0;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = r0 + wq * (32 * PER) + m * 32 + (int)lane;
      const bool v = e < n;
      rk[m] = v ? keys[e] : 0u;
      ri[m] = v ? idx[e] : (uint16_t)0;
    }
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = r0 + wq * (32 * PER) + m * 32 + (int)lane;
      const bool v = e < n;
      const uint32_t mk = (rk[m] - kmin) & pmask;
      bg[m] = __ballot_sync(0xffffffffu, v && mk > prefix);
      be[m] = __ballot_sync(0xffffffffu, v && mk == prefix);
      gt += __popc(bg[m]);
      eq += __popc(be[m]);
    }
    int* rc = ms + MS_RCNT + (rnd & 1) * 8;
    if (lane == 0) {
      rc[wq] = gt;
      rc[4 + wq] = eq;
    }
    named_bar_sync(bar_id, 128);   // round counts visible; every read of this round done
    int gb = out, eb = eq_seen, gtot = 0, etot = 0;
    for (int w = 0; w < 4; ++w) {
      if (w < wq) {
        gb += rc[w];
        eb += rc[4 + w];
      }
      gtot += rc[w];
      etot += rc[4 + w];
    }
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const bool g1 = (bg[m] >> lane) & 1u;
      const bool e1 = (be[m] >> lane) & 1u;
      const int my_g = gb + __popc(bg[m] & lt);
      const int my_e = eb + __popc(be[m] & lt);
      const int pos = my_g + (my_e < keep_eq ? my_e : keep_eq);   // kept entries before it
      const bool kp = (g1 || (e1 && my_e < keep_eq)) && DSA_IN_BOUNDS(pos < n, status);
      st_shared_u32_if(kp, keys_s + 4u * (uint32_t)pos, rk[m]);
      st_shared_u16_if(kp, idx_s + 2u * (uint32_t)pos, ri[m]);
      gb += __popc(bg[m]);
      eb += __popc(be[m]);
    }
    out += gtot;
    eq_seen += etot;
  }
  named_bar_sync(bar_id, 128);
  *count_out = out + (eq_seen < keep_eq ? eq_seen : keep_eq);
  const uint32_t edge = kmin + prefix;
  return resolved ? edge : edge - 1u;
}

// Approximate shrink from a sample: sort 128 evenly spaced entries
// (bitonic, descending), take two sample keys as candidate thresholds (see
// below), count the entries >= each exactly in one pass, and keep exactly the
// entries >= the tighter threshold whose count lies in [keep, cap_after]
// (stable, in place).  Returns false and changes nothing when neither count
// lies in the window (heavy ties, skewed samples); the caller then uses the
// radix select.  On success
// *tau_out is the new acceptance threshold (candidate - 1: later keys equal to
// it are still accepted, so nothing that may belong to the top-k is lost).
template <int PER>
__device__ __noinline__ bool wg_shrink_sampled(uint32_t* keys, uint16_t* idx, int n, int keep,
                                               int cap_after, int wq, uint32_t lane, int* ms,
                                               int bar_id, uint32_t* tau_out, int* count_out DSA_CHK_PARAM) {
  const int tid = wq * 32 + (int)lane;
  uint32_t* sbuf = reinterpret_cast<uint32_t*>(ms + MS_SORT);
  uint32_t sk = keys[(int)(((long long)tid * n) >> 7)];
#pragma unroll
  for (int k2 = 2; k2 <= 128; k2 <<= 1) {
#pragma unroll
    for (int j = k2 >> 1; j > 0; j >>= 1) {
      uint32_t other;
      if (j >= 32) {
        sbuf[tid] = sk;
        named_bar_sync(bar_id, 128);
        other = sbuf[tid ^ j];
        named_bar_sync(bar_id, 128);
      } else {
        other = __shfl_xor_sync(0xffffffffu, sk, j);
      }
      const bool desc = (tid & k2) == 0;
      const bool low = (tid & j) == 0;
      sk = (low == desc) ? max(sk, other) : min(sk, other);
    }
  }
  // Two thresholds from the sorted samples (descending: sample r has about
  // (r + 1) * n / 128 entries at or above it): a tight one aimed at keep + 1
  // sigma entries and a safe one at keep + 3 sigma, where sigma = n *
  // sqrt(f (1 - f) / 128), f = keep / n, is the spread of that count.  One
  // pass counts both; the tight one wins whenever it keeps enough.
  const float nf = (float)n, f = (float)keep / nf;
  const float sig = nf * sqrtf(f * (1.f - f) * (1.f / 128.f));
  int ra = (int)ceilf(((float)keep + sig) * 128.f / nf) - 1;
  int rs = (int)ceilf(((float)keep + 3.f * sig) * 128.f / nf) - 1;
  ra = ra < 0 ? 0 : (ra > 127 ? 127 : ra);
  rs = rs < 0 ? 0 : (rs > 127 ? 127 : rs);
  if (tid == ra) ms[MS_CAND] = (int)sk;
  if (tid == rs) ms[MS_CAND + 1] = (int)sk;
  named_bar_sync(bar_id, 128);
  const uint32_t cand_a = (uint32_t)ms[MS_CAND], cand_s = (uint32_t)ms[MS_CAND + 1];
  int ca = 0, cs = 0;
  int e = tid;
  for (; e + 384 < n; e += 512) {
    const uint32_t k0 = keys[e], k1 = keys[e + 128], k2 = keys[e + 256], k3 = keys[e + 384];
    ca += (k0 >= cand_a) + (k1 >= cand_a) + (k2 >= cand_a) + (k3 >= cand_a);
    cs += (k0 >= cand_s) + (k1 >= cand_s) + (k2 >= cand_s) + (k3 >= cand_s);
  }
  for (; e < n; e += 128) {
    const uint32_t kv = keys[e];
    ca += kv >= cand_a ? 1 : 0;
    cs += kv >= cand_s ? 1 : 0;
  }
  ca = __reduce_add_sync(0xffffffffu, ca);
  cs = __reduce_add_sync(0xffffffffu, cs);
  if (lane == 0) {
    ms[MS_CNT4 + wq] = ca;
    ms[MS_CNT4 + 4 + wq] = cs;
  }
  named_bar_sync(bar_id, 128);
  // uniform: every thread reads the same counts
  const int tot_a = ms[MS_CNT4 + 0] + ms[MS_CNT4 + 1] + ms[MS_CNT4 + 2] + ms[MS_CNT4 + 3];
  const int tot_s = ms[MS_CNT4 + 4] + ms[MS_CNT4 + 5] + ms[MS_CNT4 + 6] + ms[MS_CNT4 + 7];
  uint32_t cand;
  if (tot_a >= keep && tot_a <= cap_after)
    cand = cand_a;
  else if (tot_s >= keep && tot_s <= cap_after)
    cand = cand_s;
  else
    return false;
  // stable compaction in rounds of 128 * PER entries
  const uint32_t lt = (1u << lane) - 1u;
  const uint32_t keys_s = smem_u32(keys), idx_s = smem_u32(idx);
  int out = 0;
  for (int r0 = 0, rnd = 0; r0 < n; r0 += (128 * PER), ++rnd) {
    uint32_t rk[PER], bk[PER];
    uint16_t ri[PER];
    int cnt = 0;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = r0 + wq * (32 * PER) + m * 32 + (int)lane;
      const bool v = e < n;
      rk[m] = v ? keys[e] : 0u;
      ri[m] = v ? idx[e] : (uint16_t)0;
    }
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = r0 + wq * (32 * PER) + m * 32 + (int)lane;
      bk[m] = __ballot_sync(0xffffffffu, e < n && rk[m] >= cand);
      cnt += __popc(bk[m]);
    }
    int* rc = ms + MS_RCNT + (rnd & 1) * 8;
    if (lane == 0) rc[wq] = cnt;
    named_bar_sync(bar_id, 128);
    int base = out, tot = 0;
    for (int w = 0; w < 4; ++w) {
      if (w < wq) base += rc[w];
      tot += rc[w];
    }
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int pos = base + __popc(bk[m] & lt);
      const bool kp = ((bk[m] >> lane) & 1u) && DSA_IN_BOUNDS(pos < n, status);
      st_shared_u32_if(kp, keys_s + 4u * (uint32_t)pos, rk[m]);
      st_shared_u16_if(kp, idx_s + 2u * (uint32_t)pos, ri[m]);
      base += __popc(bk[m]);
    }
    out += tot;
  }
  named_bar_sync(bar_id, 128);
  *count_out = out;
  *tau_out = cand - 1u;
  return true;
}

// ----------------------------------------------------------------------------
// the fused kernel
// ----------------------------------------------------------------------------
template <int PREC, int H>
__global__ void __launch_bounds__(score_threads(PREC), 1)
    score_topk_kernel(const __grid_constant__ ScoreParams p) {
  constexpr bool MX = PREC == PREC_MXFP8;
  constexpr bool F8 = PREC == PREC_FP8;                // one UE8M0 scale per row (keys: in the MMA; q: in w)
  constexpr bool B1 = MX || F8;                        // one-byte operands
  constexpr int EW = epi_wgs(PREC);                   // epilogue warpgroups
  constexpr int QPW_MAX = qpw_max(PREC, H);           // queries per epilogue warpgroup
  constexpr int NCOLW = QPW_MAX * H;                  // accumulator columns a thread reads per tile
  constexpr int CK = NCOLW < 16 ? NCOLW : 16;         // columns per TMEM load instruction
  constexpr int GRP = (score_threads(PREC) <= 448 || NCOLW < 32) ? NCOLW : 32;   // columns per load/wait group
  constexpr int NGRP = NCOLW / GRP;
  constexpr int NCH = (H / 4) < 4 ? (H / 4) : 4;     // independent FFMA2 chains per query
  constexpr bool FRAG = QPW_MAX == 1 && H == 64;      // one query of 64 heads per warpgroup
  constexpr int VOTE = vote_every(PREC, H);            // batches between two votes
  static_assert(QPW_MAX >= 1 && QPW_MAX <= kMaxQpw, "queries per warpgroup");
  const ScorePlan& pl = p.plan;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  // barriers
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pl.bar_off);
  const int nst = pl.nst;
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + kMaxStages + s); };
  auto bar_tfull = [&](int s) { return smem_u32(bars + 2 * kMaxStages + s); };
  auto bar_tempty = [&](int s) { return smem_u32(bars + 2 * kMaxStages + 2 + s); };
  const uint32_t bar_qfull = smem_u32(bars + 2 * kMaxStages + 4);
  const uint32_t bar_qempty = smem_u32(bars + 2 * kMaxStages + 5);
  const uint32_t bar_drain = smem_u32(bars + 2 * kMaxStages + 6);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kMaxStages + 9);
  int* status = p.hdr;
  const uint64_t tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_tfull(s), 1);
      mbar_init(bar_tempty(s), 4 * EW);   // every epilogue warp reads every tile
    }
    mbar_init(bar_qfull, 1);
    mbar_init(bar_qempty, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    if (MX) {
      tma_prefetch_desc(&p.tm_qs);
      tma_prefetch_desc(&p.tm_ks);
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int nitems = p.hdr[1];
  const int G = gridDim.x;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      PT_DECL
      uint32_t scount = 0, st = 0, ph = 0, ptile = 0;
      bool wrapped = false;
      int it = 0;
      bool ok = true;
      const uint32_t q_bytes = pl.chunks * pl.qchunk + (MX ? pl.sfb_atoms * kSfRawWords * 4 : 0);
      const uint32_t k_bytes = kStageBytes + (B1 ? kSfTxBytes : 0);
      const int chunk_elems = kChunkBytes / (B1 ? 1 : 2);
      for (int r = 0; ok && r * G < nitems; ++r) {
        const int i = item_index(r, nitems);
        if (i < 0) continue;
        const Item m = load_item(p, i);
        if (m.ntiles == 0) continue;
        PT_MARK();
        if (it > 0 && !mbar_wait(bar_qempty, (it - 1) & 1, abort_flag, status, tmo)) {
          ok = false;
          break;
        }
        PT_ADD(0);
        mbar_arrive_expect_tx(bar_qfull, q_bytes);
        for (int c = 0; c < pl.chunks; ++c)
          tma_load_2d(sbase + pl.q_off + c * pl.qchunk, &p.tm_q, bar_qfull, c * chunk_elems, m.qrow0);
        if (MX)
          for (int a = 0; a < pl.sfb_atoms; ++a)
            tma_load_1d(sbase + pl.sfb_raw_off + a * kSfRawBytes, &p.tm_qs, bar_qfull, m.qrow0 + 128 * a);
        ++it;
        for (int t = 0; ok && t < m.ntiles; ++t) {
          const int krow = m.krow0 + t * kTileKeys;
          for (int c = 0; c < pl.chunks; ++c) {
            PT_MARK();
            if (wrapped && !mbar_wait(bar_empty(st), ph ^ 1u, abort_flag, status, tmo)) {
              ok = false;
              break;
            }
            PT_ADD(1);
            if (!(p.fault_inject == 1 && scount == 0)) {   // test hook: stage 0 is never loaded
              TRACE(15, ptile, c == 0);   // producer issues the tile's first K stage
              mbar_arrive_expect_tx(bar_full(st), k_bytes);
              tma_load_2d(sbase + pl.k_off + st * kStageBytes, &p.tm_k, bar_full(st),
                          c * chunk_elems, krow);
              if (B1)   // the tile's key scales, laid out for tcgen05.cp
                bulk_load(sbase + pl.sfa_tx_off + st * kSfTxBytes,
                          p.ksf_tiles + (size_t)(m.ktile0 + t) * (kSfTxBytes / 4), kSfTxBytes,
                          bar_full(st));
            }
            ++scount;
            if (++st == nst) {
              st = 0;
              ph ^= 1u;
              wrapped = true;
            }
          }
          ++ptile;
        }
      }
      // drain: every load this thread issued has landed before the CTA exits
      if (!ok || *abort_flag) {
        const uint32_t first = scount > (uint32_t)nst ? scount - nst : 0;
        for (uint32_t s = first; s < scount; ++s) {
          if (p.fault_inject == 1 && s == 0) continue;
          drain_wait(bar_full(s % nst), (s / nst) & 1, tmo);
        }
        if (it > 0) drain_wait(bar_qfull, (it - 1) & 1, tmo);
      }
      PT_FLUSH(0, true);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    // One MMA chain per key tile covering every query of the item (N = ncols),
    // into TMEM slot tcount & 1 (double buffered).  Lane 0 alone runs the loop:
    // the fewest instructions between a freed slot and the issued MMAs (this
    // warp shares its SM sub-partition with three busy epilogue warps).
    if (lane == 0) {
      PT_DECL
      uint32_t tcount = 0, st = 0, ph = 0;
      int it = 0;
      bool ok = true;
      const uint32_t idesc = B1 ? 0u : idesc_bf16(128, pl.ncols);
      uint32_t idesc_k[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) idesc_k[kk] = idesc_mxf8(128, pl.ncols, kk);
      const uint64_t a_desc0 = sw128_kmajor_desc(sbase + pl.k_off, 0);    // stage 0, K step 0
      const uint64_t b_desc0 = sw128_kmajor_desc(sbase + pl.q_off, 0);    // chunk 0, K step 0
      const uint64_t sf_desc0 = sf_src_desc(sbase + pl.sfa_tx_off);       // stage 0 key scales
      if (F8) {
        // per-vector FP8 runs on the block-scaled MMA: the key rows' scales
        // arrive per tile like MXFP8's (each replicated over the row's four
        // blocks); the query rows' scales are folded into the head weights,
        // so every query-scale atom holds 2^0 (0x7F), copied in once
        uint32_t* unit = reinterpret_cast<uint32_t*>(smem + pl.sfb_tx_off);
        for (int l = 0; l < kSfTxBytes / 4; ++l) unit[l] = 0x7F7F7F7Fu;
        fence_proxy_async_smem();
        tc_fence_after();
        for (int a = 0; a < pl.sfb_atoms; ++a)
          tc_cp_32x128b_warpx4(tmem + kSfbCol + 4 * a, sf_src_desc(sbase + pl.sfb_tx_off));
      }
      for (int r = 0; ok && r * G < nitems; ++r) {
        const int i = item_index(r, nitems);
        if (i < 0) continue;
        const Item m = load_item(p, i);
        if (m.ntiles == 0) continue;
        PT_MARK();
        if (!mbar_wait(bar_qfull, it & 1, abort_flag, status, tmo)) {
          ok = false;
          break;
        }
        PT_ADD(0);
        if (MX) {   // query scales of the item, re-laid out for tcgen05.cp
          for (int a = 0; a < pl.sfb_atoms; ++a) {
            const uint32_t* raw = reinterpret_cast<const uint32_t*>(smem + pl.sfb_raw_off + a * kSfRawBytes);
            uint4* tx = reinterpret_cast<uint4*>(smem + pl.sfb_tx_off + a * kSfTxBytes);
            for (int l = 0; l < 32; ++l) tx[l] = make_uint4(raw[l], raw[l + 32], raw[l + 64], raw[l + 96]);
          }
          fence_proxy_async_smem();
          tc_fence_after();
          for (int a = 0; a < pl.sfb_atoms; ++a)
            tc_cp_32x128b_warpx4(tmem + kSfbCol + 4 * a, sf_src_desc(sbase + pl.sfb_tx_off + a * kSfTxBytes));
        }
        for (int t = 0; t < m.ntiles; ++t) {
          const uint32_t slot = tcount & 1;
          PT_MARK();
          if (tcount >= 2 && !mbar_wait(bar_tempty(slot), ((tcount >> 1) - 1) & 1, abort_flag, status, tmo)) {
            ok = false;
            break;
          }
          PT_ADD(1);
          TRACE(0, tcount, true);   // the tile's TMEM slot is free
          const uint32_t d_tmem = tmem + slot * pl.ncols;
          const uint32_t sfa = tmem + kSfaCol + 4 * (tcount & 1);   // alternates per tile
          for (int c = 0; c < pl.chunks; ++c) {
            if (!mbar_wait(bar_full(st), ph, abort_flag, status, tmo)) {
              ok = false;
              break;
            }
            TRACE(14, tcount, c == 0);   // the tile's K stage has landed
            tc_fence_after();
            // descriptors: start address field + 2 per 32-byte K step
            const uint64_t ad0 = a_desc0 + (uint64_t)(st * (kStageBytes >> 4));
            const uint64_t bd0 = b_desc0 + (uint64_t)(c * (pl.qchunk >> 4));
            if (B1)   // key scales arrive laid out for tcgen05.cp with the stage
              tc_cp_32x128b_warpx4(sfa, sf_desc0 + (uint64_t)(st * (kSfTxBytes >> 4)));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
              if (B1)
                mma_mxf8(d_tmem, ad0 + 2 * kk, bd0 + 2 * kk, idesc_k[kk], sfa, tmem + kSfbCol, acc);
              else
                mma_bf16(d_tmem, ad0 + 2 * kk, bd0 + 2 * kk, idesc, acc);
            }
            tc_commit(bar_empty(st));
            if (++st == (uint32_t)nst) {
              st = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          PT_ADD(3);
          TRACE(1, tcount, true);   // MMAs of the tile issued
          tc_commit(bar_tfull(slot));
          ++tcount;
        }
        if (!ok) break;
        tc_commit(bar_qempty);
        ++it;
      }
      tc_commit(bar_drain);
      drain_wait(bar_drain, 0, tmo);
      PT_FLUSH(8, true);
    }
    __syncwarp();
  } else {
    // ======================= epilogue warpgroups =======================
    // EW warpgroups; warpgroup v owns qpw consecutive queries of the item (one
    // query at 64 heads).  Thread `row` owns key row `row` of every tile.
    const int v = (warp - kEpiWarp0) >> 2;
    const int wq = warp & 3;                      // TMEM lane quarter = key rows wq*32..
    const int row = wq * 32 + (int)lane;          // key row of the tile owned by this thread
    const int tid = row;                          // thread index inside the warpgroup
    const int bar_id = 1 + v;
    const int bar_all = 1 + EW;                   // all epilogue warps
    const int keep = pl.keep, C = pl.cand, W = p.out_width;
    const int qpw = pl.qpw;                       // queries of this warpgroup
    const int qpw_eff = QPW_MAX == 1 ? 1 : qpw;   // compile-time when a warpgroup owns one query
    const int lq0 = v * qpw;                      // first of them, local to the item
    const int col0 = lq0 * H;                     // their first accumulator column
    uint32_t* ckey_base = reinterpret_cast<uint32_t*>(smem + pl.cand_key_off) + lq0 * C;
    uint16_t* cidx_base = reinterpret_cast<uint16_t*>(smem + pl.cand_idx_off) + lq0 * C;
    const uint32_t ckey_s = smem_u32(ckey_base), cidx_s = smem_u32(cidx_base);   // shared-window addresses
    float* w_s = reinterpret_cast<float*>(smem + pl.w_off) + lq0 * H;
    int* hist = reinterpret_cast<int*>(smem + pl.hist_off) + v * 256;
    int* ms = reinterpret_cast<int*>(smem + pl.misc_off) + v * kMiscInts;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    // Key row whose score this thread reports: its own lane's row, except in
    // the fragment layout, where lane t ends with row t/4 + 8 (t % 4) of its
    // warp's rows; rmask marks the lanes whose rows precede it (ballot prefix in
    // row order, so appends stay in index order).
    const int orow = FRAG ? wq * 32 + (int)(lane >> 2) + 8 * (int)(lane & 3) : row;
    uint32_t rmask = 0u;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
      const int rl = FRAG ? (l >> 2) + 8 * (l & 3) : l;
      if (rl < orow - wq * 32) rmask |= 1u << l;
    }
    uint32_t tcount = 0, nbatch = 0;
    bool aborted = false;
    PT_DECL
    for (int r = 0; !aborted && r * G < nitems; ++r) {
      const int i = item_index(r, nitems);
      if (i < 0) continue;
      const Item m = load_item(p, i);
      const int qbase = m.t0 + lq0;               // local position of query qi = 0
      const int a = p.cu_seqlens[m.doc];
      for (int e = tid; e < qpw * H; e += 128) {
        const int t = qbase + e / H;
        float wv = 0.f;
        if (t < m.L) {
          const size_t off = (size_t)(a + t) * H + (e % H);
          wv = p.w_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.w)[off])
                        : reinterpret_cast<const float*>(p.w)[off];
          if (F8) wv = ldexpf(wv, (int)p.q_scale_vec[off] - 127);   // the q row's scale folded into w
        }
        w_s[e] = wv;
      }
      int count[QPW_MAX];
      uint32_t tau[QPW_MAX];
      int vis_lim[QPW_MAX];   // last visible key (or complete pool) of each query; -1 = none
#pragma unroll
      for (int qi = 0; qi < QPW_MAX; ++qi) {
        count[qi] = 0;
        tau[qi] = 0u;
        const int tq = qbase + qi;
        vis_lim[qi] = tq >= m.L ? -1 : (p.pool > 1 ? (tq + 1) / p.pool - 1 : m.off + tq);
      }
      named_bar_sync(bar_id, 128);
      // fragment path: this thread's 16 head weights stay in registers for the item
      float2 wp[FRAG ? 8 : 1];
      if constexpr (FRAG) {
#pragma unroll
        for (int i = 0; i < 8; ++i) wp[i] = *reinterpret_cast<const float2*>(w_s + 8 * i + 2 * (lane & 3));
      }
      PT_ADD(5);
      for (int tb = 0; tb < m.ntiles; tb += kBatch) {
        // ---- score kBatch tiles; keep keys and ballots in registers ----
        uint32_t bkey[kBatch][QPW_MAX];
        uint32_t bbal[kBatch][QPW_MAX];
        bool ok_all = true;
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
#pragma unroll
          for (int qi = 0; qi < QPW_MAX; ++qi) {
            bkey[b][qi] = 0u;
            bbal[b][qi] = 0u;
          }
          const int t = tb + b;
          if (t < m.ntiles) {
            const uint32_t slot = tcount & 1;
            ok_all &= mbar_wait(bar_tfull(slot), (tcount >> 1) & 1, abort_flag, status, tmo);
            PT_ADD(0);
            TRACE(2 + v, tcount, tid == 0);   // warpgroup v woke on the tile's accumulator
            tc_fence_after();
            const int s_idx = t * kTileKeys + orow;     // local key (or pool) index of the reported row
            const float kfac = p.sm_scale;
            if constexpr (FRAG) {
              // Fragment layout (.16x256b): thread t holds 16 heads (2(t%4) + 8i, +1) of
              // the four key rows g, g+8, g+16, g+24 (g = t/4) of its warp's 32 rows, so
              // its head weights fit in registers.  Row sums are then reduced over the
              // four threads of a row group and moved to lane = row.
              const uint32_t tcol = tmem + lane_base + slot * pl.ncols + col0;
              float2 acc[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) acc[j] = make_float2(0.f, 0.f);
              auto frag_sum = [&](const uint32_t* f, float2& a0, float2& a1) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  a0 = ffma2(wp[i], make_float2(fmaxf(__uint_as_float(f[4 * i]), 0.f),
                                                fmaxf(__uint_as_float(f[4 * i + 1]), 0.f)), a0);
                  a1 = ffma2(wp[i], make_float2(fmaxf(__uint_as_float(f[4 * i + 2]), 0.f),
                                                fmaxf(__uint_as_float(f[4 * i + 3]), 0.f)), a1);
                }
              };
              auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_tempty(slot));   // slot free for the MMA warp
                PT_ADD(6);
                TRACE(6 + v, tcount, tid == 0);   // warpgroup v released the slot
              };
              uint32_t fa[32];
              if constexpr (GRP == 64) {   // the second half loads while the first is summed
                uint32_t fb[32];
                tmem_ld_16x256b_x8(tcol, fa);
                tmem_wait_tied<16>(fa);
                tmem_wait_tied<16>(fa + 16);
                tmem_ld_16x256b_x8(tcol + (16u << 16), fb);
                frag_sum(fa, acc[0], acc[1]);
                tmem_wait_tied<16>(fb);
                tmem_wait_tied<16>(fb + 16);
                release();
                frag_sum(fb, acc[2], acc[3]);
              } else {                      // one half at a time (fewer registers)
                tmem_ld_16x256b_x8(tcol, fa);
                tmem_wait_tied<16>(fa);
                tmem_wait_tied<16>(fa + 16);
                frag_sum(fa, acc[0], acc[1]);
                tmem_ld_16x256b_x8(tcol + (16u << 16), fa);
                tmem_wait_tied<16>(fa);
                tmem_wait_tied<16>(fa + 16);
                release();
                frag_sum(fa, acc[2], acc[3]);
              }
              // reduce-scatter over the 4 lanes of a row group: lane t ends with the
              // total of row g + 8 (t % 4)
              const float s0 = acc[0].x + acc[0].y, s1 = acc[1].x + acc[1].y;
              const float s2 = acc[2].x + acc[2].y, s3 = acc[3].x + acc[3].y;
              const bool b1 = (lane >> 1) & 1u, b0 = lane & 1u;
              const float k0 = (b1 ? s2 : s0) + __shfl_xor_sync(0xffffffffu, b1 ? s0 : s2, 2);
              const float k1 = (b1 ? s3 : s1) + __shfl_xor_sync(0xffffffffu, b1 ? s1 : s3, 2);
              const float own = (b0 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, b0 ? k0 : k1, 1);
              const float sv = own * kfac;   // row orow
              const bool vis = s_idx <= vis_lim[0];
              bkey[b][0] = orderable_key(sv);
              bbal[b][0] = __ballot_sync(0xffffffffu, vis && bkey[b][0] > tau[0]);
            } else {
              float2 part[QPW_MAX][NCH];
#pragma unroll
              for (int qi = 0; qi < QPW_MAX; ++qi)
#pragma unroll
                for (int c = 0; c < NCH; ++c) part[qi][c] = make_float2(0.f, 0.f);
              // TMEM -> registers in groups of GRP columns (load, wait, reduce); the
              // slot goes back to the MMA warp as soon as the last group has landed.
              // sum_j w_j * ReLU(acc_j) with NCH independent FFMA2 chains per query.
              const uint32_t taddr = tmem + lane_base + slot * pl.ncols + col0;
#pragma unroll
              for (int gi = 0; gi < NGRP; ++gi) {
                uint32_t cb[GRP / CK][CK];
#pragma unroll
                for (int c = 0; c < GRP / CK; ++c) tmem_load_cols<CK>(taddr + gi * GRP + c * CK, cb[c]);
#pragma unroll
                for (int c = 0; c < GRP / CK; ++c) tmem_wait_tied<CK>(cb[c]);
                if (gi == NGRP - 1) {
                  tc_fence_before();
                  __syncwarp();
                  if (lane == 0) mbar_arrive(bar_tempty(slot));   // slot free for the MMA warp
                  PT_ADD(6);
                  TRACE(6 + v, tcount, tid == 0);   // warpgroup v released the slot
                }
#pragma unroll
                for (int c = 0; c < GRP / CK; ++c) {
#pragma unroll
                  for (int j4 = 0; j4 < CK / 4; ++j4) {
                    const int col = gi * GRP + c * CK + 4 * j4;
                    const int qi = col / H, hh = col % H;
                    if (qi < qpw_eff) {
                      const float4 wv = *reinterpret_cast<const float4*>(w_s + qi * H + hh);
                      const uint32_t* x = cb[c] + 4 * j4;
                      const float2 r0 = make_float2(fmaxf(__uint_as_float(x[0]), 0.f), fmaxf(__uint_as_float(x[1]), 0.f));
                      const float2 r1 = make_float2(fmaxf(__uint_as_float(x[2]), 0.f), fmaxf(__uint_as_float(x[3]), 0.f));
                      float2& pc = part[qi][(hh / 4) % NCH];
                      pc = ffma2(make_float2(wv.x, wv.y), r0, pc);
                      pc = ffma2(make_float2(wv.z, wv.w), r1, pc);
                    }
                  }
                }
              }
#pragma unroll
              for (int qi = 0; qi < QPW_MAX; ++qi) {
                if (qi < qpw_eff) {
                  float sv = 0.f;
#pragma unroll
                  for (int c = 0; c < NCH; ++c) sv += part[qi][c].x + part[qi][c].y;
                  sv *= kfac;
                  const bool vis = s_idx <= vis_lim[qi];
                  bkey[b][qi] = orderable_key(sv);
                  bbal[b][qi] = __ballot_sync(0xffffffffu, vis && bkey[b][qi] > tau[qi]);
                }
              }
            }
            TRACE(10 + v, tcount, tid == 0);   // warpgroup v finished the tile's arithmetic
            ++tcount;
            PT_ADD(1);
          }
        }
        // ---- append the batch in index order: one warpgroup barrier ----
        int* bcnt = ms + MS_BCNT + (nbatch & 1) * (kBatch * kMaxQpw * 4);
        if (lane == 0) {
#pragma unroll
          for (int b = 0; b < kBatch; ++b)
#pragma unroll
            for (int qi = 0; qi < QPW_MAX; ++qi) bcnt[(b * kMaxQpw + qi) * 4 + wq] = __popc(bbal[b][qi]);
        }
        ++nbatch;
        named_bar_sync(bar_id, 128);      // batch counts of this warpgroup visible
        TRACE(5, nbatch, tid == 0 && v == 0 && EW < 4);   // batch counts exchanged
#pragma unroll
        for (int qi = 0; qi < QPW_MAX; ++qi) {
          if (qi < qpw_eff) {
            // the query's counts for the whole batch first: no load waits behind an append
            int4 cc[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) cc[b] = *reinterpret_cast<const int4*>(bcnt + (b * kMaxQpw + qi) * 4);
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
              const int before = (wq > 0 ? cc[b].x : 0) + (wq > 1 ? cc[b].y : 0) + (wq > 2 ? cc[b].z : 0);
              const int rel = count[qi] + before + __popc(bbal[b][qi] & rmask);
              const bool mine = ((bbal[b][qi] >> lane) & 1u) && DSA_IN_BOUNDS(rel < C, status);
              const int pos = qi * C + rel;
              st_shared_u32_if(mine, ckey_s + 4u * (uint32_t)pos, bkey[b][qi]);
              st_shared_u16_if(mine, cidx_s + 2u * (uint32_t)pos, (uint16_t)((tb + b) * kTileKeys + orow));
              count[qi] += cc[b].x + cc[b].y + cc[b].z + cc[b].w;
            }
          }
        }
        PT_ADD(2);
        TRACE(9, nbatch, tid == 0 && v == 0 && EW < 4);   // batch appended
        // ---- room for the next batch, or shrink: all warpgroups together ----
        // Every VOTE-th batch of the item, one vote over every epilogue
        // thread decides, uniformly, whether to abort and whether to shrink
        // (room for the batches up to the next vote); shrinking in lockstep
        // lets the queries' compactions overlap instead of stalling the shared
        // TMEM ring one after another.  One barrier carries both votes: lane 0
        // of each warp reports an abort, lanes 1..31 a shrink, so the count it
        // returns is (warps aborting) + 31 * (warps needing room), with at most
        // 16 warps.  The item's last batch needs no vote: the final selection
        // follows, and an abort is caught at the next item's first vote.
        PT_ADD(3);
        if ((tb / kBatch) % VOTE != VOTE - 1 || tb + kBatch >= m.ntiles) continue;
        bool need = false;
#pragma unroll
        for (int qi = 0; qi < QPW_MAX; ++qi)
          need |= qi < qpw_eff && count[qi] + VOTE * kBatch * kTileKeys > C;
        need = __any_sync(0xffffffffu, need);
        const bool warp_abort = __any_sync(0xffffffffu, !ok_all || *abort_flag);
        const int votes = named_bar_popc(bar_all, EW * 128, lane == 0 ? warp_abort : need);
        if (votes % 31 != 0) {
          aborted = true;
          break;
        }
        TRACE(13, nbatch, tid == 0 && v == 0 && EW < 4);   // vote taken
        if (votes != 0) {
#pragma unroll
          for (int qi = 0; qi < QPW_MAX; ++qi) {
            if (qi < qpw_eff && count[qi] > keep + kTileKeys) {
              named_bar_sync(bar_id, 128);   // appends visible to the whole warpgroup
              const int cap = C - (VOTE * kBatch + 2) * kTileKeys;
              int kept;
              uint32_t th;
              if (wg_shrink_sampled<compact_per<PREC>()>(ckey_base + qi * C, cidx_base + qi * C, count[qi], keep, cap, wq,
                                    lane, ms, bar_id, &th, &kept DSA_CHK_ARG)) {
                tau[qi] = th;
              } else {
                tau[qi] = wg_select<compact_per<PREC>()>(ckey_base + qi * C, cidx_base + qi * C, count[qi], keep, false,
                                    cap, wq, lane, hist, ms, bar_id, &kept DSA_CHK_ARG);
              }
              count[qi] = kept;
            }
          }
        }
        PT_ADD(3);
      }
      if (aborted) break;
      named_bar_sync(bar_id, 128);
      // finalize: exactly min(keep, visible) entries per query, ascending index
#pragma unroll
      for (int qi = 0; qi < QPW_MAX; ++qi) {
        if (qi < qpw_eff && count[qi] > keep) {
          int kept;
          wg_select<compact_per<PREC>()>(ckey_base + qi * C, cidx_base + qi * C, count[qi], keep, true, keep, wq, lane, hist,
                    ms, bar_id, &kept DSA_CHK_ARG);
          count[qi] = kept;
        }
      }
      PT_ADD(7);
#pragma unroll
      for (int qi = 0; qi < QPW_MAX; ++qi) {
        const int tq = qbase + qi;
        if (qi >= qpw_eff || tq >= m.L) continue;
        if (!DSA_IN_BOUNDS((int64_t)a + tq < p.out_rows && count[qi] <= C, status)) continue;
        const size_t orow = (size_t)(a + tq) * W;
        const int n = count[qi];
        const uint32_t* ck = ckey_base + qi * C;
        const uint16_t* ci = cidx_base + qi * C;
        if (p.expand) {
          const int P = p.pool;
          const int ntail = p.tail ? (tq + 1) % P : 0;
          const int tail0 = P * ((tq + 1) / P);
          for (int e = tid; e < W; e += 128) {
            int id = -1;
            float sc = -__int_as_float(0x7f800000);
            if (e < n * P) {
              id = (int)ci[e / P] * P + (e % P);
              sc = key_to_float(ck[e / P]);
            } else if (e < n * P + ntail) {
              id = tail0 + (e - n * P);
              sc = __int_as_float(0x7f800000);
            }
            p.out_idx[orow + e] = id;
            if (p.out_score) p.out_score[orow + e] = sc;
          }
          if (tid == 0 && p.out_len) p.out_len[a + tq] = n * P + ntail;
        } else {
          for (int e = tid; e < W; e += 128) {
            const bool vv = e < n;
            p.out_idx[orow + e] = vv ? (int)ci[e] : -1;
            if (p.out_score) p.out_score[orow + e] = vv ? key_to_float(ck[e]) : -__int_as_float(0x7f800000);
          }
          if (tid == 0 && p.out_len) p.out_len[a + tq] = n;
        }
      }
      named_bar_sync(bar_id, 128);
      PT_ADD(4);
    }
    PT_FLUSH(16 + 8 * v, tid == 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------------------
// diagnostic: one raw tcgen05 tile (128 key rows x n_cols query rows)
// ----------------------------------------------------------------------------

template <int PREC>
__global__ void __launch_bounds__(128, 1) debug_mma_tile_kernel(const __grid_constant__ DebugParams p) {
  constexpr bool MX = PREC == PREC_MXFP8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  // layout: q chunks | k chunks | sfa raw | sfb raw | sfa tx | sfb tx | barriers
  const int q_off = 0, k_off = p.chunks * kStageBytes, sfa_raw = 2 * p.chunks * kStageBytes;
  const int sfb_raw = sfa_raw + kSfRawBytes, sfa_tx = sfb_raw + kSfRawBytes, sfb_tx = sfa_tx + kSfTxBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sfb_tx + kSfTxBytes);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 5);
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(bars + 0), 1);
    mbar_init(smem_u32(bars + 1), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int chunk_elems = kChunkBytes / (MX ? 1 : 2);
  if (threadIdx.x == 0) {
    const uint32_t bytes = 2 * p.chunks * kStageBytes + (MX ? 2 * kSfRawWords * 4 : 0);
    mbar_arrive_expect_tx(smem_u32(bars + 0), bytes);
    for (int c = 0; c < p.chunks; ++c) {
      tma_load_2d(sbase + q_off + c * kStageBytes, &p.tm_q, smem_u32(bars + 0), c * chunk_elems,
                  (int)p.q_row0);
      tma_load_2d(sbase + k_off + c * kStageBytes, &p.tm_k, smem_u32(bars + 0), c * chunk_elems,
                  (int)p.k_row0);
    }
    if (MX) {
      tma_load_1d(sbase + sfa_raw, &p.tm_ks, smem_u32(bars + 0), (int)(p.k_row0 & ~3LL));
      tma_load_1d(sbase + sfb_raw, &p.tm_qs, smem_u32(bars + 0), (int)(p.q_row0 & ~3LL));
    }
  }
  bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bars + 0), 0, abort_flag, p.status, p.timeout_ns));
  if (warp == 1 && ok) {
    if (MX) {
      transpose_scales(reinterpret_cast<const uint32_t*>(smem + sfa_raw), (int)(p.k_row0 & 3),
                       reinterpret_cast<uint32_t*>(smem + sfa_tx), lane);
      transpose_scales(reinterpret_cast<const uint32_t*>(smem + sfb_raw), (int)(p.q_row0 & 3),
                       reinterpret_cast<uint32_t*>(smem + sfb_tx), lane);
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) {
      tc_fence_after();
      if (MX) {
        tc_cp_32x128b_warpx4(tmem + 384, sf_src_desc(sbase + sfa_tx));
        tc_cp_32x128b_warpx4(tmem + 392, sf_src_desc(sbase + sfb_tx));
      }
      for (int c = 0; c < p.chunks; ++c)
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sw128_kmajor_desc(sbase + k_off + c * kStageBytes, kk * 32);
          const uint64_t bd = sw128_kmajor_desc(sbase + q_off + c * kStageBytes, kk * 32);
          const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
          if (MX)
            mma_mxf8(tmem, ad, bd, idesc_mxf8(128, p.n_cols, kk), tmem + 384, tmem + 392, acc);
          else
            mma_bf16(tmem, ad, bd, idesc_bf16(128, p.n_cols), acc);
        }
      tc_commit(smem_u32(bars + 1));
    }
    __syncwarp();
  }
  ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(bars + 1), 0, abort_flag, p.status, p.timeout_ns));
  tc_fence_after();
  if (ok) {
    const int rowi = warp * 32 + (int)lane;
    for (int c0 = 0; c0 < p.n_cols; c0 += 16) {
      uint32_t v[16];
      tmem_ld_x16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
      tmem_ld_wait();
      for (int j = 0; j < 16 && c0 + j < p.n_cols; ++j)
        p.out[(size_t)rowi * p.n_cols + c0 + j] = __uint_as_float(v[j]);
    }
  } else if (warp == 1 && lane == 0) {
    drain_wait(smem_u32(bars + 0), 0, p.timeout_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------------------
// launchers (called from api.cu)
// ----------------------------------------------------------------------------
cudaError_t launch_build_worklist(const int32_t* cu, const int32_t* cu_k, const int32_t* cu_comp, int num_seqs,
                                  int total_tokens, int total_k, int max_seqlen, int max_seqlen_k, int tq,
                                  int pool, int2* items, int* doc_prefix, int* tile_base, int* hdr,
                                  int max_items, cudaStream_t stream) {
  build_worklist_kernel<<<1, kWLThreads, 0, stream>>>(cu, cu_k, cu_comp, num_seqs, total_tokens, total_k, max_seqlen,
                                                      max_seqlen_k, tq, pool, items, doc_prefix, tile_base,
                                                      hdr, max_items);
  return cudaGetLastError();
}

cudaError_t launch_tiled_kscales(const uint8_t* k_scale, int64_t k_rows, int replicate, const int32_t* cu_keys,
                                 const int* tile_base, int num_seqs, int max_tiles, uint32_t* out,
                                 int sm_count, cudaStream_t stream) {
  int grid = max_tiles < sm_count * 8 ? max_tiles : sm_count * 8;
  if (grid < 1) grid = 1;
  build_tiled_kscales_kernel<<<grid, 128, 0, stream>>>(k_scale, k_rows, replicate, cu_keys, tile_base, num_seqs,
                                                       max_tiles, out);
  return cudaGetLastError();
}

cudaError_t launch_validate_inputs(const void* q, int64_t q_bytes, const void* k, int64_t k_bytes, int op_bf16,
                                   const uint8_t* qs, int64_t qs_bytes, const uint8_t* ks, int64_t ks_bytes,
                                   const void* w, int64_t w_elems, int w_bf16, int* hdr, int sm_count,
                                   cudaStream_t stream) {
  validate_inputs_kernel<<<sm_count * 4, 256, 0, stream>>>(
      reinterpret_cast<const uint8_t*>(q), q_bytes, reinterpret_cast<const uint8_t*>(k), k_bytes, op_bf16, qs, qs_bytes,
      ks, ks_bytes, w, w_elems, w_bf16, hdr);
  return cudaGetLastError();
}

template <int PREC, int H>
static cudaError_t launch_score_t(const ScoreParams& p, int grid, cudaStream_t stream) {
  auto kern = score_topk_kernel<PREC, H>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.plan.total);
  if (e != cudaSuccess) return e;
  kern<<<grid, score_threads(PREC), p.plan.total, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_score_topk(const ScoreParams& p, int grid, cudaStream_t stream) {
  const int H = p.plan.n_heads;
  if (p.plan.prec == PREC_FP8) {
    switch (p.plan.n_heads) {
      case 4: return launch_score_t<PREC_FP8, 4>(p, grid, stream);
      case 8: return launch_score_t<PREC_FP8, 8>(p, grid, stream);
      case 16: return launch_score_t<PREC_FP8, 16>(p, grid, stream);
      case 32: return launch_score_t<PREC_FP8, 32>(p, grid, stream);
      case 64: return launch_score_t<PREC_FP8, 64>(p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.plan.prec == PREC_BF16) {
    switch (H) {
      case 4: return launch_score_t<PREC_BF16, 4>(p, grid, stream);
      case 8: return launch_score_t<PREC_BF16, 8>(p, grid, stream);
      case 16: return launch_score_t<PREC_BF16, 16>(p, grid, stream);
      case 32: return launch_score_t<PREC_BF16, 32>(p, grid, stream);
      case 64: return launch_score_t<PREC_BF16, 64>(p, grid, stream);
    }
  } else {
    switch (H) {
      case 4: return launch_score_t<PREC_MXFP8, 4>(p, grid, stream);
      case 8: return launch_score_t<PREC_MXFP8, 8>(p, grid, stream);
      case 16: return launch_score_t<PREC_MXFP8, 16>(p, grid, stream);
      case 32: return launch_score_t<PREC_MXFP8, 32>(p, grid, stream);
      case 64: return launch_score_t<PREC_MXFP8, 64>(p, grid, stream);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_debug_mma_tile(const DebugParams& p, int prec, cudaStream_t stream) {
  const int smem = 2 * p.chunks * kStageBytes + 2 * kSfRawBytes + 2 * kSfTxBytes + 128 + 1024;
  if (prec == PREC_BF16) {
    auto k = debug_mma_tile_kernel<PREC_BF16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k<<<1, 128, smem, stream>>>(p);
  } else {
    auto k = debug_mma_tile_kernel<PREC_MXFP8>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k<<<1, 128, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

#ifdef DSA_PHASE_TIMERS
extern "C" void dsa_idx_debug_phase_timers(unsigned long long* out64, int reset) {
  cudaMemcpyFromSymbol(out64, g_phase_cycles, sizeof(unsigned long long) * 64);
  if (reset) {
    unsigned long long z[64] = {0};
    cudaMemcpyToSymbol(g_phase_cycles, z, sizeof(z));
  }
}
#endif

#ifdef DSA_TRACE
extern "C" void dsa_idx_debug_trace(long long* out) {
  cudaMemcpyFromSymbol(out, g_trace, sizeof(long long) * 16 * 256);
}
#endif

}  // namespace dsa
