// Fused DSA lightning-indexer score + streaming top-k for sm_103a.
//
// What it computes (Megatron-LM PR #8403 "cuDNN DSA indexer precision
// options", review findings 1-3; PR #5992 "[DeepSeek-V4] Add compact BF16 and
// MXFP8 DSA indexer support", "Key changes"; PR #7522 "KPool (pooled-key) DSA
// indexer support", "Changes"):
//   I[t,s] = sm_scale * sum_j w[t,j] * ReLU(q[t,j] . k[s])  for visible s,
//   then the `keep` best s per query t, ties to the lower index.
//
// Design (one persistent CTA per SM, 320 threads):
//   * A work item is a block of Tq = 2*qs consecutive queries of one document.
//     Its q rows (Tq*H rows of the [T*H, D] operand) stay in shared memory as
//     two UMMA B operands ("sub-blocks", N = qs*H columns each).
//   * Warp 0 streams the item's visible keys in tiles of 128 rows through a
//     ring of shared-memory stages with TMA (128-byte swizzle).
//   * Warp 1 issues tcgen05.mma (M = 128 keys, N = qs*H, K = head_dim) into a
//     ring of 128-column TMEM accumulator slots; BF16 uses kind::f16, MXFP8 the
//     block-scaled kind::mxf8f6f4 with UE8M0 scales copied into TMEM.
//   * Warps 2..9 are two epilogue warpgroups, one per sub-block.  Thread r of a
//     warpgroup owns key row r of the tile: it loads its row's qs*H fp32
//     accumulators with tcgen05.ld, applies ReLU and the head weights, masks
//     invisible keys, and offers each query's score to that query's candidate
//     buffer in shared memory.  Candidates above the running threshold are
//     appended in index order; when a buffer is full a radix select keeps
//     exactly `keep` entries and raises the threshold.  Scores never reach HBM.
//   * Every wait is bounded (status word + abort flag, no trap); see
//     dsa_device.cuh.
#include <cuda_bf16.h>

#include "dsa_device.cuh"
#include "dsa_params.h"

namespace dsa {

// ----------------------------------------------------------------------------
// Work list: items (document, first query) sorted by descending tile count so
// the persistent CTAs take the longest items first.  One block.
// ----------------------------------------------------------------------------
constexpr int kWLThreads = 1024;
constexpr int kWLMaxBins = 1025;

__global__ void __launch_bounds__(kWLThreads) build_worklist_kernel(
    const int32_t* __restrict__ cu, int num_seqs, int total_tokens, int max_seqlen, int tq,
    int pool, int2* __restrict__ items, int* __restrict__ doc_prefix, int* __restrict__ hdr,
    int max_items) {
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
  // validate cu_seqlens
  for (int d = tid; d < num_seqs; d += kWLThreads) {
    const int a = cu[d], b = cu[d + 1];
    if (b < a || b - a > max_seqlen) s_bad = 1;
  }
  if (tid == 0 && (cu[0] != 0 || cu[num_seqs] != total_tokens)) s_bad = 1;
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
    int t_end = (blk + 1) * tq;
    if (t_end > L) t_end = L;
    const int nk = pool > 1 ? t_end / pool : t_end;
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

// ----------------------------------------------------------------------------
// helpers of the fused kernel
// ----------------------------------------------------------------------------
struct Item {
  int doc, t0, L, qrow0, krow0, ntiles;
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
  int t_end = m.t0 + kG * p.plan.qs;
  if (t_end > m.L) t_end = m.L;
  const int nk = p.pool > 1 ? t_end / p.pool : t_end;
  m.ntiles = (nk + kTileKeys - 1) / kTileKeys;
  return m;
}

// Bounded wait used while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
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
  MS_WCNT = 0,          // [2][kMaxQs][4] append counts
  MS_WTOT = 64,         // [4] scan warp totals
  MS_DIGIT = 68,
  MS_ABOVE = 69,
  MS_BIN = 70,
  MS_GT = 72,           // [4]
  MS_EQ = 76,           // [4]
};

// Keep exactly `keep` of the n (> keep) candidates of one query: the largest
// keys, ties to the earlier buffer position (= lower index, the buffer is in
// index order).  Stable in place.  Returns a threshold key: every future
// candidate must be strictly larger.  All 128 threads of the warpgroup.
template <int MMAX>
__device__ __noinline__ uint32_t wg_select(uint32_t* keys, uint16_t* idx, int n, int keep, int wq,
                              uint32_t lane, int* hist, int* ms, int bar_id) {
  const int tid = wq * 32 + (int)lane;
  const int span = ((n + 127) >> 7) << 5;    // entries per warp, multiple of 32
  const int base = wq * span;
  uint32_t rk[MMAX];
  uint32_t ri[MMAX];
#pragma unroll
  for (int m = 0; m < MMAX; ++m) {
    const int e = base + m * 32 + (int)lane;
    const bool ok = (m * 32 < span) && (e < n);
    rk[m] = ok ? keys[e] : 0u;
    ri[m] = ok ? (uint32_t)idx[e] : 0u;
  }
  uint32_t prefix = 0, pmask = 0;
  int kk = keep;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += 128) hist[b] = 0;
    named_bar_sync(bar_id, 128);
#pragma unroll
    for (int m = 0; m < MMAX; ++m) {
      const int e = base + m * 32 + (int)lane;
      if ((m * 32 < span) && (e < n) && ((rk[m] & pmask) == prefix))
        atomicAdd(&hist[(rk[m] >> shift) & 0xFFu], 1);
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
    if (bin == kk) break;   // the whole bin is kept: threshold found early (uniform)
  }
  // stable compaction: keep (key & pmask) > prefix, and the first kk with == prefix
  int gt = 0, eq = 0;
#pragma unroll
  for (int m = 0; m < MMAX; ++m) {
    const int e = base + m * 32 + (int)lane;
    const bool v = (m * 32 < span) && (e < n);
    const uint32_t mk = rk[m] & pmask;
    gt += __popc(__ballot_sync(0xffffffffu, v && mk > prefix));
    eq += __popc(__ballot_sync(0xffffffffu, v && mk == prefix));
  }
  if (lane == 0) {
    ms[MS_GT + wq] = gt;
    ms[MS_EQ + wq] = eq;
  }
  named_bar_sync(bar_id, 128);
  int gbase = 0, ebase = 0;
  for (int w = 0; w < wq; ++w) {
    gbase += ms[MS_GT + w];
    ebase += ms[MS_EQ + w];
  }
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int m = 0; m < MMAX; ++m) {
    const int e = base + m * 32 + (int)lane;
    const bool v = (m * 32 < span) && (e < n);
    const uint32_t mk = rk[m] & pmask;
    const bool g1 = v && mk > prefix;
    const bool e1 = v && mk == prefix;
    const uint32_t bg = __ballot_sync(0xffffffffu, g1);
    const uint32_t be = __ballot_sync(0xffffffffu, e1);
    const int gb = gbase + __popc(bg & lt);
    const int eb = ebase + __popc(be & lt);
    if (g1 || (e1 && eb < kk)) {
      const int pos = gb + (eb < kk ? eb : kk);
      keys[pos] = rk[m];
      idx[pos] = (uint16_t)ri[m];
    }
    gbase += __popc(bg);
    ebase += __popc(be);
  }
  named_bar_sync(bar_id, 128);
  return prefix;
}

// ----------------------------------------------------------------------------
// the fused kernel
// ----------------------------------------------------------------------------
template <int PREC, int H>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_topk_kernel(const __grid_constant__ ScoreParams p) {
  constexpr int QS_MAX = (128 / H) < kMaxQs ? (128 / H) : kMaxQs;
  constexpr bool MX = PREC == PREC_MXFP8;
  const ScorePlan& pl = p.plan;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  // barriers
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pl.bar_off);
  const int nst = pl.nst, S = pl.tslots;
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + kMaxStages + s); };
  auto bar_tfull = [&](int s) { return smem_u32(bars + 2 * kMaxStages + s); };
  auto bar_tempty = [&](int s) { return smem_u32(bars + 2 * kMaxStages + 4 + s); };
  const uint32_t bar_qfull = smem_u32(bars + 2 * kMaxStages + 8);
  const uint32_t bar_qempty = smem_u32(bars + 2 * kMaxStages + 9);
  const uint32_t bar_drain = smem_u32(bars + 2 * kMaxStages + 10);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 12);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kMaxStages + 13);
  int* status = p.hdr;
  const uint64_t tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_tfull(s), 1);
      mbar_init(bar_tempty(s), 4);
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
      uint32_t scount = 0;
      int it = 0;
      bool ok = true;
      const uint32_t q_bytes = kG * pl.chunks * kStageBytes + (MX ? kG * kSfRawWords * 4 : 0);
      const uint32_t k_bytes = kStageBytes + (MX ? kSfRawWords * 4 : 0);
      const int chunk_elems = kChunkBytes / (MX ? 1 : 2);
      for (int r = 0; ok && r * G < nitems; ++r) {
        const int i = item_index(r, nitems);
        if (i < 0) continue;
        const Item m = load_item(p, i);
        if (m.ntiles == 0) continue;
        if (it > 0 && !mbar_wait(bar_qempty, (it - 1) & 1, abort_flag, status, tmo)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar_qfull, q_bytes);
        for (int g = 0; g < kG; ++g) {
          const int row = m.qrow0 + g * pl.nsub;
          for (int c = 0; c < pl.chunks; ++c)
            tma_load_2d(sbase + pl.q_off + (g * pl.chunks + c) * kStageBytes, &p.tm_q, bar_qfull,
                        c * chunk_elems, row);
          if (MX) tma_load_1d(sbase + pl.sfb_raw_off + g * kSfRawBytes, &p.tm_qs, bar_qfull, row);
        }
        ++it;
        for (int t = 0; ok && t < m.ntiles; ++t) {
          const int krow = m.krow0 + t * kTileKeys;
          for (int c = 0; c < pl.chunks; ++c) {
            const int st = scount % nst;
            if (scount >= (uint32_t)nst &&
                !mbar_wait(bar_empty(st), ((scount / nst) - 1) & 1, abort_flag, status, tmo)) {
              ok = false;
              break;
            }
            if (p.fault_inject == 1 && scount == 0) {   // test hook: never load stage 0
              ++scount;
              continue;
            }
            mbar_arrive_expect_tx(bar_full(st), k_bytes);
            tma_load_2d(sbase + pl.k_off + st * kStageBytes, &p.tm_k, bar_full(st),
                        c * chunk_elems, krow);
            if (MX)
              tma_load_1d(sbase + pl.sfa_raw_off + st * kSfRawBytes, &p.tm_ks, bar_full(st),
                          krow & ~3);
            ++scount;
          }
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
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    uint32_t scount = 0, tcount = 0;
    int it = 0;
    bool ok = true;
    const uint32_t idesc = MX ? 0u : idesc_bf16(128, pl.nsub);
    const uint32_t sfa_col = 384, sfb_col = 392;
    for (int r = 0; ok && r * G < nitems; ++r) {
      const int i = item_index(r, nitems);
      if (i < 0) continue;
      const Item m = load_item(p, i);
      if (m.ntiles == 0) continue;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_qfull, it & 1, abort_flag, status, tmo))) {
        ok = false;
        break;
      }
      if (MX) {
        for (int g = 0; g < kG; ++g)
          transpose_scales(reinterpret_cast<const uint32_t*>(smem + pl.sfb_raw_off + g * kSfRawBytes),
                           0, reinterpret_cast<uint32_t*>(smem + pl.sfb_tx_off + g * kSfTxBytes),
                           lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          for (int g = 0; g < kG; ++g)
            tc_cp_32x128b_warpx4(tmem + sfb_col + 4 * g,
                                 sf_src_desc(sbase + pl.sfb_tx_off + g * kSfTxBytes));
        }
        __syncwarp();
      }
      for (int t = 0; ok && t < m.ntiles; ++t) {
        uint32_t slot[kG];
        for (int g = 0; g < kG; ++g) {
          const uint32_t u = tcount * kG + g;
          slot[g] = u % S;
          const bool got = u < (uint32_t)S ||
                           mbar_wait(bar_tempty(slot[g]), ((u / S) - 1) & 1, abort_flag, status, tmo);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        tc_fence_after();
        const int krow = m.krow0 + t * kTileKeys;
        for (int c = 0; c < pl.chunks; ++c) {
          const int st = scount % nst;
          if (!__all_sync(0xffffffffu, mbar_wait(bar_full(st), (scount / nst) & 1, abort_flag, status, tmo))) {
            ok = false;
            break;
          }
          if (MX) {
            transpose_scales(
                reinterpret_cast<const uint32_t*>(smem + pl.sfa_raw_off + st * kSfRawBytes),
                krow & 3, reinterpret_cast<uint32_t*>(smem + pl.sfa_tx_off + st * kSfTxBytes),
                lane);
            fence_proxy_async_smem();
            __syncwarp();
          }
          if (lane == 0) {
            tc_fence_after();
            const uint32_t a_base = sbase + pl.k_off + st * kStageBytes;
            if (MX)
              tc_cp_32x128b_warpx4(tmem + sfa_col + 4 * (st & 1),
                                   sf_src_desc(sbase + pl.sfa_tx_off + st * kSfTxBytes));
            for (int g = 0; g < kG; ++g) {
              const uint32_t b_base = sbase + pl.q_off + (g * pl.chunks + c) * kStageBytes;
              const uint32_t d_tmem = tmem + slot[g] * 128;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sw128_kmajor_desc(a_base, kk * 32);
                const uint64_t bd = sw128_kmajor_desc(b_base, kk * 32);
                const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
                if (MX)
                  mma_mxf8(d_tmem, ad, bd, idesc_mxf8(128, pl.nsub, kk), tmem + sfa_col + 4 * (st & 1),
                           tmem + sfb_col + 4 * g, acc);
                else
                  mma_bf16(d_tmem, ad, bd, idesc, acc);
              }
            }
            tc_commit(bar_empty(st));
          }
          __syncwarp();
          ++scount;
        }
        if (!ok) break;
        if (lane == 0)
          for (int g = 0; g < kG; ++g) tc_commit(bar_tfull(slot[g]));
        __syncwarp();
        ++tcount;
      }
      if (!ok) break;
      if (lane == 0) tc_commit(bar_qempty);
      __syncwarp();
      ++it;
    }
    if (lane == 0) {
      tc_commit(bar_drain);
      drain_wait(bar_drain, 0, tmo);
    }
    __syncwarp();
  } else {
    // ======================= epilogue warpgroups =======================
    const int g = (warp - kEpiWarp0) >> 2;       // sub-block of this warpgroup
    const int wq = warp & 3;                      // TMEM lane quarter = key rows wq*32..
    const int row = wq * 32 + (int)lane;          // key row of the tile owned by this thread
    const int tid = row;                          // thread index inside the warpgroup
    const int bar_id = 1 + g;
    const int qs = pl.qs, keep = pl.keep, C = pl.cand, W = p.out_width;
    uint32_t* ckey_base = reinterpret_cast<uint32_t*>(smem + pl.cand_key_off) + g * qs * C;
    uint16_t* cidx_base = reinterpret_cast<uint16_t*>(smem + pl.cand_idx_off) + g * qs * C;
    float* w_s = reinterpret_cast<float*>(smem + pl.w_off) + g * qs * H;
    int* hist = reinterpret_cast<int*>(smem + pl.hist_off) + g * 256;
    int* ms = reinterpret_cast<int*>(smem + pl.misc_off) + g * kMiscInts;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t tcount = 0;
    bool aborted = false;
    for (int r = 0; !aborted && r * G < nitems; ++r) {
      const int i = item_index(r, nitems);
      if (i < 0) continue;
      const Item m = load_item(p, i);
      const int qbase = m.t0 + g * qs;            // local position of query qi = 0
      const int a = p.cu_seqlens[m.doc];
      for (int e = tid; e < qs * H; e += 128) {
        const int t = qbase + e / H;
        float wv = 0.f;
        if (t < m.L) {
          const size_t off = (size_t)(a + t) * H + (e % H);
          wv = p.w_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.w)[off])
                        : reinterpret_cast<const float*>(p.w)[off];
        }
        w_s[e] = wv;
      }
      int count[QS_MAX];
      uint32_t tau[QS_MAX];
#pragma unroll
      for (int qi = 0; qi < QS_MAX; ++qi) {
        count[qi] = 0;
        tau[qi] = 0u;
      }
      named_bar_sync(bar_id, 128);
      for (int t = 0; t < m.ntiles; ++t) {
        const uint32_t u = tcount * kG + g;
        const uint32_t slot = u % S;
        const bool ok = mbar_wait(bar_tfull(slot), (u / S) & 1, abort_flag, status, tmo);
        tc_fence_after();
        const int s_idx = t * kTileKeys + row;    // local key (or pool) index of this thread
        uint32_t key[QS_MAX];
        bool pass[QS_MAX];
#pragma unroll
        for (int qi = 0; qi < QS_MAX; ++qi) {
          pass[qi] = false;
          key[qi] = 0u;
          if (qi < qs) {
            uint32_t acc[H];
            tmem_load_cols<H>(tmem + lane_base + slot * 128 + qi * H, acc);
            tmem_ld_wait();
            const float* wq_s = w_s + qi * H;
            float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < H; j += 2) {
              const float2 wv = *reinterpret_cast<const float2*>(wq_s + j);
              const float2 rv = make_float2(fmaxf(__uint_as_float(acc[j]), 0.f),
                                            fmaxf(__uint_as_float(acc[j + 1]), 0.f));
              s2 = ffma2(wv, rv, s2);
            }
            const float v = (s2.x + s2.y) * p.sm_scale;
            const int tq = qbase + qi;
            const bool vis = tq < m.L && (p.pool > 1 ? s_idx < (tq + 1) / p.pool : s_idx <= tq);
            key[qi] = orderable_key(v);
            pass[qi] = vis && key[qi] > tau[qi];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty(slot));
        int* wcnt = ms + MS_WCNT + (tcount & 1) * (kMaxQs * 4);
        uint32_t bal[QS_MAX];
#pragma unroll
        for (int qi = 0; qi < QS_MAX; ++qi) {
          bal[qi] = 0u;
          if (qi < qs) {
            bal[qi] = __ballot_sync(0xffffffffu, pass[qi]);
            if (lane == 0) wcnt[qi * 4 + wq] = __popc(bal[qi]);
          }
        }
        if (named_bar_or(bar_id, 128, !ok || *abort_flag)) {
          aborted = true;
          break;
        }
#pragma unroll
        for (int qi = 0; qi < QS_MAX; ++qi) {
          if (qi < qs) {
            const int c0 = wcnt[qi * 4 + 0], c1 = wcnt[qi * 4 + 1], c2 = wcnt[qi * 4 + 2],
                      c3 = wcnt[qi * 4 + 3];
            const int before = (wq > 0 ? c0 : 0) + (wq > 1 ? c1 : 0) + (wq > 2 ? c2 : 0);
            if (pass[qi]) {
              const int pos = count[qi] + before + __popc(bal[qi] & lt);
              ckey_base[qi * C + pos] = key[qi];
              cidx_base[qi * C + pos] = (uint16_t)s_idx;
            }
            count[qi] += c0 + c1 + c2 + c3;
          }
        }
#pragma unroll
        for (int qi = 0; qi < QS_MAX; ++qi) {
          if (qi < qs && count[qi] + kTileKeys > C) {
            named_bar_sync(bar_id, 128);   // appends visible to the whole warpgroup
            tau[qi] = wg_select<kMaxCand / 128>(ckey_base + qi * C, cidx_base + qi * C, count[qi],
                                               keep, wq, lane, hist, ms, bar_id);
            count[qi] = keep;
          }
        }
        ++tcount;
      }
      if (aborted) break;
      named_bar_sync(bar_id, 128);
      // finalize: exactly min(keep, visible) entries per query, ascending index
#pragma unroll
      for (int qi = 0; qi < QS_MAX; ++qi) {
        if (qi < qs && count[qi] > keep) {
          wg_select<kMaxCand / 128>(ckey_base + qi * C, cidx_base + qi * C, count[qi], keep, wq,
                                    lane, hist, ms, bar_id);
          count[qi] = keep;
        }
      }
#pragma unroll
      for (int qi = 0; qi < QS_MAX; ++qi) {
        const int tq = qbase + qi;
        if (qi >= qs || tq >= m.L) continue;
        const size_t orow = (size_t)(a + tq) * W;
        const int n = count[qi];
        const uint32_t* ck = ckey_base + qi * C;
        const uint16_t* ci = cidx_base + qi * C;
        if (p.pool > 1) {
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
            const bool v = e < n;
            p.out_idx[orow + e] = v ? (int)ci[e] : -1;
            if (p.out_score) p.out_score[orow + e] = v ? key_to_float(ck[e]) : -__int_as_float(0x7f800000);
          }
          if (tid == 0 && p.out_len) p.out_len[a + tq] = n;
        }
      }
      named_bar_sync(bar_id, 128);
    }
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
cudaError_t launch_build_worklist(const int32_t* cu, int num_seqs, int total_tokens, int max_seqlen,
                                  int tq, int pool, int2* items, int* doc_prefix, int* hdr,
                                  int max_items, cudaStream_t stream) {
  build_worklist_kernel<<<1, kWLThreads, 0, stream>>>(cu, num_seqs, total_tokens, max_seqlen, tq,
                                                      pool, items, doc_prefix, hdr, max_items);
  return cudaGetLastError();
}

template <int PREC, int H>
static cudaError_t launch_score_t(const ScoreParams& p, int grid, cudaStream_t stream) {
  auto kern = score_topk_kernel<PREC, H>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.plan.total);
  if (e != cudaSuccess) return e;
  kern<<<grid, kScoreThreads, p.plan.total, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_score_topk(const ScoreParams& p, int grid, cudaStream_t stream) {
  const int H = p.plan.n_heads;
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

}  // namespace dsa
