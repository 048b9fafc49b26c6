// Launch plan and shared-memory layout of the fused score + top-k kernel,
// shared by the host planner (api.cu) and the kernel (score_topk.cu).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace dsa {

enum { PREC_BF16 = 0, PREC_MXFP8 = 1, PREC_FP8 = 2 };   // FP8: one scale per row

constexpr int kEpiWarp0 = 2;         // warp 0: TMA producer, warp 1: MMA + TMEM owner, then epilogue
constexpr int kMaxEpiWGs = 4;
constexpr int kTileKeys = 128;       // keys per tcgen05 tile (UMMA M)
constexpr int kChunkBytes = 128;     // bytes of one K-major row per smem chunk (128B swizzle)
constexpr int kStageBytes = kTileKeys * kChunkBytes;   // 16 KiB
constexpr int kSfRawWords = 132;     // 128 scale words + up to 3 words of misalignment + 1
constexpr int kSfRawBytes = 640;     // kSfRawWords*4 = 528, padded to a 128-byte multiple
constexpr int kSfTxBytes = 512;      // 32 rows x 16 bytes: the tcgen05.cp source layout
constexpr int kMaxSmem = 232448;     // 227 KiB opt-in per block on sm_100/sm_103
constexpr int kBatch = 4;            // key tiles scored between two appends
constexpr int kMaxQpw = 4;           // queries per epilogue warpgroup (at most)
constexpr int kMiscInts = 192 + 2 * kBatch * kMaxQpw * 4;   // per-warpgroup scratch ints
constexpr int kMaxStages = 6;
constexpr int kMaxCand = 8192;      // candidate entries per query (at most)
constexpr int kMaxKeep = 4096;      // entries (KPool: pools) kept per query (at most)
constexpr int kSfaCol = 384;         // MXFP8: key scales, 2 x 4 TMEM columns (alternating per tile)
constexpr int kSfbCol = 392;         // MXFP8: query scales, up to 2 atoms x 4 columns

// Per precision: the accumulator of one key tile is ncols <= max_ncols columns
// of TMEM, double buffered (BF16: 2 x 256; MXFP8: 2 x 192 + 16 scale columns),
// and one epilogue warpgroup serves each group of qpw queries.
__host__ __device__ constexpr int max_ncols(int prec) { return prec == PREC_BF16 ? 256 : 192; }
__host__ __device__ constexpr int epi_wgs(int prec) { return prec == PREC_BF16 ? 4 : 3; }
__host__ __device__ constexpr int score_threads(int prec) { return 64 + 128 * epi_wgs(prec); }
// Batches between two abort / shrink votes.  Voting every fourth batch saves
// block-wide barriers but needs room for four batches after a shrink:
// only the 8-bit 64-head plans have candidate buffers large enough for that.
__host__ __device__ constexpr int vote_every(int prec, int n_heads) {
  return prec != PREC_BF16 && n_heads == 64 ? 4 : 1;
}
__host__ __device__ constexpr int qpw_max(int prec, int n_heads) {
  return max_ncols(prec) / (epi_wgs(prec) * n_heads) < kMaxQpw ? max_ncols(prec) / (epi_wgs(prec) * n_heads)
                                                                : kMaxQpw;
}

// Sizes of one launch of the fused kernel (decided on the host).
struct ScorePlan {
  int prec, head_dim, n_heads;
  int ewgs;      // epilogue warpgroups
  int qpw;       // queries per epilogue warpgroup
  int nq;        // queries per work item (ewgs * qpw)
  int ncols;     // nq * n_heads: UMMA N, TMEM columns of one accumulator slot
  int cand;      // candidate-buffer capacity per query (multiple of 128)
  int keep;      // entries kept per query (index_topk, or index_topk / pool size)
  int nst;       // K-tile smem stages
  int chunks;    // 128-byte chunks per operand row: head_dim*elem/128
  int qchunk;    // bytes of one q-operand chunk: ncols rows x 128 bytes (TMA box of the q map)
  int sfb_atoms; // MXFP8, FP8: 128-row groups of query scales (ceil(ncols / 128))
  // byte offsets into dynamic shared memory (base 1024-aligned)
  int q_off, k_off, sfa_raw_off, sfa_tx_off, sfb_raw_off, sfb_tx_off;
  int cand_key_off, cand_idx_off, w_off, hist_off, misc_off, bar_off, total;
};

struct ScoreParams {
  CUtensorMap tm_q;    // q operand [T*H, D]   (box 128 rows x 128 bytes, 128B swizzle)
  CUtensorMap tm_k;    // key operand [rows, D] (same box)
  CUtensorMap tm_qs;   // q scales as u32 words [T*H]   (box 132 words)
  CUtensorMap tm_ks;   // key scales as u32 words [rows] (box 132 words)
  ScorePlan plan;
  const void* w;
  const int32_t* cu_seqlens;
  const int32_t* cu_keys;   // first key row of each document: cu_seqlens_k, or cu_pools in pool mode
  const int32_t* cu_seqlens_k;   // keys per document when they outnumber its queries, else null
  int32_t* out_idx;
  float* out_score;
  int32_t* out_len;
  int64_t out_rows;         // rows of the outputs (query tokens)
  const int2* items;        // device work list
  int* hdr;                 // [0] status, [1] item count
  const int* tile_base;     // first key tile of each document in ksf_tiles
  const uint32_t* ksf_tiles;   // MXFP8, FP8: key scales laid out per key tile for tcgen05.cp (512 B each)
  const uint8_t* q_scale_vec;  // FP8: one UE8M0 byte per q row [T*H]
  int64_t k_rows;              // rows of the key operand
  unsigned long long timeout_ns;
  float sm_scale;
  int w_bf16;
  int pool;                 // 1 = plain keys, else tokens per (pooled or compressed) key
  int expand;               // 1: expand each selected pool to its tokens (KPool); 0: report key indices
  int tail;                 // append the query's incomplete pool (pool mode)
  int out_width;
  int fault_inject;         // test hook: 1 = the first K stage is never loaded
};

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// K-tile stages the planner keeps before it grows the candidate buffers: two
// key tiles in flight behind the one being multiplied (a BF16 tile at
// head_dim 128 is two 128-byte chunks, so two stages).
inline int min_stages(int prec, int chunks) { return prec == PREC_BF16 ? 2 * chunks : 4; }

// Lays out shared memory for (qpw, cand, nst); returns the total bytes.
inline int layout_score_plan(ScorePlan* s, int nst) {
  const bool sf = s->prec == PREC_MXFP8;
  const bool f8 = s->prec == PREC_FP8;   // key scales per stage; one tile of unit query scales
  int off = 0;
  s->q_off = off;
  off += s->chunks * s->qchunk;
  s->k_off = off;
  s->nst = nst;
  off += nst * kStageBytes;
  s->sfa_raw_off = off;   // unused: key scales arrive already laid out for tcgen05.cp
  s->sfa_tx_off = off;
  off += sf || f8 ? nst * kSfTxBytes : 0;
  s->sfb_raw_off = off;
  off += sf ? 2 * kSfRawBytes : 0;
  s->sfb_tx_off = off;
  off += sf ? 2 * kSfTxBytes : (f8 ? kSfTxBytes : 0);
  s->cand_key_off = off;
  off += s->nq * s->cand * 4;
  s->cand_idx_off = off;
  off += s->nq * s->cand * 2;
  off = round_up(off, 16);
  s->w_off = off;
  off += s->nq * s->n_heads * 4;
  s->hist_off = off;
  off += s->ewgs * 256 * 4;
  s->misc_off = off;
  off += s->ewgs * kMiscInts * 4;
  off = round_up(off, 8);
  s->bar_off = off;
  off += 512;
  s->total = off + 1024;   // slack for aligning the dynamic smem base to 1024
  return s->total;
}

// Host-side planner: returns false when no configuration fits.  Shared memory
// goes first to min_stages() K stages, then to the candidate buffers (fewer
// shrinks; at most 4 * keep, and kMaxCand, entries per query), then to more
// stages.
inline bool make_score_plan(int prec, int head_dim, int n_heads, int keep, ScorePlan* p) {
  ScorePlan s{};
  s.prec = prec;
  s.head_dim = head_dim;
  s.n_heads = n_heads;
  s.keep = keep;
  s.ewgs = epi_wgs(prec);
  const int elem = prec == PREC_BF16 ? 2 : 1;
  const bool sf = prec == PREC_MXFP8;
  s.chunks = head_dim * elem / kChunkBytes;
  // every batch up to the next vote fits after a shrink
  const int cand_min = round_up(keep + (kBatch * vote_every(prec, n_heads) + 2) * kTileKeys, 128);
  if (cand_min > kMaxCand) return false;
  const int cand_cap = 4 * keep > cand_min ? (4 * keep < kMaxCand ? round_up(4 * keep, 128) : kMaxCand) : cand_min;
  for (int qpw = qpw_max(prec, n_heads); qpw >= 1; qpw /= 2) {
    s.qpw = qpw;
    s.nq = s.ewgs * qpw;
    s.ncols = s.nq * n_heads;
    if (s.ncols < 16 || s.ncols % 16 != 0 || s.ncols > max_ncols(prec)) return false;
    s.qchunk = s.ncols * kChunkBytes;   // multiple of 1024: keeps the swizzle atoms aligned
    s.sfb_atoms = sf || prec == PREC_FP8 ? (s.ncols + 127) / 128 : 0;
    for (int nmin = min_stages(prec, s.chunks); nmin >= 2; --nmin) {
      // the largest buffer that fits beside nmin stages
      s.cand = 0;
      const int base = layout_score_plan(&s, nmin);
      int cand = (kMaxSmem - base) / (s.nq * 6) / 128 * 128;
      if (cand > cand_cap) cand = cand_cap;
      for (; cand >= cand_min; cand -= 128) {
        s.cand = cand;
        if (layout_score_plan(&s, nmin) <= kMaxSmem) break;
      }
      if (cand < cand_min) continue;
      int nst = nmin;   // spare bytes become more stages
      while (nst < kMaxStages && layout_score_plan(&s, nst + 1) <= kMaxSmem) ++nst;
      layout_score_plan(&s, nst);
      *p = s;
      return true;
    }
  }
  return false;
}

}  // namespace dsa
