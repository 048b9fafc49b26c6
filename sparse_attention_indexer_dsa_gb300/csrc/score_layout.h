// Launch plan and shared-memory layout of the fused score + top-k kernel,
// shared by the host planner (api.cu) and the kernel (score_topk.cu).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace dsa {

enum { PREC_BF16 = 0, PREC_MXFP8 = 1 };

constexpr int kEpiWGs = 4;           // epilogue warpgroups
constexpr int kScoreThreads = 64 + 128 * kEpiWGs;   // warp 0: TMA, warp 1: MMA + TMEM, then epilogue
constexpr int kEpiWarp0 = 2;
constexpr int kG = 2;                // query sub-blocks (UMMA B operands) per work item
constexpr int kTileKeys = 128;       // keys per tcgen05 tile (UMMA M)
constexpr int kChunkBytes = 128;     // bytes of one K-major row per smem chunk (128B swizzle)
constexpr int kStageBytes = kTileKeys * kChunkBytes;   // 16 KiB
constexpr int kSfRawWords = 132;     // 128 scale words + up to 3 words of misalignment + 1
constexpr int kSfRawBytes = 640;     // kSfRawWords*4 = 528, padded to a 128-byte multiple
constexpr int kSfTxBytes = 512;      // 32 rows x 16 bytes: the tcgen05.cp source layout
constexpr int kMaxSmem = 232448;     // 227 KiB opt-in per block on sm_100/sm_103
constexpr int kMiscInts = 320;       // per-warpgroup scratch ints
constexpr int kBatch = 4;            // key tiles scored between two appends
constexpr int kMaxQpw = 4;           // queries per epilogue warpgroup (at most)
constexpr int kEpiBarAll = 1 + kEpiWGs;   // named barrier of all epilogue warps (1..kEpiWGs: per warpgroup)
constexpr int kMaxStages = 6;
constexpr int kMaxQs = 8;
constexpr int kMaxCand = 4096;

// Sizes of one launch of the fused kernel (decided on the host).
struct ScorePlan {
  int prec, head_dim, n_heads;
  int qs;        // queries per sub-block
  int nsub;      // qs * n_heads: UMMA N of one sub-block
  int cand;      // candidate-buffer capacity per query (multiple of 128)
  int keep;      // entries kept per query (index_topk, or index_topk / pool size)
  int nst;       // K-tile smem stages
  int chunks;    // 128-byte chunks per operand row: head_dim*elem/128
  int tslots;    // TMEM accumulator slots of 128 columns
  int qchunk;    // bytes of one q-operand chunk: nsub rows x 128 bytes (TMA box of the q map)
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
  const int32_t* cu_keys;   // cu_seqlens, or cu_pools in pool mode
  int32_t* out_idx;
  float* out_score;
  int32_t* out_len;
  const int2* items;        // device work list
  int* hdr;                 // [0] status, [1] item count
  unsigned long long timeout_ns;
  float sm_scale;
  int w_bf16;
  int pool;                 // 1 = plain keys
  int tail;                 // append the query's incomplete pool (pool mode)
  int out_width;
  int fault_inject;         // test hook: 1 = the first K stage is never loaded
};

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Host-side planner: returns false when no configuration fits.
inline bool make_score_plan(int prec, int head_dim, int n_heads, int keep, ScorePlan* p) {
  ScorePlan s{};
  s.prec = prec;
  s.head_dim = head_dim;
  s.n_heads = n_heads;
  s.keep = keep;
  const int elem = prec == PREC_BF16 ? 2 : 1;
  s.chunks = head_dim * elem / kChunkBytes;
  s.tslots = prec == PREC_BF16 ? 4 : 3;
  int qs = 128 / n_heads;
  if (qs > kMaxQs) qs = kMaxQs;
  const int cand_min = keep + (kBatch + 2) * kTileKeys;   // a full batch fits after a shrink
  int cand = round_up(keep * 2 > cand_min ? keep * 2 : cand_min, 128);
  if (cand > kMaxCand) cand = round_up(cand_min, 128);
  if (cand > kMaxCand) return false;
  for (;;) {
    if (qs * n_heads < 16 || (qs * kG) % kEpiWGs != 0) return false;
    s.qs = qs;
    s.nsub = qs * n_heads;
    s.cand = cand;
    s.qchunk = s.nsub * kChunkBytes;   // a multiple of 1024 (nsub % 16 == 0): keeps the swizzle atoms aligned
    // fixed part
    int off = 0;
    s.q_off = off;
    off += kG * s.chunks * s.qchunk;
    s.k_off = off;
    // the rest, independent of the stage count
    int rest = 0;
    const int sf = prec == PREC_MXFP8;
    int cand_bytes = kG * qs * cand * 6;
    rest += cand_bytes + kG * qs * n_heads * 4 + kEpiWGs * 256 * 4 + kEpiWGs * kMiscInts * 4 + 512;
    int per_stage = kStageBytes + (sf ? kSfRawBytes + kSfTxBytes : 0);
    int sfb = sf ? kG * (kSfRawBytes + kSfTxBytes) : 0;
    int nst = (kMaxSmem - 1024 - off - rest - sfb) / per_stage;
    if (nst > kMaxStages) nst = kMaxStages;
    if (nst >= 2) {
      s.nst = nst;
      off += nst * kStageBytes;
      s.sfa_raw_off = off;
      off += sf ? nst * kSfRawBytes : 0;
      s.sfa_tx_off = off;
      off += sf ? nst * kSfTxBytes : 0;
      s.sfb_raw_off = off;
      off += sf ? kG * kSfRawBytes : 0;
      s.sfb_tx_off = off;
      off += sf ? kG * kSfTxBytes : 0;
      s.cand_key_off = off;
      off += kG * qs * cand * 4;
      s.cand_idx_off = off;
      off += kG * qs * cand * 2;
      off = round_up(off, 16);
      s.w_off = off;
      off += kG * qs * n_heads * 4;
      s.hist_off = off;
      off += kEpiWGs * 256 * 4;
      s.misc_off = off;
      off += kEpiWGs * kMiscInts * 4;
      off = round_up(off, 8);
      s.bar_off = off;
      off += 512;
      s.total = off + 1024;   // slack for aligning the dynamic smem base to 1024
      *p = s;
      return s.total <= kMaxSmem;
    }
    if (cand > round_up(cand_min, 128)) {
      cand = round_up(cand_min, 128);
      continue;
    }
    if (qs > 2 && (qs / 2) * n_heads >= 16) {   // qs stays even: kG*qs splits over kEpiWGs
      qs /= 2;
      cand = round_up(keep * 2 > cand_min ? keep * 2 : cand_min, 128);
      if (cand > kMaxCand) cand = round_up(cand_min, 128);
      continue;
    }
    return false;
  }
}

}  // namespace dsa
