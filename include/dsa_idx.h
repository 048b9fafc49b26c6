/*
 * dsa_idx.h — C ABI of the GB300 (sm_103a) DSA lightning-indexer library.
 *
 * The method (DeepSeek Sparse Attention "lightning indexer" forward):
 *   per query token t and every causally visible key s of the same document
 *     I[t,s] = sm_scale * sum_j w[t,j] * ReLU(q[t,j,:] . k[s,:])
 *   over the indexer heads j (one key head shared by all query heads), then the
 *   index_topk keys with the largest I are selected per query.
 * Sources (the public Megatron-LM pull-request pages this library follows):
 *   [P1] PR #8403 "cuDNN DSA indexer precision options": "What does this PR do?"
 *        (dsa_indexer_rope_fp32, dsa_indexer_scoring_precision), "Motivation"
 *        (BF16 materialised between key LayerNorm and RoPE), review finding 1
 *        (_assert_supported_indexer_scoring(use_relu)), finding 2 (BF16 rounding
 *        of FP32 carriers at the scoring boundary; worked example q=k=1.001),
 *        finding 3 (_indexer_forward(q, k, w, ratio, sm_scale, precision) with
 *        q (1,128,32,128) against k (1,128,1,128)).
 *   [P2] PR #5992 "[DeepSeek-V4] Add compact BF16 and MXFP8 DSA indexer
 *        support": "Key changes" (MXFP8 via BF16->MXFP8 quantisation, THD
 *        cu_seqlens, caller-owned CUDA-graph-safe workspaces, deterministic
 *        Top-K tie breaking), review "THD MXFP8 scale prefixes".
 *   [P3] PR #7522 "KPool (pooled-key) DSA indexer support": "Changes"
 *        (dsa_indexer_kpool, always_select_tail, THD restart, NoPE).
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" are caller-owned CUDA device pointers, 16-byte
 *     aligned, row-major and contiguous.  The library never allocates, frees
 *     or synchronises on them; every call is enqueued on the caller's stream
 *     and returns as soon as the launches are queued (capturable in a CUDA
 *     graph).  Sizes are passed by value so no device->host read is needed
 *     ([P2] "Key changes": caller-owned workspaces, sizing done eagerly).
 *   - Sequences are packed back to back (THD).  cu_seqlens is a device int32
 *     array [num_seqs+1] with cu_seqlens[0]=0, non-decreasing, and
 *     cu_seqlens[num_seqs]=total_tokens; queries and keys share it (T=S per
 *     document, self attention).  A batch of equal-length sequences (BSHD) is
 *     the special case of equal lengths.
 *   - Causality: key s is visible to query t iff both lie in the same
 *     document and s_local <= t_local (diagonal included).
 *   - Indices written by the library are local to the document (0..len-1).
 *   - Host-side argument errors return a code before anything is launched;
 *     dsa_idx_last_error() gives the message.  Errors the device detects
 *     (inconsistent cu_seqlens, a bounded wait that ran out) are recorded in
 *     the status word at the head of the workspace; read them with
 *     dsa_idx_read_status().
 *   - MXFP8 tensors: payload bytes are OCP FP8 E4M3 codes, row-major like the
 *     source; scales are UE8M0 bytes (value 2^(byte-127)), one per 32
 *     consecutive elements along head_dim, stored row-major [rows, D/32].  The
 *     scale layout does not depend on cu_seqlens (unlike the per-sequence
 *     padded layout in [P2], whose prefixes can go stale under graph replay).
 */
#ifndef DSA_IDX_H_
#define DSA_IDX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st* dsa_stream_t;

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1, /* bad pointer, size, or inconsistent cu_seqlens */
  DSA_ERR_UNSUPPORTED = 2, /* shape / head count / device not supported */
  DSA_ERR_CUDA = 3,        /* a CUDA runtime call failed */
  DSA_ERR_WORKSPACE = 4,   /* workspace missing or too small */
  DSA_ERR_TIMEOUT = 5,     /* a device-side bounded wait gave up */
  DSA_ERR_BOUNDS = 6       /* checked build (DSA_CHECKED) only: a device-side
                              bounds check on a candidate-buffer or output
                              write failed; the write was skipped (a library
                              defect, never an input error) */
} dsa_status_t;

typedef enum { DSA_DTYPE_F32 = 0, DSA_DTYPE_BF16 = 1 } dsa_dtype_t;

/* Scoring precision.  DSA_PREC_FP8: E4M3 with one UE8M0 scale per vector
 * (the SM90 path's per-vector FP8 scoring, [P1] "What does this PR do?"):
 * q_scale [rows of q] and k_scale [rows of k] hold one byte per row. */
typedef enum { DSA_PREC_BF16 = 0, DSA_PREC_MXFP8 = 1, DSA_PREC_FP8 = 2 } dsa_precision_t;

/* UE8M0 block-exponent rule of the MXFP8 quantiser.
 * DSA_MX_SCALE_NOSAT (default): the smallest e with amax <= 448*2^e, so no
 *   element saturates (the BF16->MXFP8 conversion of [P2] "Key changes").
 * DSA_MX_SCALE_FLOOR: e = floor(log2(amax)) - 8, payload saturates at +-448. */
typedef enum { DSA_MX_SCALE_NOSAT = 0, DSA_MX_SCALE_FLOOR = 1 } dsa_mx_scale_rule_t;

/* dsa_idx_score_topk flags. */
#define DSA_FLAG_DETERMINISTIC 0x1   /* [P2] deterministic Top-K tie break; always honoured */
/* Rows in ranking order, score descending then index ascending, instead of
 * ascending index: the order of the repeated-varlen-ends regression rows in
 * [P1]'s review ("Preservation and acceptance"). */
#define DSA_FLAG_SORT_BY_SCORE 0x2
#define DSA_FLAG_KPOOL_TAIL 0x4      /* [P3] always_select_tail: append the query's incomplete pool */
/* [P2] compressed keys: kpool_size is the indexer's `ratio` (2..64); k holds
 * caller-computed compressed keys, cu_pools their per-document prefix; each
 * query keeps index_topk compressed keys, indices not expanded to tokens. */
#define DSA_FLAG_COMPRESSED_KEYS 0x8

/* Checked build.  Compiled with -DDSA_CHECKED (libdsa_idx_checked.so, built by
 * build_lib.build_checked()), the library adds, at some cost in speed:
 *   - a pass over the inputs of every score + top-k call before the fused
 *     kernel: a NaN or Inf in q, k (BF16 operands), w, an E4M3 NaN code or a
 *     UE8M0 NaN scale (0xFF) records DSA_ERR_INVALID_ARG in the status word
 *     and the call writes no output (reading of the pages' silence on
 *     non-finite inputs: undefined in the normal build);
 *   - bounds checks on every candidate-buffer and output write of the fused
 *     kernel, recording DSA_ERR_BOUNDS and skipping the write.
 * The entry points and their arguments are the same. */

/* Library version (major*10000 + minor*100 + patch). */
int dsa_idx_version(void);

/* Message of the last host-side error in this thread ("" if none). */
const char* dsa_idx_last_error(void);

/* Human-readable name of a status code. */
const char* dsa_idx_status_string(dsa_status_t s);

/* Bytes of caller-owned device workspace dsa_idx_score_topk needs for these
 * sizes (status word, device-built work list).  Pure host function.
 * Returns 0 for invalid sizes. */
size_t dsa_idx_workspace_size(int total_tokens, int num_seqs, int max_seqlen,
                              int n_heads, int head_dim, int index_topk,
                              int kpool_size, dsa_precision_t prec);

/* Width (entries per query row) of the index / score outputs of
 * dsa_idx_score_topk: index_topk, or index_topk + kpool_size - 1 in pool mode
 * with DSA_FLAG_KPOOL_TAIL. */
int dsa_idx_output_width(int index_topk, int kpool_size, int flags);

/* Key LayerNorm -> RoPE -> quantise, fused ([P1] "What does this PR do?" and
 * "Motivation": key LayerNorm then RoPE; rope_fp32 keeps the chain in FP32,
 * otherwise BF16 is materialised after the LayerNorm and after RoPE; [P1]
 * finding 2: BF16 scoring rounds FP32 carriers to BF16; [P2] "Key changes":
 * MXFP8 scoring operands).  Queries get RoPE only.  [P3] "Changes": rope_dim=0
 * is the NoPE indexer.
 *   q       device [total_tokens, n_heads, head_dim], in_dtype
 *   k       device [total_tokens, head_dim], in_dtype
 *   ln_gamma, ln_beta  device fp32 [head_dim], or both NULL = no key LayerNorm
 *   ln_eps  LayerNorm epsilon (biased variance)
 *   rope_dim  rotary dims (first rope_dim of head_dim; 0 = NoPE; multiple of 8)
 *   rope_base  theta_i = rope_base^(-2i/rope_dim); positions restart at 0 in
 *             every document
 *   rope_interleaved  0: rotate-half pairs (i, i+rope_dim/2); 1: pairs (2i, 2i+1)
 *   out_prec BF16: q_out/k_out are bf16; MXFP8: e4m3 bytes + UE8M0 scales
 *           per 32 elements; FP8: e4m3 bytes + one UE8M0 scale per row
 *   q_out   device [total_tokens*n_heads, head_dim] (bf16 or u8)
 *   q_scale_out device u8 [total_tokens*n_heads, head_dim/32] (MXFP8) or
 *           [total_tokens*n_heads] (FP8), else NULL
 *   k_out, k_scale_out  same for the keys ([total_tokens, ...])
 * Supported: head_dim in {64,128} (MXFP8 and FP8: 128), n_heads in {1..64}.
 * Non-finite inputs give unspecified outputs (no status is recorded: the
 * checked build scans the scoring call's operands instead). */
dsa_status_t dsa_idx_preprocess(
    const void* q, const void* k, dsa_dtype_t in_dtype,
    const float* ln_gamma, const float* ln_beta, float ln_eps,
    const int32_t* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
    int n_heads, int head_dim, int rope_dim, float rope_base,
    int rope_interleaved, int rope_fp32, dsa_precision_t out_prec,
    dsa_mx_scale_rule_t scale_rule,
    void* q_out, uint8_t* q_scale_out, void* k_out, uint8_t* k_scale_out,
    dsa_stream_t stream);

/* Stand-alone BF16/FP32 -> MXFP8 quantisation ([P2] "Key changes": BF16 to
 * MXFP8 with UE8M0 scales per 32 elements).
 *   x        device [rows, cols] in_dtype
 *   x_e4m3   device u8 [rows, cols]
 *   x_ue8m0  device u8 [rows, cols/32]
 * cols must be a multiple of 32 (64 or 128 for the scoring kernel).
 * Non-finite elements give unspecified codes (as in dsa_idx_preprocess). */
dsa_status_t dsa_idx_quantize_mxfp8(const void* x, dsa_dtype_t in_dtype,
                                    int64_t rows, int cols,
                                    dsa_mx_scale_rule_t scale_rule,
                                    uint8_t* x_e4m3, uint8_t* x_ue8m0,
                                    dsa_stream_t stream);

/* Stand-alone BF16/FP32 -> FP8 with one UE8M0 scale per row (the per-vector
 * FP8 scoring of [P1] "What does this PR do?"); the row exponent follows the
 * same rule as an MXFP8 block (scale_rule).
 *   x        device [rows, 128] in_dtype, 16-byte aligned
 *   x_e4m3   device u8 [rows, 128]
 *   x_ue8m0  device u8 [rows]
 * cols must be 128 (DSA_ERR_UNSUPPORTED otherwise).  Non-finite elements give
 * unspecified codes. */
dsa_status_t dsa_idx_quantize_fp8_rows(const void* x, dsa_dtype_t in_dtype,
                                       int64_t rows, int cols,
                                       dsa_mx_scale_rule_t scale_rule,
                                       uint8_t* x_e4m3, uint8_t* x_ue8m0,
                                       dsa_stream_t stream);

/* KPool key compression ([P3] "Changes", dsa_indexer_kpool > 1): in every
 * document, each complete group of pool_size consecutive keys becomes
 *   kbar_p = sum_i softmax_i(gate[p*P+i] + slot_bias[i]) * k[p*P+i]
 * (softmax over the P slots, computed in FP32), stored as bf16.  Pooling
 * restarts at document boundaries; an incomplete last group is not pooled.
 *   k          device [total_tokens, head_dim] k_dtype
 *   gate_bf16  device bf16 bits [total_tokens]
 *   slot_bias  device fp32 [pool_size]
 *   k_pooled   device bf16 [total_tokens / pool_size, head_dim]
 *              (document d's pools are rows cu_pools[d] .. cu_pools[d+1]-1)
 *   cu_pools   device int32 [num_seqs+1], written by this call
 * Supported: pool_size in {2,4,8}, head_dim in {64,128}. */
dsa_status_t dsa_idx_kpool_compress(
    const void* k, dsa_dtype_t k_dtype, const uint16_t* gate_bf16,
    const float* slot_bias, const int32_t* cu_seqlens, int num_seqs,
    int total_tokens, int head_dim, int pool_size, uint16_t* k_pooled,
    int32_t* cu_pools, dsa_stream_t stream);

/* Fused score + top-k: q.k^T on tcgen05 tensor cores, ReLU, head-weighted
 * sum, causal/document mask and a streaming per-query top-k that keeps the
 * T x S score matrix on chip.  ([P1] findings 1-3, [P2] "Key changes",
 * [P3] "Changes" for pool mode.)
 *   q        device [total_tokens*n_heads, head_dim]: bf16 (BF16) or e4m3 (MXFP8)
 *   q_scale  device u8 [total_tokens*n_heads, head_dim/32] (MXFP8) or
 *            [total_tokens*n_heads] (FP8), else NULL
 *   k        device [total_tokens, head_dim]; in pool mode the pooled keys
 *            [total_tokens/kpool_size, head_dim] from dsa_idx_kpool_compress
 *   k_scale  device u8 [rows of k, head_dim/32] (MXFP8) or [rows of k] (FP8),
 *            else NULL
 *   w        device [total_tokens, n_heads], w_dtype (FP32 or BF16)
 *   sm_scale scalar multiplier of the score
 *   index_topk  keys selected per query; in pool mode a multiple of
 *               kpool_size, and index_topk / kpool_size pools are kept
 *   prec     BF16 (kind::f16), MXFP8 (block-scaled kind::mxf8f6f4) or FP8
 *            (the same block-scaled MMA with each key row's one scale
 *            repeated over its four 32-element blocks; the query rows'
 *            scales are folded exactly into the head weights, as powers of
 *            two)
 *   flags    DSA_FLAG_* bits
 *   kpool_size  1 = plain keys; >1 = pool mode (cu_pools required): KPool
 *               pools of that size (2, 4 or 8), or with
 *               DSA_FLAG_COMPRESSED_KEYS the compression ratio (2..64) of
 *               caller-provided compressed keys.  Either way key c of a
 *               document covers its tokens c*kpool_size .. +kpool_size-1
 *               and is visible once complete; k has room for
 *               total_tokens / kpool_size rows and document d's keys are
 *               rows cu_pools[d] .. cu_pools[d+1]-1 (at least
 *               floor(L_d / kpool_size) of them; more are never visible)
 *   topk_idx    device int32 [total_tokens, W] (W = dsa_idx_output_width):
 *               selected local indices in ascending order, then -1
 *               padding; with DSA_FLAG_SORT_BY_SCORE in ranking order
 *               (score desc, index asc) instead, by a second kernel over
 *               the finished rows (topk_score is then required: NULL
 *               returns DSA_ERR_INVALID_ARG).  KPool mode: the expanded
 *               tokens of the selected pools (pools in the row order above,
 *               each pool's tokens ascending), then the tail tokens.
 *               Compressed keys: the selected compressed-key indices
 *               (W = index_topk).
 *   topk_score  device fp32 [total_tokens, W] or NULL: the score of each
 *               entry (pooled score for pool tokens, +INF for tail tokens,
 *               -INF for padding)
 *   topk_len    device int32 [total_tokens] or NULL: valid entries per row
 *   ws, ws_bytes  device workspace of dsa_idx_workspace_size() bytes
 * Ties are broken towards the lower index; -0 and +0 compare equal.
 * Supported: head_dim 128 (BF16 also 64), n_heads in {4,8,16,32,64},
 * 1 <= index_topk <= 4096 (KPool: at most 4096 pools, index_topk <= 4096 *
 * kpool_size; MXFP8 or FP8 with 4 heads: <= 1664, the candidate buffers of
 * its 12 queries per block must fit in shared memory), max_seqlen <= 65536.
 * Other shapes return DSA_ERR_UNSUPPORTED. */
dsa_status_t dsa_idx_score_topk(
    const void* q, const uint8_t* q_scale, const void* k, const uint8_t* k_scale,
    const void* w, dsa_dtype_t w_dtype, float sm_scale,
    const int32_t* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
    int n_heads, int head_dim, int index_topk, dsa_precision_t prec, int flags,
    int kpool_size, const int32_t* cu_pools,
    int32_t* topk_idx, float* topk_score, int32_t* topk_len,
    void* ws, size_t ws_bytes, dsa_stream_t stream);

/* Fused score + top-k for documents whose queries are the last tokens of a
 * longer key sequence ([P1] review finding 2: "global causal offsets", e.g.
 * a query chunk scored against its document's keys so far).  Document d has
 * T_d = cu_seqlens_q[d+1]-cu_seqlens_q[d] queries and S_d =
 * cu_seqlens_k[d+1]-cu_seqlens_k[d] >= T_d keys; its query i sits at position
 * S_d - T_d + i and sees keys 0 .. S_d - T_d + i of the document.
 *   q, q_scale, w, topk_idx, topk_score, topk_len  as in dsa_idx_score_topk,
 *               with total_q rows (tokens)
 *   k, k_scale  [total_k, head_dim] (and [total_k, head_dim/32])
 *   cu_seqlens_q, cu_seqlens_k  device int32 [num_seqs+1] each
 *   max_seqlen_q, max_seqlen_k  upper bounds of T_d and S_d (S_d <= 65536)
 *   ws, ws_bytes  dsa_idx_workspace_size() with total_tokens =
 *               max(total_q, total_k)
 * Indices are local to the document's keys.  Pool mode is not available
 * here.  T_d > S_d (or inconsistent prefixes) is caught on the device:
 * DSA_ERR_INVALID_ARG in the status word, no output written.  Equal key and
 * query lengths give exactly dsa_idx_score_topk's result. */
dsa_status_t dsa_idx_score_topk_kv(
    const void* q, const uint8_t* q_scale, const void* k, const uint8_t* k_scale,
    const void* w, dsa_dtype_t w_dtype, float sm_scale,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int num_seqs,
    int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
    int n_heads, int head_dim, int index_topk, dsa_precision_t prec, int flags,
    int32_t* topk_idx, float* topk_score, int32_t* topk_len,
    void* ws, size_t ws_bytes, dsa_stream_t stream);

/* Allocation-free dsa_idx_score_topk, for callers that cannot provide device
 * scratch memory: code that runs after a no-allocation-past-start-up point
 * (latency-critical serving loops, real-time pipelines), hosts whose device
 * memory belongs to an allocator they may not grow, and plugin-style
 * integrations that only receive input and output tensors.  The pages describe
 * no counterpart; it exists for those callers.
 * Same arguments and results as dsa_idx_score_topk without ws/ws_bytes.  The
 * scratch lives in a fixed 4 MiB device array inside the library, which every
 * GPU that loads the library holds until the process exits; sizes whose
 * dsa_idx_workspace_size exceeds 4 MiB are rejected with DSA_ERR_WORKSPACE
 * before anything is launched: about total_tokens + num_seqs above 524 000 for
 * BF16 scoring, and total_tokens above about 349 000 for MXFP8 and FP8 (their
 * per-tile key scales also live in the scratch; each document costs about 43
 * tokens' worth more).  Comparing dsa_idx_workspace_size with 4194304 gives
 * the exact answer.  It calls no cudaMalloc/cudaFree.  The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current and keeps it once found (a failed lookup is retried by the
 * next call); make that first call before capturing any stream.  The address
 * is that of the current CUDA context: a device reset while the library is
 * loaded is not supported.  All calls share the one array, so calls whose GPU
 * work overlaps (other streams, or unordered calls from several host threads)
 * race on it.  dsa_idx_score_topk_noalloc_status reads the device status word
 * the last call left in the array. */
dsa_status_t dsa_idx_score_topk_noalloc(
    const void* q, const uint8_t* q_scale, const void* k, const uint8_t* k_scale,
    const void* w, dsa_dtype_t w_dtype, float sm_scale,
    const int32_t* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
    int n_heads, int head_dim, int index_topk, dsa_precision_t prec, int flags,
    int kpool_size, const int32_t* cu_pools,
    int32_t* topk_idx, float* topk_score, int32_t* topk_len, dsa_stream_t stream);

/* Companion of dsa_idx_score_topk_noalloc (no counterpart in the pages):
 * synchronise `stream` and return in *out the device status word the last
 * dsa_idx_score_topk_noalloc call on the current device left in the library's
 * scratch array: DSA_ERR_TIMEOUT when a bounded device wait ran out (the
 * rows of that call are then incomplete), DSA_ERR_INVALID_ARG when the device
 * found cu_seqlens inconsistent, DSA_OK otherwise.  Eager helper, like
 * dsa_idx_read_status; do not call it while capturing a graph. */
dsa_status_t dsa_idx_score_topk_noalloc_status(dsa_stream_t stream, dsa_status_t* out);

/* Synchronise `stream` and return the device status word recorded in `ws` by
 * the last dsa_idx_score_topk call on it (DSA_OK if none).  Eager helper; do
 * not call it while capturing a graph. */
dsa_status_t dsa_idx_read_status(const void* ws, dsa_stream_t stream,
                                 dsa_status_t* out);

/* Test-only entry points (a raw tensor-core tile, the timeout and the
 * fault-injection hooks) are declared in dsa_idx_testing.h. */

#ifdef __cplusplus
}
#endif

#endif /* DSA_IDX_H_ */
