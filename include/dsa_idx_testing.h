/*
 * dsa_idx_testing.h — test-only entry points of the DSA lightning-indexer
 * library (dsa_idx.h).  They are exported by the same shared library so the
 * test suite can reach them, and are not part of the supported interface:
 * nothing on the hot path calls them, and a caller of dsa_idx.h never needs
 * them.
 */
#ifndef DSA_IDX_TESTING_H_
#define DSA_IDX_TESTING_H_

#include "dsa_idx.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One tcgen05 tile of the scoring contraction, written raw:
 * acc[r, c] = sum_d K[r, d] * Q[c, d] for r < 128 key rows starting at
 * k_row0 and c < n_cols query rows starting at q_row0 (block-scaled for
 * MXFP8), fp32 [128, n_cols] to `acc_out`.  It checks the tensor-core operand
 * layout (TMA boxes, 128-byte swizzle, descriptors, scale layout) in
 * isolation.  Same pointer and error conventions as dsa_idx.h. */
dsa_status_t dsa_idx_debug_mma_tile(
    const void* q, const uint8_t* q_scale, int64_t q_rows, int64_t q_row0,
    const void* k, const uint8_t* k_scale, int64_t k_rows, int64_t k_row0,
    int head_dim, int n_cols, dsa_precision_t prec, float* acc_out,
    void* ws, size_t ws_bytes, dsa_stream_t stream);

/* Bound of every device-side wait, in nanoseconds, for the following calls of
 * this process (default 2 s).  The failure-detection tests shorten it so a
 * withheld load ends with DSA_ERR_TIMEOUT quickly.  Host-side setting only. */
void dsa_idx_test_set_timeout_ns(unsigned long long ns);

/* Fault injection on the host side of the next calls: 0 = off, 1 = the fused
 * kernel's producer never issues its first key-stage load (the consumers'
 * bounded waits then run out and report DSA_ERR_TIMEOUT; nothing faults). */
void dsa_idx_test_set_fault_inject(int mode);

#ifdef __cplusplus
}
#endif

#endif /* DSA_IDX_TESTING_H_ */
