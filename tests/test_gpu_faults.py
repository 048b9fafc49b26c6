"""Failure detection without a GPU fault: a bounded device wait that runs out
(the producer withholds its first key stage through a test hook) must end the
kernel with DSA_ERR_TIMEOUT in the status word, leave the context usable,
and the next call must run clean."""
import numpy as np
import pytest
import torch

import sparse_attention_indexer_dsa_gb300 as dsa
from sparse_attention_indexer_dsa_gb300 import _abi
from sparse_attention_indexer_dsa_gb300 import workloads as W
from tests.gpu_util import bf16_dev, dev, host

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_recovers():
    rng = np.random.default_rng(5)
    lens, H, D, k = [700], 64, 128, 32
    T = sum(lens)
    qb = W.random_bf16_bits(rng, (T * H, D))
    kb = W.random_bf16_bits(rng, (T, D))
    w = (rng.standard_normal((T, H)) * 0.1).astype(np.float32)
    cu = dev(np.array([0, T], np.int32))
    ws = dsa.workspace(T, 1, T, H, D, k)
    lib = _abi.load()
    try:
        lib.dsa_idx_test_set_timeout_ns(50_000_000)        # 50 ms
        lib.dsa_idx_test_set_fault_inject(1)
        dsa.score_topk(bf16_dev(qb), None, bf16_dev(kb), None, dev(w), cu, T, H, k, "bf16", ws=ws)
        assert dsa.read_status(ws) == _abi.DSA_ERR_TIMEOUT
    finally:
        lib.dsa_idx_test_set_fault_inject(0)
        lib.dsa_idx_test_set_timeout_ns(2_000_000_000)
    idx, sc, ln = dsa.score_topk(bf16_dev(qb), None, bf16_dev(kb), None, dev(w), cu, T, H, k, "bf16", ws=ws)
    assert dsa.read_status(ws) == 0
    assert (host(ln) == np.minimum(np.arange(T) + 1, k)).all()
    torch.cuda.synchronize()
