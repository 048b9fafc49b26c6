"""One tcgen05 tile in isolation: the raw fp32 accumulator of the scoring
contraction against a float64 matmul of the same operands (BF16 kind::f16 and
block-scaled MXFP8 kind::mxf8f6f4)."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_indexer_dsa_gb300 as dsa
from sparse_attention_indexer_dsa_gb300 import workloads as W
from tests.gpu_util import bf16_dev, dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("n_cols,q_row0,k_row0", [(128, 0, 0), (32, 48, 131), (64, 200, 7)])
def test_bf16_tile(D, n_cols, q_row0, k_row0):
    rng = np.random.default_rng(100 + D + n_cols)
    qb = W.random_bf16_bits(rng, (300, D))
    kb = W.random_bf16_bits(rng, (400, D))
    acc, ws = dsa.debug_mma_tile(bf16_dev(qb), None, q_row0, bf16_dev(kb), None, k_row0, n_cols, "bf16")
    assert dsa.read_status(ws) == 0
    q = O.bf16_bits_to_float(qb)[q_row0:q_row0 + n_cols]
    k = O.bf16_bits_to_float(kb)[k_row0:k_row0 + 128]
    ref = k @ q.T
    got = host(acc)
    scale = np.abs(k) @ np.abs(q).T
    err = np.abs(got - ref)
    assert np.all(err <= 3e-5 * scale + 1e-30), (err / (scale + 1e-30)).max()


@pytest.mark.parametrize("n_cols,q_row0,k_row0", [(128, 0, 0), (128, 64, 3), (32, 4, 130), (64, 128, 257)])
def test_mxfp8_tile(n_cols, q_row0, k_row0):
    rng = np.random.default_rng(7 + n_cols + k_row0)
    qc = W.random_e4m3_codes(rng, (400, 128))
    kc = W.random_e4m3_codes(rng, (500, 128))
    qs = W.random_ue8m0(rng, (400, 4))
    ks = W.random_ue8m0(rng, (500, 4))
    acc, ws = dsa.debug_mma_tile(dev(qc), dev(qs), q_row0, dev(kc), dev(ks), k_row0, n_cols, "mxfp8")
    assert dsa.read_status(ws) == 0
    q = O.dequantize_mxfp8(qc, qs)[q_row0:q_row0 + n_cols]
    k = O.dequantize_mxfp8(kc, ks)[k_row0:k_row0 + 128]
    ref = k @ q.T
    got = host(acc)
    scale = (np.abs(k) @ np.abs(q).T)
    err = np.abs(got - ref)
    assert np.all(err <= 1e-3 * scale + 1e-30), (err / (scale + 1e-30)).max()
