"""Seeded random candidate trees through spec_verify_tree /
spec_verify_tree_distinct, every request against the oracle: B in [1, 40],
N in [1, 64] nodes, V from 2 to 70,000 (rows a multiple of 16 bytes or not),
bf16 and fp32, logit scales and draft noise varied, chains mixed with bushy
trees, a share of greedy requests, siblings independent or distinct.  A
request may differ from the oracle only inside the tree walk's near-tie
window, and at most one per batch."""
import numpy as np
import pytest
import torch

import workloads
from test_gpu_tree import _compare_tree

pytestmark = pytest.mark.gpu

N_CASES = 60


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import speculative_decoding_verification_69_gb300 as m
    m.load_library()
    return m


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_tree_case(sv, i):
    rng = np.random.default_rng(77_000 + i)
    B = int(rng.integers(1, 41))
    N = int(rng.choice([1, 2, 3, 5, 9, 16, 33, 64]))
    V = int(rng.choice([2, 40, 1000, 1001, 4096, 4100, 32000, 70000]))
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    distinct = bool(rng.random() < 0.5) and V >= N
    inp = workloads.make_tree_inputs(B, N, V, dtype, seed=6_000 + i,
                                     T=float(rng.choice([0.5, 0.8, 1.0, 1.4])),
                                     sigma=float(rng.choice([1.0, 2.5, 4.0])),
                                     noise=float(rng.choice([0.2, 0.7, 1.5])),
                                     chain_prob=float(rng.choice([0.0, 0.5, 1.0])),
                                     n_greedy=int(rng.integers(0, B // 3 + 1)), distinct=distinct)
    out, nodes, acc, st = _compare_tree(sv, inp, max_flag_frac=1.0, distinct=distinct)
    assert st == 0
    assert ((acc >= 0) & (acc <= N - 1)).all()
