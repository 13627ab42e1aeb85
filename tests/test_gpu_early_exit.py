"""Early-exit verification (spec_verify_early_exit): positions verified in two
waves, [0, W) then [W, K), with the second wave reading rows only for requests
still open.  Its outputs must be bit-identical to spec_verify's on the same
inputs (which the parity tests pin to the oracle), for every split W; and it
must agree with the oracle directly on the small workload.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import compare, host_inputs, oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import speculative_decoding_verification_69_gb300 as m
    m.load_library()
    return m


def _run(sv, inp, early_exit):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, acc = sv.verify(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                         inp["temperature"], inp["seed"], dev_status=st, early_exit=early_exit)
    torch.cuda.synchronize()
    return out.cpu().numpy(), acc.cpu().numpy(), int(st.item())


def _schedule(sv, inp):
    if "draft_maxprob" in inp:
        inp["verify_len"] = sv.schedule_len(inp["draft_maxprob"], inp["threshold"])
    return inp


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_full_size_identical_to_single_pass(sv, cfg):
    inp = _schedule(sv, workloads.make_inputs(cfg, rep=3))
    K = inp["tokens"].shape[1]
    ref_out, ref_acc, ref_st = _run(sv, inp, 0)
    for W in sorted({1, 2, 4, K - 1, K, K + 3}):
        out, acc, st = _run(sv, inp, W)
        assert np.array_equal(acc, ref_acc), (cfg, W)
        assert np.array_equal(out, ref_out), (cfg, W)
        assert st == ref_st


@pytest.mark.parametrize("greedy", [False, True])
def test_c0_against_oracle(sv, greedy):
    idx = list(range(64))
    inp = workloads.make_inputs(0, rep=5, B=64, greedy=greedy)
    out, acc, _ = _run(sv, inp, 2)
    h = host_inputs(inp)
    orc = oracle_run(h, idx)
    gpu = dict(out_tokens=out, accept_len=acc)
    ng, ns, nu, nsamp, nflag = compare(gpu, orc, h, idx)
    assert ng == 0 and nu == 0, (ng, nu)
    assert ns <= max(1, int(1e-4 * max(nsamp, 1)))


def test_ragged_mixed_invalid_identical(sv):
    """Zero and full verify lengths, greedy and sampled rows, an out-of-range
    draft token and out-of-range lengths: same outputs and status bits."""
    B, K, V = 24, 6, 3000
    g = torch.Generator(device="cuda").manual_seed(12)
    tgt = (torch.randn((B, K + 1, V), generator=g, device="cuda") * 2.0).to(torch.bfloat16)
    drf = (tgt[:, :K].float() + 0.4 * torch.randn((B, K, V), generator=g, device="cuda")).to(torch.bfloat16)
    T = torch.tensor([0.0 if b % 5 == 0 else 0.4 + 0.05 * b for b in range(B)], device="cuda")
    tok = torch.empty((B, K), dtype=torch.int32, device="cuda")
    for b in range(B):
        t = float(T[b])
        if t > 0:
            pr = torch.softmax(drf[b].float() / t, dim=-1)
            tok[b] = torch.multinomial(pr, 1, generator=g).view(K).to(torch.int32)
        else:
            tok[b] = drf[b].float().argmax(dim=-1).to(torch.int32)
    tok[3, 2] = V + 7
    L = torch.tensor([0, 1, 2, 3, 4, 5, 6, 6, 9, -2] + [K] * (B - 10), dtype=torch.int32, device="cuda")
    inp = dict(target=tgt.contiguous(), draft=drf.contiguous(), tokens=tok, temperature=T,
               verify_len=L, seed=99)
    ref = _run(sv, inp, 0)
    for W in (1, 2, 3, 5):
        got = _run(sv, inp, W)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), W
        assert got[2] == ref[2] and got[2] != 0


def test_repeated_calls_reuse_workspace(sv):
    """The per-request wave state lives in the workspace: back-to-back calls
    with different inputs must not see each other's state."""
    a = workloads.make_inputs(1, rep=8, B=16)
    b = workloads.make_inputs(1, rep=9, B=16)
    ra, rb = _run(sv, a, 0), _run(sv, b, 0)
    for _ in range(2):
        assert np.array_equal(_run(sv, a, 3)[0], ra[0])
        assert np.array_equal(_run(sv, b, 3)[0], rb[0])


def test_large_vocabulary_identical(sv):
    """A 600K-element vocabulary (more than 128 statistics items per row, so
    the decision combines each row in blocks, and 293 sampler chunks): the two
    waves give the single pass's outputs bit for bit, greedy and sampled."""
    inp = workloads.make_inputs(1, rep=11, B=8, K=4, V=600_000)
    inp["temperature"][::3] = 0.0  # some greedy requests
    ref = _run(sv, inp, 0)
    for W in (1, 2, 3):
        got = _run(sv, inp, W)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), W
        assert got[2] == ref[2] == 0
