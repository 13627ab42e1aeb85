"""Failure path of the bounded device waits, without a GPU fault: with the
diagnostic switch on, every warp of the bulk-copy kernels waits on a barrier
nothing completes; the wait runs out and the warp gives up as on a real
timeout.  The call must report SPEC_DEV_TIMEOUT in the status word (the warps
still let their copies land before exiting), and the next call must be correct
again (the context stays usable)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import compare, gpu_run, host_inputs, oracle_run

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_recoverable():
    import speculative_decoding_verification_69_gb300 as sv
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    sv.load_library()
    inp = workloads.make_inputs(1, rep=17, B=16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        sv.force_wait_timeout(True)
        out, acc = sv.verify(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                             inp["temperature"], inp["seed"], dev_status=st)
        torch.cuda.synchronize()
    finally:
        sv.force_wait_timeout(False)
    assert int(st.item()) & sv.DEV_TIMEOUT
    acc = acc.cpu().numpy()
    assert ((acc >= 0) & (acc <= 8)).all()          # undefined but in range
    idx = list(range(16))
    gpu = gpu_run(inp)
    assert gpu["status"] == 0
    h = host_inputs(inp)
    ng, ns, nu, nsamp, nflag = compare(gpu, oracle_run(h, idx), h, idx)
    assert ng == 0 and nu == 0


@pytest.mark.parametrize("cfg,ee", [(1, 0), (4, 0), (2, 4)])
def test_poisoned_workspace_and_outputs(cfg, ee):
    """Every workspace byte set to 0xFF (NaN floats, -1 ints) and the outputs
    pre-filled with garbage: the results must equal a clean run's, and every
    output element must be written (no read of an unwritten workspace byte,
    no output slot left over)."""
    import speculative_decoding_verification_69_gb300 as sv
    inp = workloads.make_inputs(cfg, rep=23, B=64)
    B, K = inp["tokens"].shape
    clean = sv.Verifier()
    o1, a1 = clean(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                   inp["temperature"], inp["seed"], early_exit=ee)
    v = sv.Verifier()
    ws, n = v.workspace(B, K, inp["target"].shape[2], inp["target"].dtype, inp["target"].device)
    ws.fill_(0xFF)
    o2 = torch.full((B, K + 1), 123456, dtype=torch.int32, device="cuda")
    a2 = torch.full((B,), -99, dtype=torch.int32, device="cuda")
    v(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"], inp["temperature"],
      inp["seed"], out_tokens=o2, accept_len=a2, early_exit=ee)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(a1, a2)
    assert (o2 != 123456).all() and (a2 >= 0).all()


def test_tree_walk_wait_timeout_is_reported():
    """The sampled tree walk's staging wait: with the diagnostic switch on, each
    warp first gives up on a barrier nothing completes and reports
    SPEC_DEV_TIMEOUT, then waits for its copies, so the outputs equal a clean
    run's; the next call reports nothing."""
    import speculative_decoding_verification_69_gb300 as sv
    inp = workloads.make_tree_inputs(32, 16, 151936, torch.bfloat16, seed=41, T=1.0)
    args = (inp["target"], inp["draft"], inp["parent"], inp["tokens"], inp["temperature"],
            inp["seed"])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        sv.force_wait_timeout(True)
        o1, n1, a1 = sv.verify_tree(*args, dev_status=st)
        torch.cuda.synchronize()
    finally:
        sv.force_wait_timeout(False)
    assert int(st.item()) & sv.DEV_TIMEOUT
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    o2, n2, a2 = sv.verify_tree(*args, dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert torch.equal(o1, o2) and torch.equal(n1, n2) and torch.equal(a1, a2)


def test_bad_tokens_at_the_wave_boundary():
    """Draft tokens outside [0, V) at positions W - 1, W and W + 1 of a
    two-wave call (the cut is applied by the decision kernel, after the rows
    were listed from the clamped lengths): a poisoned workspace gives the
    outputs and status of a clean single-pass call, which match the oracle."""
    import speculative_decoding_verification_69_gb300 as sv
    inp = workloads.make_inputs(2, rep=29, B=48)
    B, K = inp["tokens"].shape
    V = inp["target"].shape[2]
    W = 4
    tok = inp["tokens"].clone()
    for b in range(0, B, 4):
        tok[b, W - 1 + (b // 4) % 3] = V + b  # W - 1, W or W + 1
    inp["tokens"] = tok.contiguous()
    st1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1, a1 = sv.Verifier()(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                           inp["temperature"], inp["seed"], dev_status=st1)
    v = sv.Verifier()
    ws, n = v.workspace(B, K, V, inp["target"].dtype, inp["target"].device)
    ws.fill_(0xFF)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    o2, a2 = v(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"], inp["temperature"],
               inp["seed"], early_exit=W, dev_status=st2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(a1, a2)
    assert int(st1.item()) & sv.DEV_BAD_TOKEN and int(st2.item()) & sv.DEV_BAD_TOKEN
    idx = list(range(B))
    h = host_inputs(inp)
    gpu = dict(out_tokens=o1.cpu().numpy(), accept_len=a1.cpu().numpy())
    ng, ns, nu, nsamp, nflag = compare(gpu, oracle_run(h, idx), h, idx)
    assert ng == 0 and nu == 0 and ns <= 1
