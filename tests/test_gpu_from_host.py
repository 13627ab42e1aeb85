"""spec_verify_from_host: inputs in host memory, only the rows the step reads
copied to the device.  Its outputs must equal spec_verify's on the same
inputs, whatever the device buffers held in the rows it does not copy, and
the bytes it copies must be exactly those rows plus the small arrays."""
import numpy as np
import pytest
import torch

import workloads
from test_gpu_parity import _rand_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import speculative_decoding_verification_69_gb300 as m
    m.load_library()
    return m


def _host(inp):
    h = {k: inp[k].cpu().pin_memory() for k in ("target", "draft", "tokens", "temperature")}
    h["verify_len"] = None if inp["verify_len"] is None else inp["verify_len"].cpu().pin_memory()
    return h


def _expected_bytes(inp):
    """Small arrays, then per request target rows 0..L and, when sampled,
    draft rows 0..L-1 (L clamped to [0, K])."""
    B, K1, V = inp["target"].shape
    K = K1 - 1
    row = V * inp["target"].element_size()
    L = (np.full(B, K) if inp["verify_len"] is None else
         np.clip(inp["verify_len"].cpu().numpy(), 0, K))
    T = inp["temperature"].cpu().numpy()
    sampled = np.isfinite(T) & (T >= np.finfo(np.float32).tiny)
    n = B * K * 4 + B * 4 + (0 if inp["verify_len"] is None else B * 4)
    return n + int(((L + 1) * row).sum()) + int((L * row)[sampled].sum())


def _compare(sv, inp, poison=True):
    st_d = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_d, a_d = sv.verify(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                         inp["temperature"], inp["seed"], dev_status=st_d)
    h = _host(inp)
    hv = sv.HostVerifier()
    st_h = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_h, a_h = hv(h["target"], h["draft"], h["tokens"], h["verify_len"], h["temperature"],
                  inp["seed"], dev_status=st_h)
    torch.cuda.synchronize()
    if poison:  # rows the step does not read keep their contents: make them NaN
        d = hv._buffers(*inp["target"].shape[:1], inp["target"].shape[1] - 1,
                        inp["target"].shape[2], inp["target"].dtype)
        d["target"].fill_(float("nan"))
        d["draft"].fill_(float("nan"))
        st_h.zero_()
        o_h, a_h = hv(h["target"], h["draft"], h["tokens"], h["verify_len"], h["temperature"],
                      inp["seed"], dev_status=st_h)
        torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(a_h, a_d.cpu())
    assert int(st_h.item()) == int(st_d.item())
    assert hv.last_h2d_bytes == _expected_bytes(inp)
    return hv


def test_ragged_mixed_and_invalid(sv):
    B, K, V = 16, 6, 4096
    L = [0, 1, 2, 3, 4, 5, 6, 6, 0, 3, 6, 1, 2, 5, 4, 0]
    T = [0.0 if b % 4 == 0 else 0.5 + 0.1 * b for b in range(B)]
    inp = _rand_inputs(B, K, V, torch.bfloat16, seed=77, T=T, L=L)
    _compare(sv, inp)
    inp["tokens"][3, 1] = V + 5
    inp["tokens"][5, 0] = -2
    inp["verify_len"][7] = 9
    inp["verify_len"][9] = -1
    _compare(sv, inp)


@pytest.mark.parametrize("dtype,V", [(torch.float32, 3000), (torch.bfloat16, 1001)])
def test_no_lengths_and_scalar_rows(sv, dtype, V):
    """verify_len None (every request verifies K), rows whose byte size is not
    a multiple of 16 (the scalar path)."""
    inp = _rand_inputs(6, 4, V, dtype, seed=5 + V, T=[0.0, 0.7, 1.0, 0.0, 1.3, 0.9], L=None)
    _compare(sv, inp)


def test_full_size_workload(sv):
    """B=32, K=8, V=151936 bf16 (every row of every request read)."""
    _compare(sv, workloads.make_inputs(1), poison=False)


@pytest.mark.parametrize("cfg,B,sched", [(3, 64, "threshold"), (3, 64, "budget"), (4, 48, "threshold"),
                                         (0, 1, "budget")])
def test_scheduled_from_host(sv, cfg, B, sched):
    """Lengths from the schedule of given confidences formed on the device and
    read back, then only their rows copied: the outputs, lengths and status
    equal spec_verify_scheduled's, with the unread device rows set to NaN, and
    the bytes copied are the confidences, the listed rows and the small arrays."""
    inp = workloads.make_inputs(cfg, rep=8, B=B)
    K = inp["tokens"].shape[1]
    if "draft_maxprob" not in inp:
        inp["draft_maxprob"] = sv.draft_confidence(inp["draft"], inp["temperature"])
    kw = dict(threshold=0.3) if sched == "threshold" else dict(budget=max(1, (K * B) // 3))
    st_d = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_d, a_d, vl_d, _ = sv.verify_scheduled(inp["target"], inp["draft"], inp["tokens"],
                                            inp["temperature"], inp["seed"],
                                            draft_maxprob=inp["draft_maxprob"], dev_status=st_d,
                                            **kw)
    torch.cuda.synchronize()
    h = _host(inp)
    mp_h = inp["draft_maxprob"].cpu().pin_memory()
    hv = sv.HostVerifier()
    hv.scheduled(h["target"], h["draft"], h["tokens"], h["temperature"], inp["seed"], mp_h, **kw)
    torch.cuda.synchronize()
    d = hv._buffers(B, K, inp["target"].shape[2], inp["target"].dtype)
    d["target"].fill_(float("nan"))
    d["draft"].fill_(float("nan"))
    st_h = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_h, a_h, vl_h = hv.scheduled(h["target"], h["draft"], h["tokens"], h["temperature"],
                                  inp["seed"], mp_h, dev_status=st_h, **kw)
    torch.cuda.synchronize()
    assert torch.equal(vl_h, vl_d.cpu())
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(a_h, a_d.cpu())
    assert int(st_h.item()) == int(st_d.item())
    want = dict(inp, verify_len=vl_d)
    assert hv.last_h2d_bytes == _expected_bytes(want) + B * K * 4
