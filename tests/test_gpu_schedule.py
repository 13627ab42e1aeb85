"""Confidence-scheduled verification on the GPU: the draft confidences
(spec_draft_confidence) against the oracle within 1e-5 relative, and the
load-aware schedule (spec_schedule_budget) bit-exact against the oracle's sort,
including ties, clamped and NaN probabilities and the edge budgets."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import speculative_decoding_verification_69_gb300 as m
    m.load_library()
    return m


@pytest.mark.parametrize("cfg,n", [(3, 24), (4, 24), (0, 1)])
def test_draft_confidence_against_oracle(sv, cfg, n):
    inp = workloads.make_inputs(cfg, rep=2)
    got = sv.draft_confidence(inp["draft"], inp["temperature"]).cpu().numpy()
    ref = oracle.draft_confidence(workloads.to_numpy_logits(inp["draft"][:n]),
                                  inp["temperature"][:n].cpu().numpy())
    assert np.allclose(got[:n], ref, rtol=1e-5, atol=0.0), np.abs(got[:n] / ref - 1).max()
    greedy = np.array([oracle.is_greedy(t) for t in inp["temperature"].cpu().numpy()])
    assert (got[greedy] == 1.0).all()
    assert ((got > 0) & (got <= 1.0 + 1e-6)).all()


def test_draft_confidence_shapes(sv):
    """Odd vocabularies (vector path with bounds), fp32, -inf entries, and a
    vocabulary past 128 statistics items per row (the looping combine)."""
    g = torch.Generator(device="cuda").manual_seed(21)
    for B, K, V, dt in [(3, 2, 1001, torch.bfloat16), (2, 5, 999, torch.float32),
                        (4, 3, 16384 + 8, torch.bfloat16),
                        (2, 2, 600_000, torch.bfloat16)]:  # > 128 statistics items per row
        d = (torch.randn((B, K, V), generator=g, device="cuda") * 3.0).to(dt)
        d[0, 0, ::2] = float("-inf")
        T = torch.tensor([0.7, 1.3, 0.2, 2.0][:B], device="cuda")
        got = sv.draft_confidence(d.contiguous(), T).cpu().numpy()
        ref = oracle.draft_confidence(workloads.to_numpy_logits(d), T.cpu().numpy())
        assert np.allclose(got, ref, rtol=1e-5, atol=0.0), (B, K, V)


def _budget_cases():
    rng = np.random.default_rng(3)
    for B, K in [(1, 1), (7, 5), (256, 16), (4096, 32), (20000, 3)]:
        mp = rng.uniform(0.0, 1.0, size=(B, K)).astype(np.float32)
        mp[rng.random((B, K)) < 0.1] = 1.0          # ties: survival stays put
        mp[rng.random((B, K)) < 0.02] = 0.0
        if B > 1:
            mp[0, 0] = np.nan                        # counts as 0
            mp[1, 0] = 1.5                           # clamped to 1
        n = B * K
        for budget in sorted({0, 1, n // 3, n // 2, n - 1, n, n + 5}):
            yield mp, budget


def test_schedule_budget_bitexact(sv):
    for mp, budget in _budget_cases():
        got = sv.schedule_budget(torch.from_numpy(mp).cuda(), budget).cpu().numpy()
        ref = oracle.schedule_budget(mp, budget)
        assert np.array_equal(got, ref), (mp.shape, budget)
        assert got.sum() == min(max(budget, 0), mp.size)


def test_schedule_budget_equals_threshold_schedule(sv):
    """Budget = positions whose survival reaches the threshold: the GPU's
    budgeted lengths equal the GPU's threshold schedule (c3's draft
    max-probabilities)."""
    inp = workloads.make_inputs(3, rep=1)
    mp = inp["draft_maxprob"]
    L = sv.schedule_len(mp, inp["threshold"])
    got = sv.schedule_budget(mp, int(L.sum().item()))
    assert torch.equal(got, L)


def test_confidence_budget_verify_chain(sv):
    """The whole chain on the device: confidences from the draft logits, a
    budget of 5 positions per request, verification; the lengths follow the
    oracle's schedule of the same confidences."""
    inp = workloads.make_inputs(3, rep=4, B=32)
    conf = sv.draft_confidence(inp["draft"], inp["temperature"])
    B = conf.shape[0]
    vl = sv.schedule_budget(conf, 5 * B)
    assert np.array_equal(vl.cpu().numpy(), oracle.schedule_budget(conf.cpu().numpy(), 5 * B))
    out, acc = sv.verify(inp["target"], inp["draft"], inp["tokens"], vl, inp["temperature"],
                         inp["seed"])
    torch.cuda.synchronize()
    assert (acc.cpu() <= vl.cpu()).all()


def _unfused(sv, inp, threshold=None, budget=None, given=None):
    """The chain as separate calls: confidences (unless given), the schedule,
    then spec_verify."""
    conf = given if given is not None else sv.draft_confidence(inp["draft"], inp["temperature"])
    if threshold is not None:
        vl = sv.schedule_len(conf, threshold)
    else:
        vl = sv.schedule_budget(conf, budget)
    out, acc = sv.verify(inp["target"], inp["draft"], inp["tokens"], vl, inp["temperature"],
                         inp["seed"])
    torch.cuda.synchronize()
    return out.clone(), acc.clone(), vl.clone(), conf.clone()


@pytest.mark.parametrize("cfg,B", [(3, 256), (4, 128), (2, 64), (0, 1)])
@pytest.mark.parametrize("sched", ["threshold", "budget"])
@pytest.mark.parametrize("computed", [True, False])
def test_verify_scheduled_equals_separate_calls(sv, cfg, B, sched, computed):
    """spec_verify_scheduled (one call; with computed confidences the draft rows
    are read once and their statistics reused by the step) gives bit-identical
    tokens, accept lengths, verify lengths and confidences to the separate
    calls on the same inputs."""
    inp = workloads.make_inputs(cfg, rep=5, B=B)
    K = inp["tokens"].shape[1]
    if "draft_maxprob" not in inp:
        inp["draft_maxprob"] = sv.draft_confidence(inp["draft"], inp["temperature"])
    kw = dict(threshold=0.3) if sched == "threshold" else dict(budget=max(1, (K * B) // 3))
    given = None if computed else inp["draft_maxprob"]
    ref_out, ref_acc, ref_vl, ref_conf = _unfused(sv, inp, given=given, **kw)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, acc, vl, conf = sv.verify_scheduled(inp["target"], inp["draft"], inp["tokens"],
                                             inp["temperature"], inp["seed"], draft_maxprob=given,
                                             dev_status=st, **kw)
    torch.cuda.synchronize()
    assert torch.equal(vl, ref_vl)
    assert torch.equal(acc, ref_acc)
    assert torch.equal(out, ref_out)
    if computed:
        assert torch.equal(conf, ref_conf)
    else:
        assert conf is None
    assert int(st.item()) == 0
    if cfg == 3 or sched == "budget" and B > 1:
        assert len(set(vl.cpu().tolist())) > 1  # ragged lengths


def test_verify_scheduled_against_oracle(sv):
    """The fused call's outputs against the oracle, with the oracle's own
    confidences and threshold schedule: lengths bit-exact, tokens equal
    except oracle-flagged near ties (c3 shapes, 64 requests)."""
    from gpu_helpers import compare, host_inputs, oracle_run
    inp = workloads.make_inputs(3, rep=6, B=64)
    out, acc, vl, conf = sv.verify_scheduled(inp["target"], inp["draft"], inp["tokens"],
                                             inp["temperature"], inp["seed"], threshold=0.3)
    torch.cuda.synchronize()
    ref_conf = oracle.draft_confidence(workloads.to_numpy_logits(inp["draft"]),
                                       inp["temperature"].cpu().numpy())
    assert np.allclose(conf.cpu().numpy(), ref_conf, rtol=1e-5, atol=0.0)
    ref_vl = oracle.schedule_len(conf.cpu().numpy(), 0.3)
    assert np.array_equal(vl.cpu().numpy(), ref_vl)
    h = host_inputs(inp, verify_len=vl)
    idx = list(range(64))
    orc = oracle_run(h, idx)
    gpu = dict(out_tokens=out.cpu().numpy(), accept_len=acc.cpu().numpy())
    ng, ns, nu, nsamp, nflag = compare(gpu, orc, h, idx)
    assert ng == 0 and nu == 0 and ns <= 1


def test_bench_c3_scheduled_call_full_size(sv):
    """The c3 step exactly as the benchmark times it (one spec_verify_scheduled
    call, threshold 0.3 on the given confidences): lengths bit-exact with the
    oracle's schedule, every one of the 256 requests against the oracle."""
    from gpu_helpers import compare, host_inputs, oracle_run
    inp = workloads.make_inputs(3)
    out, acc, vl, _ = sv.verify_scheduled(inp["target"], inp["draft"], inp["tokens"],
                                          inp["temperature"], inp["seed"], threshold=0.3,
                                          draft_maxprob=inp["draft_maxprob"])
    torch.cuda.synchronize()
    ref_vl = oracle.schedule_len(inp["draft_maxprob"].cpu().numpy(), 0.3)
    assert np.array_equal(vl.cpu().numpy(), ref_vl)
    B = inp["tokens"].shape[0]
    h = host_inputs(inp, verify_len=vl)
    idx = list(range(B))
    gpu = dict(out_tokens=out.cpu().numpy(), accept_len=acc.cpu().numpy())
    ng, ns, nu, nsamp, nflag = compare(gpu, oracle_run(h, idx), h, idx)
    assert ng == 0 and nu == 0 and ns <= 1, (ng, ns, nu, nsamp, nflag)


def test_bench_chain_call_full_size(sv):
    """The --chain step at c3 (confidences computed from the draft rows, a
    budget of 5 positions per request): confidences within 1e-5 of the
    oracle's, lengths equal to the oracle's budget schedule of the GPU's
    confidences, all 256 requests against the oracle."""
    from gpu_helpers import compare, host_inputs, oracle_run
    inp = workloads.make_inputs(3)
    B = inp["tokens"].shape[0]
    out, acc, vl, conf = sv.verify_scheduled(inp["target"], inp["draft"], inp["tokens"],
                                             inp["temperature"], inp["seed"], budget=5 * B)
    torch.cuda.synchronize()
    ref_conf = oracle.draft_confidence(workloads.to_numpy_logits(inp["draft"][:16]),
                                       inp["temperature"][:16].cpu().numpy())
    assert np.allclose(conf[:16].cpu().numpy(), ref_conf, rtol=1e-5, atol=0.0)
    assert np.array_equal(vl.cpu().numpy(), oracle.schedule_budget(conf.cpu().numpy(), 5 * B))
    h = host_inputs(inp, verify_len=vl)
    idx = list(range(B))
    gpu = dict(out_tokens=out.cpu().numpy(), accept_len=acc.cpu().numpy())
    ng, ns, nu, nsamp, nflag = compare(gpu, oracle_run(h, idx), h, idx)
    assert ng == 0 and nu == 0 and ns <= 1, (ng, ns, nu, nsamp, nflag)


@pytest.mark.parametrize("i", range(30))
def test_verify_scheduled_random_cases(sv, i):
    """Seeded random shapes (the fuzz test's generator) through the fused
    scheduled call, threshold or budget, confidences computed or given:
    bit-identical to the separate calls, and the lengths equal to the
    oracle's schedule of the same confidences."""
    from test_gpu_fuzz import _case
    rng = np.random.default_rng(55_000 + i)
    inp = _case(200 + i)
    B, K = inp["tokens"].shape
    sched = "threshold" if rng.random() < 0.5 else "budget"
    kw = (dict(threshold=float(rng.choice([0.05, 0.3, 0.8]))) if sched == "threshold"
          else dict(budget=int(rng.integers(0, B * K + 3))))
    given = None
    if rng.random() < 0.5:
        given = torch.from_numpy(rng.uniform(0.0, 1.0, size=(B, K)).astype(np.float32)).cuda()
    ref_out, ref_acc, ref_vl, ref_conf = _unfused(sv, inp, given=given, **kw)
    out, acc, vl, conf = sv.verify_scheduled(inp["target"], inp["draft"], inp["tokens"],
                                             inp["temperature"], inp["seed"], draft_maxprob=given,
                                             **kw)
    torch.cuda.synchronize()
    assert torch.equal(vl, ref_vl) and torch.equal(acc, ref_acc) and torch.equal(out, ref_out)
    mp = (given if given is not None else conf).cpu().numpy()
    want = (oracle.schedule_len(mp, kw["threshold"]) if sched == "threshold"
            else oracle.schedule_budget(mp, kw["budget"]))
    assert np.array_equal(vl.cpu().numpy(), want)
