"""The LM-head path (spec_verify_lmhead) against the oracle: logits H W^T in
float64 from the same bf16 hidden states and weights, then the oracle's
verification of those logits.

With small-integer inputs every partial sum of a logit is exact in float32, so
the tensor-core product equals the float64 one and the step is held to the
bars of the logits path: greedy bit-exact, sampled requests equal unless the
oracle flags a near tie (at most one such difference).  With random inputs the
float32 accumulation differs from the float64 product by rounding: the row
statistics agree within 1e-5 relative, and greedy argmaxes are bit-exact
wherever the top-two gap exceeds the accumulation bound."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import NEAR_TIE, REL_TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import speculative_decoding_verification_69_gb300 as m
    m.load_library()
    return m


def _oracle_logits(inp, b_idx=None):
    """float64 logits of the target and draft rows (requests b_idx, or all)."""
    ht, hd = inp["hidden_target"], inp["hidden_draft"]
    if b_idx is not None:
        ht, hd = ht[b_idx], hd[b_idx]
    w = workloads.bf16_bits(inp["w"])
    return oracle.lm_logits(workloads.bf16_bits(ht), w), oracle.lm_logits(workloads.bf16_bits(hd), w)


def _run(sv, inp, debug=False):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = sv.verify_lmhead(inp["hidden_target"], inp["hidden_draft"], inp["w"], inp["w"],
                         inp["tokens"], inp["verify_len"], inp["temperature"], inp["seed"],
                         dev_status=st, debug=debug)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in r] + [int(st.item())]


def _compare(out, acc, r, T, idx=None):
    """(greedy mismatches, sampled mismatches, unflagged sampled mismatches)."""
    idx = range(len(acc)) if idx is None else idx
    ng = ns = nu = 0
    for i, b in enumerate(idx):
        same = acc[b] == r["accept_len"][i] and np.array_equal(out[b], r["out_tokens"][i])
        if same:
            continue
        if oracle.is_greedy(T[b]):
            ng += 1
        else:
            ns += 1
            if min(r["accept_margin"][i], r["cdf_margin"][i]) >= NEAR_TIE:
                nu += 1
    return ng, ns, nu


@pytest.mark.parametrize("B,K,V,d,T,n_greedy", [
    (8, 4, 1000, 64, 1.0, 2),       # one m tile, a ragged vocabulary tile
    (16, 8, 4096, 128, 0.8, 4),     # 144 rows: two m tiles, the second ragged
    (64, 8, 3000, 128, 1.0, 16),    # 576 rows: 4.5 m tiles
    (6, 3, 2052, 192, 1.3, 0),      # 2052 = 8 tiles of 256 + 4
    (3, 2, 32000, 256, 1.0, 1),     # many vocabulary tiles per row
    (40, 16, 1024, 64, 0.7, 8),     # K = 16
    (1, 1, 512, 64, 1.0, 0),        # one request, one draft: 2 + 1 rows in two segments
    (4, 4, 2048, 8192, 1.0, 1),     # a large hidden size: 128 k blocks per tile
])
def test_lmhead_exact_products_against_oracle(sv, B, K, V, d, T, n_greedy):
    inp = workloads.make_lmhead_inputs(B, K, V, d, seed=B * 100 + K + V + d, T=T,
                                       n_greedy=n_greedy, exact=True)
    out, acc, st = _run(sv, inp)
    assert st == 0
    zt, zd = _oracle_logits(inp)
    Tn = inp["temperature"].cpu().numpy()
    r = oracle.verify(zt, zd, inp["tokens"].cpu().numpy(), inp["verify_len"].cpu().numpy(), Tn,
                      inp["seed"])
    ng, ns, nu = _compare(out, acc, r, Tn)
    assert ng == 0 and nu == 0 and ns <= 1, (ng, ns, nu)
    if B >= 4:
        assert acc.max() >= 1  # some drafts are accepted


def test_lmhead_ragged_lengths_and_bad_tokens(sv):
    """Verify lengths below K, out of range (clamped) and draft tokens outside
    [0, V) (the length is cut): the status bits and outputs of spec_verify's
    rule, against the oracle."""
    B, K, V, d = 12, 6, 1500, 64
    inp = workloads.make_lmhead_inputs(B, K, V, d, seed=77, exact=True, n_greedy=3)
    vl = torch.tensor([6, 0, 3, 9, -2, 6, 1, 5, 6, 2, 4, 6], dtype=torch.int32, device="cuda")
    tok = inp["tokens"].clone()
    tok[5, 2] = V + 7
    tok[8, 0] = -1
    inp.update(verify_len=vl, tokens=tok.contiguous())
    out, acc, st = _run(sv, inp)
    assert st & sv.DEV_BAD_LEN and st & sv.DEV_BAD_TOKEN
    zt, zd = _oracle_logits(inp)
    Tn = inp["temperature"].cpu().numpy()
    r = oracle.verify(zt, zd, tok.cpu().numpy(), vl.cpu().numpy(), Tn, inp["seed"])
    ng, ns, nu = _compare(out, acc, r, Tn)
    assert ng == 0 and nu == 0 and ns <= 1


def _accumulation_bound(h, w):
    """Per logit, a bound on |fp32 tensor-core sum - exact sum|: at most
    d/16 + 16 roundings of a float32 sum, each below 2^-24 of the sum of
    |h_j w_vj| (h [M, d], w [V, d] as float64)."""
    d = h.shape[1]
    return (d / 16 + 16) * 2.0 ** -24 * (np.abs(h) @ np.abs(w).T)


@pytest.mark.parametrize("B,K,V,d", [(12, 4, 8192, 512), (4, 8, 32000, 1024)])
def test_lmhead_random_products_row_statistics(sv, B, K, V, d):
    """Random normal inputs: row max, log-sum and p(x), q(x) within 1e-5
    relative of the oracle's (on float64 logits); greedy requests bit-exact
    wherever every row's top-two gap exceeds the accumulation bound; sampled
    outputs within the valid range."""
    inp = workloads.make_lmhead_inputs(B, K, V, d, seed=B + V + d, T=1.0, n_greedy=B // 2)
    out, acc, rs, pr, st = _run(sv, inp, debug=True)
    assert st == 0
    zt, zd = _oracle_logits(inp)
    Tn = inp["temperature"].cpu().numpy()
    tok = inp["tokens"].cpu().numpy()
    worst = 0.0
    for b in range(B):
        if oracle.is_greedy(Tn[b]):
            continue
        for k in range(K + 1):
            rows = [(k, zt[b, k])] + ([(K + 1 + k, zd[b, k])] if k < K else [])
            for slot, row in rows:
                x = int(tok[b, k]) if k < K else -1
                m, ls, px = oracle.row_intermediates(row, Tn[b], x)
                gm, gls = rs[b, slot]
                worst = max(worst, abs(gm - m) / max(abs(m), 1e-30), abs(gls - ls) / max(abs(ls), 1.0))
                if k < K:
                    gp = pr[b, k, 0 if slot <= K else 1]
                    worst = max(worst, abs(gp - px) / max(abs(px), 1e-30))
    assert worst < REL_TOL, worst
    # greedy requests whose rows all have a clear top-two gap: bit-exact
    w = workloads.bf16_bits(inp["w"]).astype(np.uint32) << 16
    w = w.view(np.float32).astype(np.float64)
    checked = 0
    for b in range(B):
        if not oracle.is_greedy(Tn[b]):
            continue
        h = (workloads.bf16_bits(inp["hidden_target"][b]).astype(np.uint32) << 16)
        h = h.view(np.float32).astype(np.float64)
        bound = _accumulation_bound(h, w)
        clear = True
        for k in range(K + 1):
            o = np.argsort(-zt[b, k], kind="stable")
            clear &= zt[b, k, o[0]] - zt[b, k, o[1]] > bound[k, o[0]] + bound[k, o[1]]
        if not clear:
            continue
        ot = oracle.verify(zt[b:b + 1], zd[b:b + 1], tok, None, Tn, inp["seed"], b0=b, b1=b + 1,
                           broadcast_rows=True)
        assert acc[b] == ot["accept_len"][0] and np.array_equal(out[b], ot["out_tokens"][0]), b
        checked += 1
    assert checked >= 1
    for b in range(B):
        assert 0 <= acc[b] <= K and np.array_equal(out[b, :acc[b]], tok[b, :acc[b]])
        assert 0 <= out[b, acc[b]] < V and (out[b, acc[b] + 1:] == -1).all()


def test_lmhead_bench_shape_one_request(sv):
    """The benchmark's shapes (B=32, K=8, V=151936, d=4096) with exact
    products: the whole batch through the GPU path, the last request (its rows
    in the last m tile) against the oracle, invariants on all."""
    B, K, V, d = 32, 8, 151936, 4096
    inp = workloads.make_lmhead_inputs(B, K, V, d, seed=4242, T=1.0, exact=True, n_greedy=8)
    out, acc, st = _run(sv, inp)
    assert st == 0
    b = B - 1
    zt, zd = _oracle_logits(inp, slice(b, b + 1))
    Tn = inp["temperature"].cpu().numpy()
    tok = inp["tokens"].cpu().numpy()
    # request b with its own Philox index: the oracle reads the one request's
    # logits for request b of the full token / temperature arrays
    r = oracle.verify(zt, zd, tok, None, Tn, inp["seed"], b0=b, b1=b + 1, broadcast_rows=True)
    same = acc[b] == r["accept_len"][0] and np.array_equal(out[b], r["out_tokens"][0])
    flagged = min(r["accept_margin"][0], r["cdf_margin"][0]) < NEAR_TIE
    assert same or flagged
    for i in range(B):
        assert 0 <= acc[i] <= K and np.array_equal(out[i, :acc[i]], tok[i, :acc[i]])
        assert 0 <= out[i, acc[i]] < V and (out[i, acc[i] + 1:] == -1).all()


@pytest.mark.parametrize("B,K,V,d", [(16, 8, 4096, 128), (40, 4, 2052, 64)])
def test_lmhead_separate_draft_head(sv, B, K, V, d):
    """A drafter with a head of its own (w_draft a different matrix): the
    target and draft rows take separate products and separate recomputes;
    exact products against the oracle with each head."""
    inp = workloads.make_lmhead_inputs(B, K, V, d, seed=B * 3 + V, T=0.9, n_greedy=B // 4,
                                       exact=True)
    g = torch.Generator(device="cuda").manual_seed(B + d)
    s = inp["w"].float().abs().max().item()  # the target head's step (2^-s)
    wd = (torch.randint(-1, 2, (V, d), generator=g, device="cuda").float() * s).to(torch.bfloat16)
    wd = torch.where(torch.rand((V, d), generator=g, device="cuda") < 0.8, inp["w"], wd).contiguous()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, acc = sv.verify_lmhead(inp["hidden_target"], inp["hidden_draft"], inp["w"], wd,
                                inp["tokens"], inp["verify_len"], inp["temperature"], inp["seed"],
                                dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    zt = oracle.lm_logits(workloads.bf16_bits(inp["hidden_target"]), workloads.bf16_bits(inp["w"]))
    zd = oracle.lm_logits(workloads.bf16_bits(inp["hidden_draft"]), workloads.bf16_bits(wd))
    Tn = inp["temperature"].cpu().numpy()
    r = oracle.verify(zt, zd, inp["tokens"].cpu().numpy(), inp["verify_len"].cpu().numpy(), Tn,
                      inp["seed"])
    ng, ns, nu = _compare(out.cpu().numpy(), acc.cpu().numpy(), r, Tn)
    assert ng == 0 and nu == 0 and ns <= 1, (ng, ns, nu)


def test_lmhead_bounded_waits_run_out(sv):
    """The product's failure path without a fault: under the diagnostic switch
    the producer copies nothing, every CTA's bounded wait runs out (1 ms),
    SPEC_DEV_TIMEOUT is reported, the TMEM is freed and the call returns; the
    next call, with the switch off, is correct."""
    B, K, V, d = 8, 4, 1000, 64
    inp = workloads.make_lmhead_inputs(B, K, V, d, seed=515, exact=True, n_greedy=2)
    ws = torch.zeros(sv.lmhead_workspace_bytes(B, K, V, d), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.force_wait_timeout(True)
    try:
        sv.verify_lmhead(inp["hidden_target"], inp["hidden_draft"], inp["w"], inp["w"],
                         inp["tokens"], inp["verify_len"], inp["temperature"], inp["seed"],
                         dev_status=st, workspace=ws)
        torch.cuda.synchronize()
    finally:
        sv.force_wait_timeout(False)
    assert int(st.item()) & sv.DEV_TIMEOUT
    out, acc, st2 = _run(sv, inp)
    assert st2 == 0
    zt, zd = _oracle_logits(inp)
    Tn = inp["temperature"].cpu().numpy()
    r = oracle.verify(zt, zd, inp["tokens"].cpu().numpy(), inp["verify_len"].cpu().numpy(), Tn,
                      inp["seed"])
    ng, ns, nu = _compare(out, acc, r, Tn)
    assert ng == 0 and nu == 0 and ns <= 1


@pytest.mark.parametrize("i", range(24))
def test_lmhead_random_exact_cases(sv, i):
    """Seeded random shapes with exact products: B in [1, 48], K up to 16, V a
    multiple of 4 from 4 to 20,000, d a multiple of 64 up to 512, mixed
    temperatures and greedy shares; the logits path's bars against the
    oracle."""
    rng = np.random.default_rng(33_000 + i)
    B = int(rng.integers(1, 49))
    K = int(rng.choice([1, 2, 4, 8, 16]))
    V = int(rng.choice([4, 100, 512, 1000, 2052, 4100, 20000]))
    d = int(rng.choice([64, 128, 192, 320, 512]))
    T = float(rng.choice([0.5, 1.0, 1.5]))
    inp = workloads.make_lmhead_inputs(B, K, V, d, seed=40_000 + i, T=T,
                                       n_greedy=int(rng.integers(0, B + 1)), exact=True)
    out, acc, st = _run(sv, inp)
    assert st == 0
    zt, zd = _oracle_logits(inp)
    Tn = inp["temperature"].cpu().numpy()
    r = oracle.verify(zt, zd, inp["tokens"].cpu().numpy(), inp["verify_len"].cpu().numpy(), Tn,
                      inp["seed"])
    ng, ns, nu = _compare(out, acc, r, Tn)
    assert ng == 0 and nu == 0 and ns <= 1, (i, ng, ns, nu)
