"""Greedy verification of candidate trees (spec_verify_tree_greedy) against the
oracle, bit-exact: random trees over several sizes and vocabularies, chains
(which must equal the linear greedy verification), and invalid parents."""
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


def _random_trees(B, N, V, dtype, seed):
    """Trees whose tokens often follow the target's argmax (so paths go deep);
    the generator only draws numbers."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    tgt = (torch.randn((B, N, V), generator=g, device="cuda") * 2.0).to(dtype)
    rng = np.random.default_rng(seed)
    parent = np.full((B, N), -1, np.int32)
    tok = np.zeros((B, N), np.int32)
    # the lowest-index argmax (the walk's rule; torch's argmax may pick any of tied maxima,
    # which are common in bf16 rows of a large vocabulary)
    am = np.argmax(tgt.float().cpu().numpy(), axis=-1)  # exact values; the first maximum
    for b in range(B):
        for n in range(1, N):
            p = int(rng.integers(0, n))
            parent[b, n] = p
            tok[b, n] = am[b, p] if rng.random() < 0.5 else int(rng.integers(0, V))
    return tgt.contiguous(), torch.from_numpy(parent).cuda(), torch.from_numpy(tok).cuda()


@pytest.mark.parametrize("B,N,V,dtype", [
    (64, 1, 1000, torch.bfloat16), (64, 2, 1000, torch.bfloat16), (32, 9, 3000, torch.float32),
    (16, 64, 4096 + 8, torch.bfloat16), (8, 33, 1001, torch.bfloat16), (4, 17, 151936, torch.bfloat16),
    (16, 9, 600_000, torch.bfloat16),  # more than 128 statistics items per row
])
def test_random_trees_against_oracle(sv, B, N, V, dtype):
    tgt, parent, tok = _random_trees(B, N, V, dtype, seed=B * 100 + N)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, nodes, acc = sv.verify_tree_greedy(tgt, parent, tok, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    h_t = workloads.to_numpy_logits(tgt)
    p, t = parent.cpu().numpy(), tok.cpu().numpy()
    out, nodes, acc = out.cpu().numpy(), nodes.cpu().numpy(), acc.cpu().numpy()
    deep = 0
    for b in range(B):
        ot, on, a = oracle.verify_tree_greedy(h_t[b], p[b], t[b])
        assert acc[b] == a and np.array_equal(out[b], ot) and np.array_equal(nodes[b], on), b
        deep = max(deep, a)
    assert N < 3 or deep >= 2  # some paths go past the first level


def test_chain_trees_equal_linear_greedy(sv):
    """A chain tree is the linear draft: same outputs as spec_verify at T = 0 on
    c4's shapes (the target rows of a K = 8 call are the chain's node rows)."""
    inp = workloads.make_inputs(4, rep=6, B=64, greedy=True)
    B, K1, V = inp["target"].shape
    out_l, acc_l = sv.verify(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                             inp["temperature"], inp["seed"])
    parent = torch.arange(-1, K1 - 1, dtype=torch.int32, device="cuda").expand(B, K1).contiguous()
    tok = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device="cuda"), inp["tokens"]], dim=1)
    out_t, nodes, acc_t = sv.verify_tree_greedy(inp["target"], parent, tok.contiguous())
    torch.cuda.synchronize()
    assert torch.equal(acc_t, acc_l) and torch.equal(out_t, out_l)


def test_invalid_parents_flagged(sv):
    tgt, parent, tok = _random_trees(4, 6, 500, torch.bfloat16, seed=3)
    parent[1, 3] = 5   # not an earlier node
    parent[2, 4] = -2
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, nodes, acc = sv.verify_tree_greedy(tgt, parent.contiguous(), tok, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & sv.DEV_BAD_TREE
    h_t = workloads.to_numpy_logits(tgt)
    for b in range(4):
        ot, on, a = oracle.verify_tree_greedy(h_t[b], parent[b].cpu().numpy(), tok[b].cpu().numpy())
        assert acc[b].item() == a and np.array_equal(out[b].cpu().numpy(), ot)


# ---------------------------------------------------------------- sampled trees

# Near-tie window of the sampled tree walk: the residual after a rejection is
# formed from float weights whose exp2 carries ~2^-22 relative error, so its
# normalised CDF is known to ~1e-6 / Z; a request may differ from the oracle
# only when the oracle's uniform lies within this distance of a decision
# boundary.
TREE_NEAR_TIE = 1e-5


def _oracle_tree(inp, b0=0, distinct=False):
    """Oracle results for the batch (Philox keys use the request index, the
    first row being request b0).  The draft rows are padded to N with zeros:
    the last node has no children, so the oracle never reads that row."""
    t = workloads.to_numpy_logits(inp["target"])
    B, N, V = t.shape
    d = workloads.to_numpy_logits(inp["draft"]) if N > 1 else np.zeros((B, 0, V), t.dtype)
    d = np.concatenate([d, np.zeros((B, 1, V), d.dtype)], axis=1)
    return oracle.verify_tree(t, d, inp["parent"].cpu().numpy(), inp["tokens"].cpu().numpy(),
                              inp["temperature"].cpu().numpy(), inp["seed"], b0=b0,
                              distinct=distinct)


def _compare_tree(sv, inp, max_flag_frac=0.1, distinct=False):
    """GPU against the oracle: every request equal unless the oracle flags a
    near tie; returns the GPU outputs and the device status."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, nodes, acc = sv.verify_tree(inp["target"], inp["draft"], inp["parent"], inp["tokens"],
                                     inp["temperature"], inp["seed"], dev_status=st,
                                     distinct=distinct)
    torch.cuda.synchronize()
    out, nodes, acc = out.cpu().numpy(), nodes.cpu().numpy(), acc.cpu().numpy()
    r = _oracle_tree(inp, distinct=distinct)
    same = ((acc == r["accept_len"]) & (out == r["out_tokens"]).all(axis=1)
            & (nodes == r["out_nodes"]).all(axis=1))
    flagged = (r["accept_margin"] < TREE_NEAR_TIE) | (r["cdf_margin"] < TREE_NEAR_TIE)
    bad = np.flatnonzero(~same & ~flagged)
    assert bad.size == 0, (bad, acc[bad], r["accept_len"][bad])
    # differences inside the window stay rare: at most one per batch
    assert (~same).sum() <= 1, np.flatnonzero(~same)
    assert flagged.sum() <= max_flag_frac * len(acc) + 1, flagged.sum()
    return out, nodes, acc, int(st.item())


@pytest.mark.parametrize("B,N,V,dtype,T", [
    (48, 1, 1000, torch.bfloat16, 1.0), (48, 2, 1000, torch.bfloat16, 1.0),
    (32, 9, 3000, torch.float32, 0.8), (16, 16, 4096 + 8, torch.bfloat16, 1.3),
    (8, 33, 1001, torch.bfloat16, 1.0), (6, 17, 151936, torch.bfloat16, 1.0),
    (12, 64, 2048, torch.bfloat16, 0.7), (8, 12, 999, torch.float32, 1.0),
    (10, 10, 4100, torch.float32, 1.0),  # staged fp32 rows whose last vector is half past V
    (3, 6, 600_000, torch.bfloat16, 1.0),  # 147 statistics items per row: the looping combine
])
def test_sampled_trees_against_oracle(sv, B, N, V, dtype, T):
    inp = workloads.make_tree_inputs(B, N, V, dtype, seed=B * 1000 + N + V, T=T,
                                     n_greedy=B // 8)
    out, nodes, acc, st = _compare_tree(sv, inp)
    assert st == 0
    if N > 3:
        assert acc.max() >= 2  # some paths go past the first level


@pytest.mark.parametrize("cfg", [1, 2, 4])
def test_sampled_chain_trees_equal_linear(sv, cfg):
    """A chain tree is the linear draft, with the same rows, tokens and Philox
    keys: the tree walk gives spec_verify's outputs, except where the oracle
    flags a near tie (the two paths form the residual differently)."""
    inp = workloads.make_inputs(cfg, rep=9, B=64)
    B, K1, V = inp["target"].shape
    out_l, acc_l = sv.verify(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                             inp["temperature"], inp["seed"])
    parent = torch.arange(-1, K1 - 1, dtype=torch.int32, device="cuda").expand(B, K1).contiguous()
    tok = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device="cuda"), inp["tokens"]], dim=1)
    out_t, nodes, acc_t = sv.verify_tree(inp["target"], inp["draft"], parent, tok.contiguous(),
                                         inp["temperature"], inp["seed"])
    torch.cuda.synchronize()
    diff = torch.nonzero((acc_t != acc_l) | (out_t != out_l).any(dim=1)).flatten().tolist()
    assert len(diff) <= B // 10, diff
    if diff:
        h_t = workloads.to_numpy_logits(inp["target"])
        h_d = workloads.to_numpy_logits(inp["draft"])
        r = oracle.verify(h_t, h_d, inp["tokens"].cpu().numpy(), None,
                          inp["temperature"].cpu().numpy(), inp["seed"])
        for b in diff:
            assert min(r["accept_margin"][b], r["cdf_margin"][b]) < TREE_NEAR_TIE, b
    a = acc_t.cpu().numpy()
    n = nodes.cpu().numpy()
    for b in range(B):
        assert n[b, :a[b]].tolist() == list(range(1, a[b] + 1))


def test_sampled_edge_cases(sv):
    """Invalid tokens (no candidate), invalid parents (no path through them,
    SPEC_DEV_BAD_TREE), a node whose children all carry tokens with zero draft
    mass, and duplicated sibling tokens."""
    inp = workloads.make_tree_inputs(8, 10, 700, torch.bfloat16, seed=77, T=1.0)
    tok, par = inp["tokens"].clone(), inp["parent"].clone()
    tok[0, 1:4] = torch.tensor([-5, 700, 10 ** 6], dtype=torch.int32)
    par[1, 4] = 7          # not an earlier node
    par[2, 5] = -3
    par[3, 1:] = 0         # nine siblings under the root
    tok[3, 1:] = tok[3, 1]  # all carrying the same token
    dr = inp["draft"].clone()
    dr[4, 0, :] = float("-inf")
    dr[4, 0, 5] = 0.0      # the root's draft is a point mass on token 5
    par[4, 1:4] = 0
    tok[4, 1:4] = torch.tensor([5, 6, 5], dtype=torch.int32)
    inp.update(tokens=tok.contiguous(), parent=par.contiguous(), draft=dr.contiguous())
    out, nodes, acc, st = _compare_tree(sv, inp, max_flag_frac=0.3)
    assert st & sv.DEV_BAD_TREE


def test_greedy_requests_take_the_greedy_walk(sv):
    inp = workloads.make_tree_inputs(16, 12, 2000, torch.bfloat16, seed=5, n_greedy=16)
    out, nodes, acc = sv.verify_tree(inp["target"], inp["draft"], inp["parent"], inp["tokens"],
                                     inp["temperature"], inp["seed"])
    out_g, nodes_g, acc_g = sv.verify_tree_greedy(inp["target"], inp["parent"], inp["tokens"])
    torch.cuda.synchronize()
    assert torch.equal(out, out_g) and torch.equal(nodes, nodes_g) and torch.equal(acc, acc_g)


def test_sampled_tree_mismatch_rate(sv):
    """Many small requests: no unflagged mismatch and few flagged ones."""
    inp = workloads.make_tree_inputs(2048, 8, 512, torch.bfloat16, seed=31, T=1.0)
    _compare_tree(sv, inp, max_flag_frac=0.02)


def test_sampled_tree_first_token_law(sv):
    """'Утверждение 1' (kiosknews.app) through the GPU path: with three
    siblings drafted independently from the root's draft row, the first
    emitted token of 200 000 requests (one set of logits, Philox keyed by the
    request) follows the target distribution p of the root row (chi-square);
    a copy whose siblings all carry the draft's most likely token does not."""
    scipy_stats = pytest.importorskip("scipy.stats")
    B, N, V, T = 200000, 4, 12, 1.0
    g = torch.Generator(device="cuda").manual_seed(99)
    trow = torch.randn((N, V), generator=g, device="cuda") * 1.5
    drow = (trow[:N - 1] + torch.randn((N - 1, V), generator=g, device="cuda") * 1.0)
    tgt = trow.expand(B, N, V).contiguous()
    drf = drow.expand(B, N - 1, V).contiguous()
    parent = torch.tensor([-1, 0, 0, 0], dtype=torch.int32, device="cuda").expand(B, N).contiguous()
    q0 = torch.softmax(drow[0] / T, dim=-1)
    draws = torch.multinomial(q0.expand(B, V), N - 1, replacement=True, generator=g)
    tok = torch.cat([torch.zeros((B, 1), dtype=torch.int64, device="cuda"), draws], 1)
    temp = torch.full((B,), T, device="cuda")
    p = oracle.row_softmax(trow[0].cpu().numpy().astype(np.float32), T)[0]
    for tokens, lossless in ((tok, True), (torch.where(tok > 0, torch.full_like(tok, int(q0.argmax())), tok), False)):
        out, nodes, acc = sv.verify_tree(tgt, drf, parent, tokens.to(torch.int32).contiguous(), temp, 1234)
        first = out[:, 0].long().cpu().numpy()
        counts = np.bincount(first, minlength=V)
        _, pval = scipy_stats.chisquare(counts, p * B)
        if lossless:
            assert pval > 1e-4, (pval, counts, p * B)
        else:
            assert pval < 1e-6, pval


@pytest.mark.parametrize("cfg,N,b0,n_check,distinct", [(1, 16, 0, 32, False), (4, 9, 112, 48, False),
                                                       (1, 16, 0, 32, True)])
def test_sampled_trees_at_bench_workloads(sv, cfg, N, b0, n_check, distinct):
    """The sampled-tree workloads the benchmark times (same generator, seed and
    launch configuration: clusters with staged slices at c1, one CTA per
    request at c4 with its quarter of greedy requests), against the oracle on
    requests [b0, b0 + n_check) (c4: greedy requests 112-127, sampled after)."""
    c = workloads.CONFIGS[cfg]
    T = c["T"] if isinstance(c["T"], float) else 1.0
    noise = c["noise"] if isinstance(c["noise"], float) else 0.5
    inp = workloads.make_tree_inputs(c["B"], N, c["V"], c["dtype"], seed=workloads.seed_for(cfg, 0),
                                     T=T, sigma=c["sigma"], noise=noise,
                                     n_greedy=c.get("n_greedy", 0), distinct=distinct)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, nodes, acc = sv.verify_tree(inp["target"], inp["draft"], inp["parent"], inp["tokens"],
                                     inp["temperature"], inp["seed"], dev_status=st,
                                     distinct=distinct)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sl = slice(b0, b0 + n_check)
    sub = {k: (v[sl] if torch.is_tensor(v) else v) for k, v in inp.items()}
    r = _oracle_tree(sub, b0=b0, distinct=distinct)
    out, nodes, acc = out[sl].cpu().numpy(), nodes[sl].cpu().numpy(), acc[sl].cpu().numpy()
    same = ((acc == r["accept_len"]) & (out == r["out_tokens"]).all(axis=1)
            & (nodes == r["out_nodes"]).all(axis=1))
    flagged = (r["accept_margin"] < TREE_NEAR_TIE) | (r["cdf_margin"] < TREE_NEAR_TIE)
    assert not (~same & ~flagged).any(), np.flatnonzero(~same & ~flagged)
    # at V >= 128k the CDF window flags many rows (much of the mass sits in
    # tokens of tiny probability), so the gate counts actual mismatches
    assert (~same).sum() <= 1, np.flatnonzero(~same)


# ---------------------------------------------------------------- distinct siblings

@pytest.mark.parametrize("B,N,V,dtype,T,sigma", [
    (48, 4, 64, torch.bfloat16, 1.0, 3.0), (32, 9, 40, torch.float32, 0.7, 3.0),
    (16, 16, 4096 + 8, torch.bfloat16, 1.3, 2.5), (8, 33, 1001, torch.bfloat16, 1.0, 4.0),
    (6, 17, 151936, torch.bfloat16, 1.0, 2.5), (12, 64, 2048, torch.bfloat16, 0.7, 3.0),
    (10, 10, 4100, torch.float32, 1.0, 3.0),
])
def test_distinct_trees_against_oracle(sv, B, N, V, dtype, T, sigma):
    """Siblings drawn without replacement (top-k style candidates), checked
    with spec_verify_tree_distinct against the oracle's distinct rule; small
    vocabularies with peaked drafts make the rejected siblings' mass large."""
    inp = workloads.make_tree_inputs(B, N, V, dtype, seed=B * 7000 + N + V, T=T, sigma=sigma,
                                     noise=0.7, chain_prob=0.3, n_greedy=B // 8, distinct=True)
    # at V >= 128k the CDF window flags many rows (much of the mass sits in
    # tokens of tiny probability): mismatches are gated, the flags only counted
    out, nodes, acc, st = _compare_tree(sv, inp, distinct=True,
                                        max_flag_frac=0.5 if V > 100000 else 0.1)
    assert st == 0
    if N > 3:
        assert acc.max() >= 2


def test_distinct_rule_differs_from_independent(sv):
    """On distinct draws with peaked drafts the two rules give different walks
    for some requests (the flag changes the arithmetic), and each matches its
    own oracle."""
    inp = workloads.make_tree_inputs(256, 6, 32, torch.float32, seed=404, T=1.0, sigma=3.0,
                                     noise=0.7, chain_prob=0.0, distinct=True)
    a = _compare_tree(sv, inp, distinct=True)
    b = _compare_tree(sv, inp, distinct=False)
    assert (a[2] != b[2]).any() or (a[0] != b[0]).any()


@pytest.mark.parametrize("cfg", [1, 4])
def test_distinct_chains_equal_independent(sv, cfg):
    """One child per node: nothing is ever removed from a draft row, so the
    distinct walk is the independent one, bit for bit."""
    inp = workloads.make_inputs(cfg, rep=9, B=32)
    B, K1, V = inp["target"].shape
    parent = torch.arange(-1, K1 - 1, dtype=torch.int32, device="cuda").expand(B, K1).contiguous()
    tok = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device="cuda"), inp["tokens"]], 1)
    r1 = sv.verify_tree(inp["target"], inp["draft"], parent, tok.contiguous(), inp["temperature"],
                        inp["seed"])
    r2 = sv.verify_tree(inp["target"], inp["draft"], parent, tok.contiguous(), inp["temperature"],
                        inp["seed"], distinct=True)
    torch.cuda.synchronize()
    for x, y in zip(r1, r2):
        assert torch.equal(x, y)


def test_distinct_duplicates_and_point_mass(sv):
    """Inputs no draw without replacement gives: repeated sibling tokens (no
    candidate after the first is rejected) and a point-mass draft (no mass
    left after its token is rejected); GPU and oracle agree."""
    inp = workloads.make_tree_inputs(8, 10, 700, torch.bfloat16, seed=78, T=1.0, distinct=True)
    tok, par = inp["tokens"].clone(), inp["parent"].clone()
    par[3, 1:] = 0
    tok[3, 1:] = tok[3, 1]          # nine siblings, one token
    dr = inp["draft"].clone()
    dr[4, 0, :] = float("-inf")
    dr[4, 0, 5] = 0.0               # the root's draft is a point mass on token 5
    par[4, 1:4] = 0
    tok[4, 1:4] = torch.tensor([5, 6, 7], dtype=torch.int32)
    inp.update(tokens=tok.contiguous(), parent=par.contiguous(), draft=dr.contiguous())
    _compare_tree(sv, inp, max_flag_frac=0.3, distinct=True)


def test_distinct_tree_first_token_law(sv):
    """'Утверждение 1' (kiosknews.app) for top-k style candidates through the
    GPU path: three sibling tokens drawn without replacement from the root's
    draft row, 200 000 requests; the first emitted token follows p
    (chi-square).  The independent-siblings rule on the same draws does not."""
    scipy_stats = pytest.importorskip("scipy.stats")
    B, N, V, T = 200000, 4, 12, 1.0
    g = torch.Generator(device="cuda").manual_seed(99)
    trow = torch.randn((N, V), generator=g, device="cuda") * 1.5
    drow = (trow[:N - 1] + torch.randn((N - 1, V), generator=g, device="cuda") * 1.0)
    tgt = trow.expand(B, N, V).contiguous()
    drf = drow.expand(B, N - 1, V).contiguous()
    parent = torch.tensor([-1, 0, 0, 0], dtype=torch.int32, device="cuda").expand(B, N).contiguous()
    q0 = torch.softmax(drow[0] / T, dim=-1)
    draws = torch.multinomial(q0.expand(B, V), N - 1, replacement=False, generator=g)
    tok = torch.cat([torch.zeros((B, 1), dtype=torch.int64, device="cuda"), draws], 1)
    tok = tok.to(torch.int32).contiguous()
    temp = torch.full((B,), T, device="cuda")
    p = oracle.row_softmax(trow[0].cpu().numpy().astype(np.float32), T)[0]
    for distinct in (True, False):
        out, nodes, acc = sv.verify_tree(tgt, drf, parent, tok, temp, 1234, distinct=distinct)
        counts = np.bincount(out[:, 0].long().cpu().numpy(), minlength=V)
        _, pval = scipy_stats.chisquare(counts, p * B)
        if distinct:
            assert pval > 1e-4, (pval, counts, p * B)
        else:
            assert pval < 1e-6, pval
