"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test names the passage it follows.  The oracle is test infrastructure;
these tests are what make it trustworthy as the parity reference.
"""
import itertools
import math

import numpy as np
import pytest

from conftest import golden_lines


# ---------------------------------------------------------------- Philox

def test_philox_known_answers(oracle):
    """Random123 known-answer vectors for Philox4x32-10 (Salmon et al., SC'11)."""
    rows = golden_lines("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for ln in rows:
        lhs, rhs = ln.split("->")
        vals = [int(x, 16) for x in lhs.split()]
        want = [int(x, 16) for x in rhs.split()]
        assert oracle.philox4x32_10(vals[:4], vals[4:6]) == want


def test_uniform_mapping(oracle):
    """u_accept uses the top 24 bits of word 0, u_sample the top 53 bits of
    (w0:w1); counter = (b, k, draw, 0), key = (lo32(seed), hi32(seed))."""
    seed = 0x0123456789ABCDEF
    for b, k in [(0, 0), (5, 3), (511, 15), (2**31, 7)]:
        w = oracle.philox4x32_10([b, k, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.u_accept(seed, b, k) == (w[0] >> 8) / 2.0**24
        w = oracle.philox4x32_10([b, k, 1, 0], [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.u_sample(seed, b, k) == (((w[0] << 32) | w[1]) >> 11) / 2.0**53
    us = [oracle.u_accept(7, b, 0) for b in range(2000)]
    assert 0.0 <= min(us) and max(us) < 1.0
    assert abs(np.mean(us) - 0.5) < 0.03


def test_uniform_mapping_from_known_answers(oracle):
    """The acceptance uniform of (seed 0, request 0, position 0) is the first
    known-answer vector's word 0 (counter and key all zero, read from the
    golden fixture, not from the oracle's generator) shifted to 24 bits; the
    acceptance uniforms lie on the 2^-24 grid and the sampling uniforms are
    uniform on [0, 1) (Kolmogorov-Smirnov)."""
    lhs, rhs = golden_lines("philox4x32_10_kat.txt")[0].split("->")
    assert [int(x, 16) for x in lhs.split()] == [0] * 6
    w0 = int(rhs.split()[0], 16)
    assert oracle.u_accept(0, 0, 0) == (w0 >> 8) * 2.0 ** -24
    ua = np.array([oracle.u_accept(99, b, k) for b in range(200) for k in range(8)])
    assert np.all(ua * 2.0 ** 24 == np.floor(ua * 2.0 ** 24))
    stats = pytest.importorskip("scipy.stats")
    us = np.array([oracle.u_sample(2026, b, k) for b in range(4000) for k in range(5)])
    assert stats.kstest(us, "uniform").pvalue > 1e-3
    assert len(np.unique(us)) == us.size


# ---------------------------------------------------------------- hand rule

def _logp(p):
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.where(p > 0, np.log(np.where(p > 0, p, 1.0)), -np.inf)


def test_hand_rule_4_tokens(oracle):
    """'Правило проверки' (kiosknews.app, 'Немного теории'), worked by hand."""
    rows = golden_lines("hand_rule_4tok.txt")
    assert len(rows) >= 8
    for ln in rows:
        name, p, q, x, ua, acc, us, tok = [f.strip() for f in ln.split("|")]
        p = [float(v) for v in p.split()]
        q = [float(v) for v in q.split()]
        x, acc, tok = int(x), int(acc), int(tok)
        ua, us = float(ua), float(us)
        target = np.stack([_logp(p), np.zeros(4)])       # row 1: bonus row (uniform)
        draft = _logp(q)[None, :]
        out, a = oracle.verify_request_u(target, draft, [x], 1, 1.0, [ua], us)
        assert a == acc, name
        if acc:
            assert out[0] == x, name
        else:
            assert out[0] == tok, name
        assert out[1] == (-1 if not acc else out[1]), name


def test_hand_bonus_token(oracle):
    """All drafts accepted -> one more token from the target row K+1 (braintools.ru,
    'Как это работает': 'ещё один следующий токен – итого шесть')."""
    p1 = [0.1, 0.2, 0.3, 0.4]  # bonus row
    target = np.stack([_logp([0.25] * 4), _logp(p1)])
    draft = _logp([0.25] * 4)[None, :]
    # C = (.1,.3,.6,1.0)
    for u, want in [(0.0, 0), (0.05, 0), (0.15, 1), (0.35, 2), (0.7, 3), (0.999, 3)]:
        out, a = oracle.verify_request_u(target, draft, [2], 1, 1.0, [0.5], u)
        assert a == 1 and out[0] == 2 and out[1] == want


def test_inverse_cdf_edges(oracle):
    assert oracle.inverse_cdf([0.0, 0.0, 1.0, 0.0], 0.0)[0] == 2
    assert oracle.inverse_cdf([0.0, 0.0, 1.0, 0.0], 0.999999)[0] == 2
    assert oracle.inverse_cdf([1.0, 1.0], 0.5)[0] == 1       # C_0 = 1 is not > 1
    assert oracle.inverse_cdf([1.0, 1.0], 0.4999)[0] == 0
    # residual with Z == 0 falls back to p
    t, _ = oracle.sample_residual([0.5, 0.5], [0.5, 0.5], 0.75)
    assert t == 1


# ---------------------------------------------------------------- exact law

def _tables(rng, V, K, spread=1.0):
    """Context-dependent target P(.|prefix) for prefixes of length 0..K and
    draft Q(.|prefix) for lengths 0..K-1, as dicts keyed by prefix tuples."""
    P, Q = {}, {}
    for n in range(K + 1):
        for pre in itertools.product(range(V), repeat=n):
            P[pre] = rng.dirichlet(np.full(V, spread))
            if n < K:
                Q[pre] = rng.dirichlet(np.full(V, spread))
    return P, Q


def _bisect(f, lo=0.0, hi=1.0, iters=60):
    """Largest u in [lo,hi) with f(u) True assuming f is True then False."""
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if f(mid):
            lo = mid
        else:
            hi = mid
    return lo


def _emitted_law(oracle, P, Q, V, K, T):
    """Exact output law of the oracle for every draft sequence, integrating
    the acceptance and sampling uniforms by bisection on the oracle's own
    decisions (which are monotone in u).  Returns {emitted tuple: prob}."""
    law = {}
    one = 1.0 - 2.0**-40
    T = float(np.float32(T))  # the oracle reads T as float32
    for x in itertools.product(range(V), repeat=K):
        wx = 1.0
        for k in range(K):
            wx *= Q[x[:k]][x[k]]
        tgt = np.stack([np.log(P[x[:k]]) * T for k in range(K + 1)])
        drf = np.stack([np.log(Q[x[:k]]) * T for k in range(K)])

        def run(ua, us):
            return oracle.verify_request_u(tgt, drf, x, K, T, ua, us)

        # acceptance probability at each position, positions before it forced
        # to accept (u = 0 accepts since every p > 0)
        acc = []
        for k in range(K):
            def accepted(u, k=k):
                ua = [0.0] * K
                ua[k] = u
                return run(ua, 0.5)[1] > k
            if accepted(one):
                acc.append(1.0)
            else:
                acc.append(_bisect(accepted))
        reach = 1.0
        for a in range(K + 1):
            if a < K:
                pr_stop = reach * (1.0 - acc[a])
            else:
                pr_stop = reach
            if pr_stop > 0.0:
                ua = [0.0] * K
                if a < K:
                    ua[a] = one
                # token(u) is non-decreasing in u: find each boundary
                prev = 0.0
                for v in range(V):
                    if v < V - 1:
                        bnd = _bisect(lambda u: run(ua, u)[0][a] <= v)
                        if run(ua, 0.0)[0][a] > v:
                            bnd = 0.0
                    else:
                        bnd = 1.0
                    pv = max(0.0, bnd - prev)
                    prev = max(prev, bnd)
                    if pv > 0.0:
                        e = tuple(x[:a]) + (v,)
                        law[e] = law.get(e, 0.0) + wx * pr_stop * pv
            if a < K:
                reach *= acc[a]
    return law


@pytest.mark.parametrize("V,K,T,seed", [(4, 3, 1.0, 1), (5, 2, 0.7, 2), (8, 2, 1.3, 3)])
def test_lossless_exact_enumeration(oracle, V, K, T, seed):
    """'Утверждение 1' (kiosknews.app): the emitted tokens follow the target
    law exactly, whatever q.  Continuing with target sampling after the
    emitted prefix must reproduce P_target for every length-(K+1) sequence."""
    rng = np.random.default_rng(seed)
    P, Q = _tables(rng, V, K)
    law = _emitted_law(oracle, P, Q, V, K, T)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    worst = 0.0
    for s in itertools.product(range(V), repeat=K + 1):
        want = 1.0
        for j in range(K + 1):
            want *= P[s[:j]][s[j]]
        got = 0.0
        for n in range(1, K + 2):
            e = s[:n]
            if e in law:
                cont = 1.0
                for j in range(n, K + 1):
                    cont *= P[s[:j]][s[j]]
                got += law[e] * cont
        worst = max(worst, abs(got - want))
    assert worst < 1e-12
    # first emitted token ~ p_0
    first = np.zeros(V)
    for e, pr in law.items():
        first[e[0]] += pr
    assert np.max(np.abs(first - P[()])) < 1e-12


MUTANTS = {
    # the acceptance ratio inverted: accept with min(1, q/p)
    "inverted_ratio": ("return u * q_x < p_x;", "return u * p_x < q_x;"),
    # residual of the wrong sign: max(0, q - p)
    "residual_sign": ("double d = p[v] - q[v];", "double d = q[v] - p[v];"),
    # after a rejection sample from p instead of the residual
    "resample_from_p": ("return svo_inverse_cdf(r_scratch, V, u, margin);",
                        "return svo_inverse_cdf(p, V, u, margin);"),
    # bonus token taken from the last draft row's target row instead of row K
    "bonus_row": ("svo_row_softmax(svo_row(tgt, dtype, (size_t)a, V), dtype, V, Td, p, NULL, NULL);",
                  "svo_row_softmax(svo_row(tgt, dtype, (size_t)(a > 0 ? a - 1 : 0), V), dtype, V, Td, p, NULL, NULL);"),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_exact_enumeration_catches_planted_mistakes(oracle, mutant, tmp_path):
    """The enumeration check is sensitive: a copy of the oracle with one
    planted mistake (compiled on the CPU into a temporary library) breaks the
    lossless identity."""
    import ctypes
    import os
    import subprocess
    import oracle.build as ob
    src = open(ob.SRC).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) == 1, mutant
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    subprocess.check_call(["gcc", *ob.CFLAGS, str(path), "-o", so, "-lm", "-lpthread"])
    good = oracle.lib()
    mut = ctypes.CDLL(so)
    mut.svo_verify_request_u.argtypes = good.svo_verify_request_u.argtypes
    rng = np.random.default_rng(5)
    V, K = 4, 2
    P, Q = _tables(rng, V, K)
    oracle._lib = mut
    try:
        law = _emitted_law(oracle, P, Q, V, K, 1.0)
    finally:
        oracle._lib = good
    worst = 0.0
    for s in itertools.product(range(V), repeat=K + 1):
        want = 1.0
        for j in range(K + 1):
            want *= P[s[:j]][s[j]]
        got = 0.0
        for n in range(1, K + 2):
            e = s[:n]
            if e in law:
                cont = 1.0
                for j in range(n, K + 1):
                    cont *= P[s[:j]][s[j]]
                got += law[e] * cont
        worst = max(worst, abs(got - want))
    assert worst > 1e-4, mutant


# ---------------------------------------------------------------- greedy

def test_greedy_equals_argmax_decoding(oracle):
    """braintools.ru, 'Почему ответ не портится': at temperature 0 the check is
    an argmax comparison, so the output equals autoregressive argmax decoding
    for accept_len + 1 steps; ties go to the lowest index."""
    rng = np.random.default_rng(11)
    V, K = 5, 3
    P = {}
    for n in range(K + 1):
        for pre in itertools.product(range(V), repeat=n):
            z = rng.integers(-3, 3, size=V).astype(np.float32)  # integer logits: many ties
            P[pre] = z
    for x in itertools.product(range(V), repeat=K):
        tgt = np.stack([P[x[:k]] for k in range(K + 1)])
        for T in (0.0, -1.0, float("nan"), 1e-45):  # all greedy
            out, a = oracle.verify_request_u(tgt, None, x, K, T, [0.5] * K, 0.5)
            g = []
            for j in range(K + 1):
                pre = tuple(g)
                z = P[pre]
                g.append(int(np.flatnonzero(z == z.max())[0]))
                if j < K and x[j] != g[-1]:
                    break
            assert a == len(g) - 1
            assert list(out[:a + 1]) == g
            assert all(v == -1 for v in out[a + 1:])


def test_greedy_bf16_ties_lowest_index(oracle):
    bits = np.array([0x3F80, 0x4000, 0x4000, 0x3F80], dtype=np.uint16)  # 1, 2, 2, 1
    assert oracle.row_argmax(bits) == 1
    assert oracle.row_argmax(np.array([-np.inf, -np.inf, 3.0, 3.0], np.float32)) == 2


# ---------------------------------------------------------------- statistics

def test_chi_square_first_token(oracle):
    """10^6 seeded oracle trials (its own Philox): the first emitted token is
    distributed as p_0 ('Утверждение 1'); chi-square p-value > 0.01."""
    stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(20261202)
    V, K, T, N = 16, 3, 0.9, 1_000_000
    tgt = rng.normal(0, 1.5, size=(1, K + 1, V)).astype(np.float32)
    drf = (tgt[:, :K] + rng.normal(0, 1.0, size=(1, K, V))).astype(np.float32)
    q = np.stack([oracle.row_softmax(drf[0, k], T)[0] for k in range(K)])
    p0 = oracle.row_softmax(tgt[0, 0], T)[0]
    toks = np.stack([rng.choice(V, size=N, p=q[k] / q[k].sum()) for k in range(K)], axis=1)
    res = oracle.verify(tgt, drf, toks.astype(np.int32), None, np.full(N, T, np.float32),
                        seed=99, nthreads=oracle.cpu_count(), broadcast_rows=True)
    counts = np.bincount(res["out_tokens"][:, 0], minlength=V).astype(np.float64)
    exp = p0 * N
    order = np.argsort(exp)
    obs_m, exp_m, acc_o, acc_e = [], [], 0.0, 0.0
    for i in order:  # merge small bins until expected >= 5
        acc_o += counts[i]
        acc_e += exp[i]
        if acc_e >= 5:
            obs_m.append(acc_o)
            exp_m.append(acc_e)
            acc_o = acc_e = 0.0
    if acc_e > 0:
        obs_m[-1] += acc_o
        exp_m[-1] += acc_e
    exp_m = np.array(exp_m) * (N / np.sum(exp_m))
    pval = stats.chisquare(obs_m, exp_m).pvalue
    assert pval > 0.01, pval
    # the draft is poor on purpose: many rejections were exercised
    assert np.mean(res["accept_len"]) < 2.0


def test_mean_accept_length_closed_form(oracle):
    """'Утверждение 2' (kiosknews.app): E[A] = sum_k P(A >= k); with x_k ~ q_k
    drawn independently, P(A >= j) = prod_{k<j} beta_k, beta_k = sum min(p_k, q_k)."""
    from oracle import tau
    rng = np.random.default_rng(3)
    V, K, T, N = 12, 4, 1.0, 200_000
    tgt = rng.normal(0, 1.0, size=(1, K + 1, V)).astype(np.float32)
    drf = (tgt[:, :K] + rng.normal(0, 0.6, size=(1, K, V))).astype(np.float32)
    p = np.stack([oracle.row_softmax(tgt[0, k], T)[0] for k in range(K)])
    q = np.stack([oracle.row_softmax(drf[0, k], T)[0] for k in range(K)])
    beta = np.minimum(p, q).sum(axis=1)
    toks = np.stack([rng.choice(V, size=N, p=q[k] / q[k].sum()) for k in range(K)], axis=1)
    res = oracle.verify(tgt, drf, toks.astype(np.int32), None, np.full(N, T, np.float32),
                        seed=5, nthreads=oracle.cpu_count(), broadcast_rows=True)
    a = res["accept_len"].astype(np.float64)
    want = tau.mean_accept_len(beta)
    assert abs(a.mean() - want) < 4.0 * a.std() / math.sqrt(N)
    # survival profile matches position by position
    for j in range(1, K + 1):
        pj = np.prod(beta[:j])
        got = np.mean(a >= j)
        assert abs(got - pj) < 4.0 * math.sqrt(pj * (1 - pj) / N) + 1e-12


# ---------------------------------------------------------------- tau helpers

def test_tau_helpers_match_printed_values():
    """Numbers printed by braintools.ru ('Сколько это даёт') and the DFlash 2
    survival profile and table of kiosknews.app ('Утверждение 2')."""
    from oracle import tau
    for ln in golden_lines("tau_values.txt"):
        lhs, rhs = ln.split("=")
        f = lhs.split()
        kind, args = f[0], [float(v) for v in f[1:]]
        vals = [float(v) for v in rhs.split()]
        tol = vals[-1]
        if kind == "expected_tokens":
            assert abs(tau.expected_tokens(args[0], int(args[1])) - vals[0]) < tol
        elif kind == "speedup":
            assert abs(tau.speedup(args[0], int(args[1]), args[2]) - vals[0]) < tol
        elif kind == "best_gamma":
            g, s = tau.best_gamma(args[0], args[1])
            assert g == int(vals[0]) and abs(s - vals[1]) < tol
        elif kind == "best_speedup":
            assert abs(tau.best_gamma(args[0], args[1])[1] - vals[0]) < tol
        elif kind == "survival":
            assert abs(tau.tau_from_survival(args) - vals[0]) < tol
        else:
            raise AssertionError(kind)


# ---------------------------------------------------------------- schedule

def test_schedule_hand_cases(oracle):
    """DSpark (iitog.ru): verify length from the survival probability of the
    draft prefix, read as the running product of draft max-probabilities."""
    mp = np.array([[0.9, 0.8, 0.5],
                   [0.9, 0.8, 0.5],
                   [0.2, 0.9, 0.9],
                   [1.0, 1.0, 1.0],
                   [0.9, float("nan"), 1.0]], dtype=np.float32)
    thr = [0.3, 0.4, 0.3, 0.3, 0.3]
    # products 0.9, 0.72, 0.36: all >= 0.3 -> 3; 0.36 < 0.4 -> 2; 0.2 < 0.3 -> 0
    want = [3, 2, 0, 3, 1]
    for b in range(5):
        assert oracle.schedule_len(mp[b:b + 1], thr[b])[0] == want[b]
    assert list(oracle.schedule_len(mp, 0.3)) == [3, 3, 0, 3, 1]
    assert oracle.schedule_len(np.array([[0.5, 0.5]], np.float32), 0.25)[0] == 2  # 0.25 >= 0.25
    assert oracle.schedule_len(np.array([[0.5]], np.float32), 1.5)[0] == 0
    # float32 rounding of the running product decides: 0.1f*0.1f*... vs threshold
    c = np.float32(0.7)
    prods = np.cumprod(np.full(6, c, dtype=np.float32), dtype=np.float32)
    thr6 = prods[3]  # exactly the 4th float32 product
    assert oracle.schedule_len(np.full((1, 6), c, np.float32), thr6)[0] == 4


# ---------------------------------------------------------------- validation

def test_length_clamp_and_bad_tokens(oracle):
    rng = np.random.default_rng(0)
    V, K = 6, 3
    tgt = rng.normal(size=(4, K + 1, V)).astype(np.float32)
    drf = rng.normal(size=(4, K, V)).astype(np.float32)
    toks = np.array([[1, 2, 3], [1, 9, 3], [-1, 2, 3], [0, 0, 0]], np.int32)
    vl = np.array([5, 3, 2, -2], np.int32)
    res = oracle.verify(tgt, drf, toks, vl, np.zeros(4, np.float32), seed=1)
    st = res["status"]
    assert st[0] == oracle.BAD_LEN            # 5 > K
    assert st[1] == oracle.BAD_TOKEN          # token 9 >= V at position 1
    assert res["accept_len"][1] <= 1
    assert st[2] == oracle.BAD_TOKEN and res["accept_len"][2] == 0
    assert st[3] == oracle.BAD_LEN and res["accept_len"][3] == 0
    for b in range(4):
        a = res["accept_len"][b]
        assert all(v == -1 for v in res["out_tokens"][b, a + 1:])


# ---------------------------------------------------------------- load-aware schedule, confidence

def test_schedule_budget_hand_cases(oracle):
    """"DSpark ... верификацией по уверенности" (iitog.ru), "Ключевые факты": the
    verify length follows the prefix's survival probability and the engine's load.
    Survival of (b, k) is the running product of the draft max-probabilities; a
    budget of N positions keeps the N most likely to survive."""
    import numpy as np
    mp = np.array([[0.9, 0.8, 0.5], [0.95, 0.1, 1.0]], np.float32)
    # survival: request 0: 0.9, 0.72, 0.36; request 1: 0.95, 0.095, 0.095
    assert oracle.schedule_budget(mp, 3).tolist() == [2, 1]
    assert oracle.schedule_budget(mp, 4).tolist() == [3, 1]
    assert oracle.schedule_budget(mp, 5).tolist() == [3, 2]   # tie 0.095: lower k first
    assert oracle.schedule_budget(mp, 0).tolist() == [0, 0]
    assert oracle.schedule_budget(mp, 100).tolist() == [3, 3]
    ones = np.ones((2, 4), np.float32)                        # all survival 1: lower b first
    assert oracle.schedule_budget(ones, 5).tolist() == [4, 1]
    odd = np.array([[np.nan, 0.5], [1.5, 0.5]], np.float32)   # NaN -> 0, 1.5 -> 1
    assert oracle.schedule_budget(odd, 1).tolist() == [0, 1]
    assert oracle.schedule_budget(odd, 3).tolist() == [1, 2]


def test_schedule_budget_matches_threshold_rule(oracle):
    """With the budget set to the number of positions whose survival reaches a
    threshold, the kept set is exactly the threshold schedule's (the separately
    pinned confidence-scheduled verify length)."""
    import numpy as np
    rng = np.random.default_rng(5)
    for trial in range(20):
        mp = rng.uniform(0.05, 1.0, size=(64, 12)).astype(np.float32)
        tau = float(rng.uniform(0.05, 0.6))
        L = oracle.schedule_len(mp, tau)
        assert oracle.schedule_budget(mp, int(L.sum())).tolist() == L.tolist()


def test_draft_confidence_hand_values(oracle):
    """max_v q(v) at temperature T: a uniform row gives 1/V; logits (ln 3, 0) give
    3/4; halving T squares the odds (9/10); a greedy request's q is a point mass."""
    import numpy as np
    d = np.zeros((2, 2, 4), np.float64)
    d[0, 1] = [np.log(3.0), 0.0, -np.inf, -np.inf]
    d[1, 0] = [np.log(3.0), 0.0, -np.inf, -np.inf]
    c = oracle.draft_confidence(d, np.array([1.0, 0.5], np.float32))
    assert np.allclose(c[0], [0.25, 0.75], rtol=1e-14)
    assert abs(c[1, 0] - 0.9) < 1e-14 and abs(c[1, 1] - 0.25) < 1e-14
    g = oracle.draft_confidence(d, np.array([0.0, float("nan")], np.float32))
    assert (g == 1.0).all()


# ---------------------------------------------------------------- tree verification (greedy)

def test_tree_greedy_hand_case(oracle):
    """Root argmax 2 -> node 2 (the child carrying 2); node 2's argmax 1 has no
    child: one accepted node, then token 1.  Siblings carrying the same token:
    the lowest-index node is taken."""
    import numpy as np
    t = np.zeros((5, 6))
    t[0, 2] = 1; t[1, 3] = 1; t[2, 1] = 1; t[3, 4] = 1; t[4, 5] = 1
    ot, on, a = oracle.verify_tree_greedy(t, [-1, 0, 0, 1, 2], [0, 3, 2, 3, 1])
    assert a == 2 and ot.tolist() == [2, 1, 5, -1, -1] and on.tolist() == [2, 4, -1, -1, -1]
    ot, on, a = oracle.verify_tree_greedy(t, [-1, 0, 0, 0, 2], [0, 2, 2, 3, 1])  # nodes 1, 2 both carry 2
    assert a == 1 and on.tolist()[:1] == [1] and ot.tolist()[:2] == [2, 3]


def test_tree_greedy_chain_is_linear_verification(oracle):
    """A chain tree (parent[n] = n - 1) is the linear draft: same accepted count
    and tokens as the (separately pinned) greedy verification of K = N - 1
    drafts on the same target rows."""
    import numpy as np
    rng = np.random.default_rng(8)
    for trial in range(40):
        N, V = int(rng.integers(1, 10)), int(rng.integers(2, 7))
        tgt = rng.integers(-2, 3, size=(N, V)).astype(np.float64)
        tok = rng.integers(0, V, size=N).astype(np.int32)
        for n in range(1, N):  # make some drafts right
            if rng.random() < 0.6:
                tok[n] = int(np.argmax(tgt[n - 1]))
        ot, on, a = oracle.verify_tree_greedy(tgt, np.arange(-1, N - 1), tok)
        K = N - 1
        if K == 0:
            assert a == 0 and ot[0] == int(np.argmax(tgt[0]))
            continue
        r = oracle.verify(tgt[None], np.zeros((1, K, V)), tok[None, 1:], None,
                          np.zeros(1, np.float32), 1)
        assert a == r["accept_len"][0]
        assert ot.tolist() == r["out_tokens"][0].tolist()


def test_tree_greedy_matches_valid_set(oracle):
    """Brute force on random trees: a node is valid when its parent is valid, its
    token is the argmax of the parent's row and no lower-index sibling carries
    that token; the valid nodes form one chain and the accepted count is the
    depth of its deepest node."""
    import numpy as np
    rng = np.random.default_rng(9)
    for trial in range(200):
        N, V = int(rng.integers(1, 12)), int(rng.integers(2, 5))
        tgt = rng.integers(-1, 2, size=(N, V)).astype(np.float32)
        parent = np.array([-1] + [int(rng.integers(0, n)) for n in range(1, N)], np.int32)
        tok = rng.integers(0, V, size=N).astype(np.int32)
        am = [int(np.argmax(tgt[n])) for n in range(N)]
        valid, depth = {0}, {0: 0}
        for v in range(1, N):
            u = parent[v]
            first = min(c for c in range(1, N) if parent[c] == u and tok[c] == tok[v])
            if u in valid and tok[v] == am[u] and first == v:
                valid.add(v)
                depth[v] = depth[u] + 1
        deepest = max(valid, key=lambda v: depth[v])
        ot, on, a = oracle.verify_tree_greedy(tgt, parent, tok)
        assert a == depth[deepest]
        assert ot[a] == am[deepest]


# ---------------------------------------------------------------- tree verification (sampled)

def test_tree_sampled_chain_is_linear_verification(oracle):
    """A chain tree (parent[n] = n - 1) is the linear draft: with one child per
    node the multi-candidate rule is the pages' rule ('Правило проверки',
    kiosknews.app) step for step, and the Philox keys of node c (acceptance of
    position c - 1, sampling at position c) are the linear ones, so the
    (separately pinned) linear verification gives the same tokens and counts,
    including invalid tokens, which cut the chain."""
    rng = np.random.default_rng(12)
    for trial in range(60):
        B, N, V = int(rng.integers(1, 5)), int(rng.integers(1, 9)), int(rng.integers(2, 40))
        T = rng.choice([1.0, 0.6, 1.7, 0.0], size=B).astype(np.float32)
        tgt = rng.normal(size=(B, N, V)) * 1.5
        drf = tgt + rng.normal(size=(B, N, V)) * 0.7   # drafts near the target: long chains
        tok = np.zeros((B, N), np.int32)
        for b in range(B):
            for n in range(1, N):
                z = drf[b, n - 1] / max(float(T[b]), 0.5)
                e = np.exp(z - z.max())
                tok[b, n] = rng.choice(V, p=e / e.sum())
        if trial % 7 == 3 and N > 2:
            tok[0, N // 2] = V + 3                     # cuts the chain
        parent = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
        seed = int(rng.integers(1, 2**62))
        r = oracle.verify_tree(tgt, drf, parent, tok, T, seed)
        if N == 1:
            assert (r["accept_len"] == 0).all()
            continue
        lin = oracle.verify(tgt, drf[:, :N - 1], tok[:, 1:], None, T, seed)
        assert np.array_equal(r["accept_len"], lin["accept_len"]), trial
        assert np.array_equal(r["out_tokens"], lin["out_tokens"]), trial
        a = r["accept_len"]
        for b in range(B):
            assert r["out_nodes"][b, :a[b]].tolist() == list(range(1, a[b] + 1))


def _tree_law(run, parent, tok, N, V, one=1.0 - 2.0**-40):
    """Exact law of the emitted tokens of one tree walk, integrating every
    acceptance and sampling uniform by bisection on the oracle's own decisions
    (each monotone in its uniform).  run(ua, us) -> (out_tokens, out_nodes, a).
    Returns {emitted tuple: probability}."""
    law = {}

    def explore(ua, cur, depth, prob, prefix):
        reach = prob
        ua = list(ua)
        for c in [c for c in range(cur + 1, N) if parent[c] == cur]:
            if reach == 0.0:
                break

            def accepted(u, c=c):
                w = list(ua)
                w[c] = u
                _, on, a = run(w, [0.5] * N)
                return a > depth and on[depth] == c
            t = 1.0 if accepted(one) else (_bisect(accepted) if accepted(0.0) else 0.0)
            if t > 0.0:
                w = list(ua)
                w[c] = 0.0
                explore(w, c, depth + 1, reach * t, prefix + (int(tok[c]),))
            ua[c] = one
            reach *= 1.0 - t
        if reach == 0.0:
            return
        prev = 0.0
        for v in range(V):
            def at_most(u):
                us = [0.5] * N
                us[cur] = u
                return run(ua, us)[0][depth] <= v
            if v == V - 1:
                bnd = 1.0
            elif not at_most(0.0):
                bnd = 0.0
            else:
                bnd = _bisect(at_most)
            pv = max(0.0, bnd - prev)
            prev = max(prev, bnd)
            if pv > 0.0:
                e = prefix + (v,)
                law[e] = law.get(e, 0.0) + reach * pv

    explore([0.0] * N, 0, 0, 1.0, ())
    return law


def _tree_from_tables(P, Q, parent, tok, T, K):
    """Node rows of a tree whose node n follows the token prefix of its path:
    target row log P(.|prefix)*T, draft row log Q(.|prefix)*T (zeros where the
    prefix is longer than the tables)."""
    N = len(parent)
    V = len(P[()])
    pre = [()] * N
    for n in range(1, N):
        pre[n] = pre[parent[n]] + (int(tok[n]),)
    tgt = np.stack([np.log(P[pre[n]]) * T for n in range(N)])
    drf = np.stack([np.log(Q[pre[n]]) * T if len(pre[n]) < K else np.zeros(V) for n in range(N)])
    return tgt, drf, pre


def _assignment_weight(Q, pre, parent, tok, distinct):
    """Probability of one token assignment of the candidates: each child drawn
    from its parent's draft distribution, independently, or (distinct) the
    siblings one after another in index order without replacement (a child's
    law is the draft law without its earlier siblings' tokens, renormalised)."""
    N = len(parent)
    w = 1.0
    for n in range(1, N):
        q = Q[pre[parent[n]]]
        if not distinct:
            w *= q[tok[n]]
            continue
        used = [int(tok[m]) for m in range(1, n) if parent[m] == parent[n]]
        if int(tok[n]) in used:
            return 0.0
        w *= q[tok[n]] / (1.0 - sum(q[u] for u in used))
    return w


def _tree_lossless_worst(oracle, P, Q, parent, V, K, T, distinct=False):
    """Largest error of the tree walk's law against the target law, over every
    token assignment of the candidates (each child drawn from its parent's
    draft distribution, independently or, with distinct, siblings without
    replacement), every continuation filled in by target sampling up to K + 1
    tokens."""
    T = float(np.float32(T))
    N = len(parent)
    agg = {}
    for assign in itertools.product(range(V), repeat=N - 1):
        tok = np.array((0,) + assign, np.int32)
        tgt, drf, pre = _tree_from_tables(P, Q, parent, tok, T, K)
        w = _assignment_weight(Q, pre, parent, tok, distinct)
        if w == 0.0:
            continue
        law = _tree_law(lambda ua, us: oracle.verify_tree_u(tgt, drf, parent, tok, T, ua, us,
                                                            distinct=distinct),
                        parent, tok, N, V)
        for e, pr in law.items():
            agg[e] = agg.get(e, 0.0) + w * pr
    assert abs(sum(agg.values()) - 1.0) < 1e-12
    worst = 0.0
    for s in itertools.product(range(V), repeat=K + 1):
        want = 1.0
        for j in range(K + 1):
            want *= P[s[:j]][s[j]]
        got = 0.0
        for n in range(1, K + 2):
            if s[:n] in agg:
                cont = 1.0
                for j in range(n, K + 1):
                    cont *= P[s[:j]][s[j]]
                got += agg[s[:n]] * cont
        worst = max(worst, abs(got - want))
    return worst


TREE_SHAPES = {
    # parents of nodes 1..N-1 (node 0 is the root)
    "three_siblings": ([-1, 0, 0, 0], 4, 1),
    "two_levels": ([-1, 0, 0, 1, 1, 2], 3, 2),
}


@pytest.mark.parametrize("shape,T,seed", [("three_siblings", 1.0, 1), ("three_siblings", 0.7, 2),
                                          ("two_levels", 1.0, 3), ("two_levels", 1.4, 4)])
def test_tree_sampled_lossless_exact_enumeration(oracle, shape, T, seed):
    """'Утверждение 1' (kiosknews.app) for trees: whatever the draft, when every
    child is drawn independently from its parent's draft distribution the
    emitted tokens follow the target law exactly.  Enumerates every token
    assignment of the candidates and integrates every uniform; siblings share
    a draft row, so this checks the residual updates between them, and the
    two-level tree checks that the walk reads the accepted node's rows."""
    parent, V, K = TREE_SHAPES[shape]
    rng = np.random.default_rng(seed)
    P, Q = _tables(rng, V, K)
    worst = _tree_lossless_worst(oracle, P, Q, np.array(parent, np.int32), V, K, T)
    assert worst < 1e-12, worst


TREE_MUTANTS = {
    # siblings tested against p again instead of the updated residual
    "tree_no_residual_update": ("double w = r[v] / Z - q[v];", "double w = r[v] / Z;"),
    # the residual's normaliser left out of the acceptance test
    "tree_unnormalised": ("const double rx = r[x] / Z;", "const double rx = r[x];"),
    # rows of the node at the path's depth instead of the current node
    "tree_row_by_depth": (
        "svo_row_softmax(svo_row(target, dtype, (size_t)cur, V), dtype, V, Td, p, NULL, NULL);",
        "svo_row_softmax(svo_row(target, dtype, (size_t)depth, V), dtype, V, Td, p, NULL, NULL);"),
    # the emitted token sampled from p after rejected siblings
    "tree_sample_p": ("out_tokens[depth] = svo_inverse_cdf(r, V, u_s[cur], &d.cdf_margin);",
                      "out_tokens[depth] = svo_inverse_cdf(p, V, u_s[cur], &d.cdf_margin);"),
}


@pytest.mark.parametrize("mutant", sorted(TREE_MUTANTS))
def test_tree_enumeration_catches_planted_mistakes(oracle, mutant, tmp_path):
    """The tree enumeration is sensitive: a copy of the oracle with one planted
    mistake in the tree walk breaks the lossless identity on one of the shapes."""
    import ctypes
    import subprocess
    import oracle.build as ob
    src = open(ob.SRC).read()
    old, new = TREE_MUTANTS[mutant]
    assert src.count(old) == 1, mutant
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    subprocess.check_call(["gcc", *ob.CFLAGS, str(path), "-o", so, "-lm", "-lpthread"])
    good = oracle.lib()
    mut = ctypes.CDLL(so)
    mut.svo_verify_tree_u.argtypes = good.svo_verify_tree_u.argtypes
    mut.svo_verify_tree_u.restype = good.svo_verify_tree_u.restype
    oracle._lib = mut
    try:
        worst = 0.0
        for shape, seed in (("three_siblings", 1), ("two_levels", 3)):
            parent, V, K = TREE_SHAPES[shape]
            P, Q = _tables(np.random.default_rng(seed), V, K)
            try:
                worst = max(worst, _tree_lossless_worst(oracle, P, Q, np.array(parent, np.int32),
                                                        V, K, 1.0))
            except AssertionError:
                worst = 1.0   # the law does not even sum to 1
            if worst > 1e-4:
                break
    finally:
        oracle._lib = good
    assert worst > 1e-4, mutant


def test_tree_sampled_hand_case(oracle):
    """Two siblings carrying tokens 0 and 1 under p = (0.5, 0.5, 0), q = (0.75,
    0.25, 0): the first is accepted iff u < p/q = 2/3; after its rejection the
    residual is max(0, p - q) = (0, 0.25, 0), normalised (0, 1, 0), so the
    second (token 1, q = 0.25) is always accepted."""
    T = 1.0
    tgt = np.log(np.array([[0.5, 0.5, 1e-300], [1.0, 1.0, 1.0], [1.0, 1.0, 1.0]]))
    drf = np.log(np.array([[0.75, 0.25, 1e-300], [1.0, 1.0, 1.0], [1.0, 1.0, 1.0]]))
    parent = [-1, 0, 0]
    tok = [0, 0, 1]
    ot, on, a = oracle.verify_tree_u(tgt, drf, parent, tok, T, [0, 0.66, 0.0], 0.5)
    assert a == 1 and on[0] == 1 and ot[0] == 0
    ot, on, a = oracle.verify_tree_u(tgt, drf, parent, tok, T, [0, 0.67, 0.999], 0.5)
    assert a == 1 and on[0] == 2 and ot[0] == 1
    # leaf row 2 uniform: the emitted token after node 2 follows u_s of node 2
    ot, on, a = oracle.verify_tree_u(tgt, drf, parent, tok, T, [0, 0.67, 0.0], [0.5, 0.5, 0.9])
    assert ot[:2].tolist() == [1, 2] and ot[2] == -1
    # a token outside [0, V) is no candidate: the second sibling is tested first
    ot, on, a = oracle.verify_tree_u(tgt, drf, parent, [0, 7, 1], T, [0, 0.0, 0.4], 0.5)
    assert a == 1 and on[0] == 2


def test_tree_batch_offset_keeps_philox_index(oracle):
    """Row b of a sliced batch with b0 is request b0 + b: the slice reproduces
    the full batch's results for those requests."""
    rng = np.random.default_rng(21)
    B, N, V = 7, 6, 30
    tgt = rng.normal(size=(B, N, V))
    drf = tgt + rng.normal(size=(B, N, V)) * 0.8
    parent = np.array([[-1] + [int(rng.integers(0, n)) for n in range(1, N)] for _ in range(B)], np.int32)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    T = np.full(B, 1.0, np.float32)
    full = oracle.verify_tree(tgt, drf, parent, tok, T, 99)
    part = oracle.verify_tree(tgt[3:6], drf[3:6], parent[3:6], tok[3:6], T[3:6], 99, b0=3)
    for k in ("out_tokens", "out_nodes", "accept_len"):
        assert np.array_equal(full[k][3:6], part[k])


# ---------------------------------------------------------------- distinct siblings

DISTINCT_SHAPES = {
    "three_siblings": ([-1, 0, 0, 0], 4, 1),
    "two_levels": ([-1, 0, 0, 1, 1, 2], 3, 2),
    "four_of_four": ([-1, 0, 0, 0, 0], 4, 1),   # the siblings use up the whole vocabulary
}


@pytest.mark.parametrize("shape,T,seed", [("three_siblings", 1.0, 5), ("three_siblings", 0.6, 6),
                                          ("two_levels", 1.0, 7), ("two_levels", 1.3, 8),
                                          ("four_of_four", 1.0, 9)])
def test_tree_distinct_lossless_exact_enumeration(oracle, shape, T, seed):
    """'Утверждение 1' (kiosknews.app) for top-k style candidates: siblings are
    distinct tokens drawn one after another without replacement from their
    parent's draft distribution (the EAGLE top-k and DFlash 2 candidates of
    alesha.pro and kiosknews.app, '7. DFlash 2').  With each child's draft law
    taken as q without the rejected siblings' tokens, renormalised, the emitted
    tokens follow the target law exactly: every ordered distinct assignment of
    the candidates, weighted by its draw probability, and every uniform
    integrated."""
    parent, V, K = DISTINCT_SHAPES[shape]
    rng = np.random.default_rng(seed)
    P, Q = _tables(rng, V, K)
    worst = _tree_lossless_worst(oracle, P, Q, np.array(parent, np.int32), V, K, T, distinct=True)
    assert worst < 1e-12, worst


def test_tree_independent_rule_is_not_lossless_for_distinct_draws(oracle):
    """The independent-siblings rule applied to siblings drawn without
    replacement misses the target law: the two rules are not interchangeable,
    so the enumeration above tests something."""
    parent, V, K = DISTINCT_SHAPES["three_siblings"]
    P, Q = _tables(np.random.default_rng(5), V, K)
    par = np.array(parent, np.int32)
    T = 1.0
    agg = {}
    for assign in itertools.product(range(V), repeat=len(parent) - 1):
        tok = np.array((0,) + assign, np.int32)
        tgt, drf, pre = _tree_from_tables(P, Q, par, tok, T, K)
        w = _assignment_weight(Q, pre, par, tok, True)
        if w == 0.0:
            continue
        law = _tree_law(lambda ua, us: oracle.verify_tree_u(tgt, drf, par, tok, T, ua, us),
                        par, tok, len(parent), V)
        for e, pr in law.items():
            agg[e] = agg.get(e, 0.0) + w * pr
    first = np.zeros(V)
    for e, pr in agg.items():
        first[e[0]] += pr
    assert np.abs(first - P[()]).max() > 1e-3


def test_tree_distinct_hand_case(oracle):
    """p = (0.2, 0.5, 0.3), q = (0.6, 0.2, 0.2), siblings carrying tokens 0 then
    2.  The first is accepted iff u < p/q = 1/3.  After its rejection the
    residual is max(0, p - q) = (0, 0.3, 0.1), normalised (0, 0.75, 0.25), and
    the second sibling's draft law is q without token 0, renormalised:
    (0, 0.5, 0.5).  So it is accepted iff u * 0.5 < 0.25, u < 1/2 (under the
    independent rule, u * 0.2 < 0.25 always holds).  After its rejection the
    residual is max(0, (0, 0.75, 0.25) - (0, 0.5, 0.5)) = (0, 0.25, 0): token 1
    for every sampling uniform."""
    T = 1.0
    tgt = np.log(np.array([[0.2, 0.5, 0.3]] + [[1.0, 1.0, 1.0]] * 2))
    drf = np.log(np.array([[0.6, 0.2, 0.2]] + [[1.0, 1.0, 1.0]] * 2))
    parent, tok = [-1, 0, 0], [0, 0, 2]
    # first sibling accepted below 1/3
    ot, on, a = oracle.verify_tree_u(tgt, drf, parent, tok, T, [0, 0.33, 0.9], 0.5, distinct=True)
    assert a == 1 and on[0] == 1
    # second sibling: accepted below 1/2, rejected above
    ot, on, a = oracle.verify_tree_u(tgt, drf, parent, tok, T, [0, 0.34, 0.49], 0.5, distinct=True)
    assert a == 1 and on[0] == 2 and ot[0] == 2
    for us in (0.0, 0.5, 0.999):
        ot, on, a = oracle.verify_tree_u(tgt, drf, parent, tok, T, [0, 0.34, 0.51], us,
                                         distinct=True)
        assert a == 0 and ot[0] == 1, us
    # the independent rule accepts the second sibling at the same uniforms
    ot, on, a = oracle.verify_tree_u(tgt, drf, parent, tok, T, [0, 0.34, 0.51], 0.5)
    assert a == 1 and on[0] == 2
    # a sibling repeating a rejected sibling's token is no candidate
    tgt4 = np.concatenate([tgt, tgt[1:2]])
    drf4 = np.concatenate([drf, drf[1:2]])
    ot, on, a = oracle.verify_tree_u(tgt4, drf4, [-1, 0, 0, 0], [0, 0, 0, 2], T,
                                     [0, 0.34, 0.0, 0.49], 0.5, distinct=True)
    assert a == 1 and on[0] == 3


def test_tree_distinct_chain_equals_independent(oracle):
    """With one child per node no sibling is ever rejected before another is
    checked, so the distinct rule is the independent one (and the linear
    verification) on chains."""
    rng = np.random.default_rng(31)
    for trial in range(20):
        B, N, V = 3, int(rng.integers(2, 8)), int(rng.integers(3, 30))
        T = np.array([1.0, 0.7, 0.0], np.float32)
        tgt = rng.normal(size=(B, N, V)) * 1.5
        drf = tgt + rng.normal(size=(B, N, V)) * 0.7
        tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
        parent = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
        a = oracle.verify_tree(tgt, drf, parent, tok, T, 17 + trial)
        b = oracle.verify_tree(tgt, drf, parent, tok, T, 17 + trial, distinct=True)
        for k in ("out_tokens", "out_nodes", "accept_len"):
            assert np.array_equal(a[k], b[k]), (trial, k)


# (Leaving the rejected token's mass in q while renormalising the rest is no
# mistake: after a rejection r(x) = 0, and x is never checked again, so q(x)
# takes part in nothing.)
DISTINCT_MUTANTS = {
    # the renormalisation inverted: multiplied by the remaining mass
    "distinct_renormalise_inverted": ("for (int v = 0; v < V; ++v) q[v] = q[v] / rest;",
                                      "for (int v = 0; v < V; ++v) q[v] = q[v] * rest;"),
    # q not renormalised after the rejected token is removed
    "distinct_no_renormalise": ("for (int v = 0; v < V; ++v) q[v] = q[v] / rest;",
                                "for (int v = 0; v < V; ++v) q[v] = q[v];"),
    # siblings checked as if drawn independently
    "distinct_as_independent": ("if (distinct) {  /* the next sibling is drawn from q without x */",
                                "if (0) {"),
}


@pytest.mark.parametrize("mutant", sorted(DISTINCT_MUTANTS))
def test_tree_distinct_enumeration_catches_planted_mistakes(oracle, mutant, tmp_path):
    """A copy of the oracle with one planted mistake in the without-replacement
    update breaks the distinct enumeration."""
    import ctypes
    import subprocess
    import oracle.build as ob
    src = open(ob.SRC).read()
    old, new = DISTINCT_MUTANTS[mutant]
    assert src.count(old) == 1, mutant
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    subprocess.check_call(["gcc", *ob.CFLAGS, str(path), "-o", so, "-lm", "-lpthread"])
    good = oracle.lib()
    mut = ctypes.CDLL(so)
    mut.svo_verify_tree_u.argtypes = good.svo_verify_tree_u.argtypes
    mut.svo_verify_tree_u.restype = good.svo_verify_tree_u.restype
    oracle._lib = mut
    try:
        parent, V, K = DISTINCT_SHAPES["three_siblings"]
        P, Q = _tables(np.random.default_rng(5), V, K)
        try:
            worst = _tree_lossless_worst(oracle, P, Q, np.array(parent, np.int32), V, K, 1.0,
                                         distinct=True)
        except AssertionError:
            worst = 1.0   # the law does not even sum to 1
    finally:
        oracle._lib = good
    assert worst > 1e-4, mutant


# ---------------------------------------------------------------- LM-head logits

def _bf16_bits(x):
    """float32 values that are exactly bf16 -> their uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    assert ((b & 0xFFFF) == 0).all()
    return (b >> 16).astype(np.uint16)


def test_lm_logits_unit_vectors(oracle):
    """Hidden states that are unit vectors pick weight columns: z[i, v] =
    w[v, j_i] exactly."""
    rng = np.random.default_rng(40)
    d, V = 16, 7
    w = rng.normal(size=(V, d)).astype(np.float32)
    w = (w.view(np.uint32) & 0xFFFF0000).view(np.float32)   # round toward zero to bf16
    j = np.array([3, 0, 15, 7])
    h = np.zeros((4, d), np.float32)
    h[np.arange(4), j] = 1.0
    z = oracle.lm_logits(_bf16_bits(h), _bf16_bits(w))
    assert np.array_equal(z, w[:, j].T.astype(np.float64))


def test_lm_logits_small_integers_exact(oracle):
    """Small integer entries: every partial sum is an integer, so the result is
    exact in any order; checked against Python's exact integer arithmetic."""
    rng = np.random.default_rng(41)
    M, V, d = 5, 9, 64
    hi = rng.integers(-3, 4, size=(M, d))
    wi = rng.integers(-3, 4, size=(V, d))
    z = oracle.lm_logits(_bf16_bits(hi.astype(np.float32)), _bf16_bits(wi.astype(np.float32)))
    want = [[sum(int(a) * int(b) for a, b in zip(hi[i], wi[v])) for v in range(V)] for i in range(M)]
    assert np.array_equal(z, np.array(want, dtype=np.float64))


def test_lm_logits_against_library_matmul(oracle):
    """Random bf16 inputs against numpy's float64 matrix product of the same
    values (an independent summation): equal to within double rounding."""
    rng = np.random.default_rng(42)
    M, V, d = 6, 50, 256
    h = rng.normal(size=(M, d)).astype(np.float32)
    w = rng.normal(size=(V, d)).astype(np.float32) * 0.05
    h = (h.view(np.uint32) & 0xFFFF0000).view(np.float32)
    w = (w.view(np.uint32) & 0xFFFF0000).view(np.float32)
    z = oracle.lm_logits(_bf16_bits(h), _bf16_bits(w))
    ref = h.astype(np.float64) @ w.astype(np.float64).T
    scale = np.abs(h).astype(np.float64) @ np.abs(w).astype(np.float64).T
    assert (np.abs(z - ref) <= 1e-14 * scale + 1e-300).all()
    # the batch shape is kept
    z3 = oracle.lm_logits(_bf16_bits(h).reshape(2, 3, d), _bf16_bits(w))
    assert z3.shape == (2, 3, V) and np.array_equal(z3.reshape(M, V), z)
