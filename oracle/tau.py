"""Tokens-per-pass and speedup helpers (test infrastructure).

"Спекулятивный декодинг в проде" (kiosknews.app), "Немного теории",
"Утверждение 2": with A the number of accepted draft tokens, a pass yields A+1
tokens and, A being a non-negative integer, E[A] = sum_{k>=1} P(A >= k), so
tau = 1 + sum_k P(A >= k).  With independent acceptance at a single rate alpha
this is (1 - alpha^(K+1)) / (1 - alpha).

"speculative decoding от черновика до проверки" (braintools.ru), "Сколько это
даёт": the time speedup with a draft pass costing a fraction c of a target pass
is tau / (gamma * c + 1), and the best draft length maximises it.

These are restated from the formulas, not copied; tests pin them to the numbers
the pages print.
"""


def expected_tokens(alpha: float, gamma: int) -> float:
    """tau for i.i.d. acceptance rate alpha and draft length gamma."""
    if alpha == 1.0:
        return float(gamma + 1)
    total, term = 0.0, 1.0
    for _ in range(gamma + 1):  # 1 + alpha + ... + alpha^gamma
        total += term
        term *= alpha
    return total


def tau_from_survival(survival):
    """tau = 1 + sum_k P(A >= k) from a survival profile P(A>=1), P(A>=2), ..."""
    return 1.0 + float(sum(survival))


def speedup(alpha: float, gamma: int, c: float) -> float:
    return expected_tokens(alpha, gamma) / (gamma * c + 1.0)


def best_gamma(alpha: float, c: float, max_gamma: int = 15):
    best = None
    for g in range(1, max_gamma + 1):
        s = speedup(alpha, g, c)
        if best is None or s > best[1]:
            best = (g, s)
    return best


def mean_accept_len(beta):
    """E[a] for a verify length L = len(beta) when position k is accepted
    independently with probability beta[k]: sum_{j=1..L} prod_{k<j} beta[k]."""
    total, prod = 0.0, 1.0
    for b in beta:
        prod *= b
        total += prod
    return total
