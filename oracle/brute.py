"""Exact joint output law of one verify step by rational enumeration (test infrastructure only).

For context-independent rows (each slot i has its own fixed target distribution p_i and draft
distribution q_i, and the draft token x_i is drawn from q_i), the law of the verify step's output is a
finite sum over the drafted tokens and the accept/reject branch at each slot. This module writes that
sum out with ``fractions.Fraction``: no floating point, no sampling. It follows the 4-step algorithm and
rules of the velog article "6-1편. Speculative Decoding":
  §2 step 3 / §2-1: slot i's draft x is accepted with probability min(1, p_i(x)/q_i(x));
  §2 step 4 / §2-2: the first rejected slot draws from p'_i = norm(max(0, p_i - q_i)); when all gamma
                    drafts are accepted, one bonus token is drawn from p_gamma;
  §2-3: beta_i = sum_x min(p_i(x), q_i(x)) is the acceptance probability and the emitted token's law is
        p_i (losslessness), which tests check on the enumeration's marginals.
"""
from __future__ import annotations

import itertools
from fractions import Fraction


def residual(p, q):
    """p' = norm(max(0, p - q)) ([velog] §2-2); falls back to p when the residual mass is 0."""
    w = [max(Fraction(0), pk - qk) for pk, qk in zip(p, q)]
    s = sum(w)
    if s == 0:
        return list(p)
    return [wk / s for wk in w]


def beta(p, q):
    """beta = sum_x min(p(x), q(x)) ([velog] §2-3 item 1)."""
    return sum(min(pk, qk) for pk, qk in zip(p, q))


def joint_law(ps, qs):
    """Exact law of (n, emitted tokens) for one sequence.

    ps: gamma + 1 target distributions (lists of Fractions), qs: gamma draft distributions.
    Returns {(n, (t_0, ..., t_n)): probability} where n is the number of accepted drafts and
    t_0..t_n the n + 1 emitted tokens.
    """
    gamma = len(qs)
    V = len(ps[0])
    law: dict = {}
    for xs in itertools.product(range(V), repeat=gamma):
        px = Fraction(1)
        for i, x in enumerate(xs):
            px *= qs[i][x]
        if px == 0:
            continue
        # walk the slots: reach slot i with probability `reach` having accepted xs[:i]
        reach = px
        for i in range(gamma + 1):
            if i == gamma:  # bonus draw from p_gamma
                for t, pt in enumerate(ps[gamma]):
                    if pt:
                        key = (gamma, tuple(xs) + (t,))
                        law[key] = law.get(key, Fraction(0)) + reach * pt
                break
            x = xs[i]
            q_x, p_x = qs[i][x], ps[i][x]
            acc = Fraction(1) if q_x <= p_x else p_x / q_x
            rej = 1 - acc
            if rej:
                for t, r in enumerate(residual(ps[i], qs[i])):
                    if r:
                        key = (i, tuple(xs[:i]) + (t,))
                        law[key] = law.get(key, Fraction(0)) + reach * rej * r
            reach *= acc
            if reach == 0:
                break
    return law


def marginal_token(law, position):
    """Law of the token emitted at ``position`` conditional on at least position + 1 tokens."""
    num: dict = {}
    tot = Fraction(0)
    for (n, toks), pr in law.items():
        if n >= position:
            num[toks[position]] = num.get(toks[position], Fraction(0)) + pr
            tot += pr
    return {t: v / tot for t, v in num.items()}, tot
