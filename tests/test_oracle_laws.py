"""Statistical and exact pins of the oracle's output law (CPU).

  * exact joint law of (n, tokens) by rational enumeration (oracle/brute.py) for V = 3, gamma = 2;
  * beta = sum_x min(p, q) equals the empirical acceptance rate (velog "6-1편. Speculative Decoding" §2-3);
  * losslessness: emitted tokens follow p (velog §2-3 item 3), chi-square over 10^6 trials;
  * E[N] = (1 - alpha^(gamma+1)) / (1 - alpha) and P(N >= k) = alpha^(k-1) (velog §3-1), with the
    printed worked example (velog §3 "예시로 한눈에 보기") from tests/golden;
  * the printed sampling example 0.6 / 0.3 / 0.1 (velog §2-2 "샘플링이란") from tests/golden.
All runs drive the oracle's full logits path (softmax, Philox uniforms, accept scan, inverse CDF).
"""
import json
import os
from fractions import Fraction as F

import numpy as np
import pytest
from scipy.stats import chi2

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run_iid(ps, qs, N, seed=0, step=0):
    """N independent sequences, all with the same per-slot distributions (context-independent rows).

    Logits are log-probabilities in float32 (T = 1); draft tokens are drawn from q_i with numpy.
    Returns (num_accepted[N], tokens[N, gamma+1]).
    """
    g = len(qs)
    V = len(ps[0])
    with np.errstate(divide="ignore"):
        lt = np.log(np.array(ps, dtype=np.float64)).astype(np.float32)
        ld = np.log(np.array(qs, dtype=np.float64)).astype(np.float32) if g else np.zeros((0, V), np.float32)
    target = np.tile(lt, (N, 1))
    draft = np.tile(ld, (N, 1)) if g else None
    rng = np.random.default_rng(seed)
    toks = np.zeros((N, g), dtype=np.int32)
    for i in range(g):
        toks[:, i] = rng.choice(V, size=N, p=np.array(qs[i], dtype=np.float64))
    offs = np.arange(N + 1, dtype=np.int32) * g
    r = oracle.verify(target, draft, toks.reshape(-1), offs, np.full(N, g, np.int32), V, 1.0, seed + 17, step)
    assert r.status == 0
    return r.num_accepted, r.tokens.reshape(N, g + 1)


def chi2_pvalue(counts, probs):
    counts = np.asarray(counts, dtype=np.float64)
    exp = np.asarray(probs, dtype=np.float64) * counts.sum()
    keep = exp > 0
    assert counts[~keep].sum() == 0, "outcome with zero probability observed"
    stat = ((counts[keep] - exp[keep]) ** 2 / exp[keep]).sum()
    return chi2.sf(stat, keep.sum() - 1)


PS = [[F(1, 2), F(1, 3), F(1, 6)], [F(1, 5), F(3, 5), F(1, 5)], [F(1, 10), F(3, 10), F(6, 10)]]
QS = [[F(1, 4), F(1, 2), F(1, 4)], [F(1, 3), F(1, 3), F(1, 3)]]


def test_brute_force_law_is_lossless_and_matches_beta():
    law = brute.joint_law(PS, QS)
    assert sum(law.values()) == 1
    m0, tot0 = brute.marginal_token(law, 0)
    assert tot0 == 1 and all(m0.get(t, 0) == PS[0][t] for t in range(3))       # velog §2-3 item 3
    m1, tot1 = brute.marginal_token(law, 1)
    assert tot1 == brute.beta(PS[0], QS[0])                                     # P(n >= 1) = beta_0
    assert all(m1.get(t, 0) == PS[1][t] for t in range(3))
    m2, tot2 = brute.marginal_token(law, 2)
    assert tot2 == brute.beta(PS[0], QS[0]) * brute.beta(PS[1], QS[1])
    assert all(m2.get(t, 0) == PS[2][t] for t in range(3))
    # p' = (p - min(p, q)) / (1 - beta)  (velog §2-3 item 2)
    b0 = brute.beta(PS[0], QS[0])
    assert brute.residual(PS[0], QS[0]) == [(p - min(p, q)) / (1 - b0) for p, q in zip(PS[0], QS[0])]


@pytest.mark.slow
def test_oracle_joint_law_matches_brute_force():
    law = brute.joint_law(PS, QS)
    keys = sorted(law)
    index = {k: i for i, k in enumerate(keys)}
    N = 1_000_000
    n, toks = run_iid([[float(x) for x in p] for p in PS], [[float(x) for x in q] for q in QS], N, seed=3)
    counts = np.zeros(len(keys))
    for nn, row in zip(n, toks):
        counts[index[(int(nn), tuple(int(t) for t in row[: nn + 1]))]] += 1
    pv = chi2_pvalue(counts, [float(law[k]) for k in keys])
    assert pv > 1e-4, pv


@pytest.mark.slow
def test_beta_equals_empirical_acceptance():
    rng = np.random.default_rng(11)
    for V in (4, 16):
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V))
        beta = np.minimum(p, q).sum()
        N = 1_000_000
        n, _ = run_iid([p, p], [q], N, seed=V)
        rate = (n >= 1).mean()
        assert abs(rate - beta) < 5 * np.sqrt(beta * (1 - beta) / N), (V, rate, beta)


@pytest.mark.slow
@pytest.mark.parametrize("V", [4, 8, 16])
def test_emitted_tokens_follow_p(V):
    rng = np.random.default_rng(100 + V)
    # keep every probability above 1e-3 so each chi-square cell is well populated
    ps = [0.001 + 0.999 * rng.dirichlet(np.ones(V) * 0.7) for _ in range(3)]
    ps = [p / p.sum() for p in ps]
    qs = [0.001 + 0.999 * rng.dirichlet(np.ones(V) * 0.7) for _ in range(2)]
    qs = [q / q.sum() for q in qs]
    N = 1_000_000
    n, toks = run_iid(ps, qs, N, seed=V)
    assert chi2_pvalue(np.bincount(toks[:, 0], minlength=V), ps[0]) > 1e-4
    sel = n >= 1
    assert chi2_pvalue(np.bincount(toks[sel, 1], minlength=V), ps[1]) > 1e-4


@pytest.mark.slow
def test_expected_tokens_matches_worked_example():
    gold = json.load(open(os.path.join(GOLDEN, "velog_worked_example.json")))
    a, g = gold["alpha"], gold["gamma"]
    # p = (0.6, 0.4), q = (0.4, 0.6): sum min(p, q) = 0.8 = alpha at every slot
    ps = [[0.6, 0.4]] * (g + 1)
    qs = [[0.4, 0.6]] * g
    N = 1_000_000
    n, _ = run_iid(ps, qs, N, seed=21)
    emitted = n + 1
    closed = (1 - a ** (g + 1)) / (1 - a)
    assert closed * (1 - a) == pytest.approx(gold["printed_numerator"], abs=5e-5)
    assert abs(closed - gold["printed_E_N"]) <= gold["printed_rounding"]
    se = emitted.std() / np.sqrt(N)
    assert abs(emitted.mean() - closed) < 5 * se, (emitted.mean(), closed)
    assert emitted.max() == gold["printed_table_max_tokens"]
    for k in range(1, g + 2):
        pk = (emitted >= k).mean()
        assert abs(pk - a ** (k - 1)) < 5 * np.sqrt(a ** (k - 1) * (1 - a ** (k - 1)) / N + 1e-12)


@pytest.mark.slow
def test_printed_sampling_example():
    gold = json.load(open(os.path.join(GOLDEN, "velog_sampling_example.json")))
    p = gold["probabilities"]
    N = 1_000_000
    _, toks = run_iid([p], [], N, seed=5)
    freq = np.bincount(toks[:, 0], minlength=3) / N
    np.testing.assert_allclose(freq, gold["printed_frequencies"], atol=5 * np.sqrt(0.25 / N))
    assert chi2_pvalue(np.bincount(toks[:, 0], minlength=3), p) > 1e-4
