"""Pins of the oracle's draw bracket, its beta output and its multi-step entry (CPU).

``oracle_draw_bracket`` decides, in the GPU parity tests, whether a GPU/oracle disagreement lies inside
the 1e-6 decision band; it is pinned here by hand-worked brackets on V <= 5 (velog "6-1편. Speculative
Decoding", §2-2: the draw is "in proportion" to the corrected distribution p' = norm(max(0, p - q)), read
as an inverse CDF in vocabulary index order), for bonus, residual and point-mass-excluded draws, with the
queried token both the drawn one and another one.

beta_i = sum_x min(p_i(x), q_i(x)) (velog §2-3) is pinned by the printed hand case (beta = 0.7 for
p = (0.6, 0.3, 0.1), q = (0.3, 0.5, 0.2)), by 1 - beta = sum max(0, p - q) (the residual mass, §2-3
item 2), by beta = p(x) for a point-mass draft, and by the empirical acceptance rate.

``oracle_verify_steps`` is pinned to repeated calls of ``oracle_verify`` (step by step, bit for bit).
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_35_gb300 import synth


def logits_of(p):
    """float32 logits whose softmax at T = 1 is p (up to the float32 rounding of log p); -inf for p = 0."""
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, dtype=np.float64)).astype(np.float32)


def bracket(p, q, k, u=0.5, x_excl=-1):
    trow = logits_of(p)
    drow = None if q is None else logits_of(q)
    return oracle.draw_bracket(trow, drow, len(p), 1.0, u, k, x_excl)


TOL = 1e-6  # float32 rounding of the logits moves every probability by about 1e-7 relative


def test_bonus_brackets_are_the_running_sums_of_p():
    p = [0.1, 0.2, 0.3, 0.4]
    C = [0.0, 0.1, 0.3, 0.6, 1.0]
    for k in range(4):
        tok, lo, hi, S = bracket(p, None, k, u=0.35)
        assert tok == 2  # 0.3 <= 0.35 < 0.6
        assert lo == pytest.approx(C[k], abs=TOL) and hi == pytest.approx(C[k + 1], abs=TOL)
        assert S == pytest.approx(1.0, abs=1e-12)
    for u, want in [(0.0, 0), (0.0999, 0), (0.1001, 1), (0.5999, 2), (0.6001, 3), (1 - 2 ** -24, 3)]:
        assert bracket(p, None, 0, u=u)[0] == want


def test_residual_brackets_follow_norm_max_p_minus_q():
    # p - q = (0.3, -0.2, 0.2, -0.3): p' = (0.6, 0, 0.4, 0), S = 0.5
    p = [0.4, 0.1, 0.3, 0.2]
    q = [0.1, 0.3, 0.1, 0.5]
    want = [(0.0, 0.6), (0.6, 0.6), (0.6, 1.0), (1.0, 1.0)]
    for k in range(4):
        tok, lo, hi, S = bracket(p, q, k, u=0.7)
        assert tok == 2  # the query token need not be the drawn one
        assert (lo, hi) == (pytest.approx(want[k][0], abs=TOL), pytest.approx(want[k][1], abs=TOL))
        assert S == pytest.approx(0.5, abs=TOL)
    assert bracket(p, q, 0, u=0.59)[0] == 0 and bracket(p, q, 0, u=0.61)[0] == 2
    # the velog §2-2 case: p' = norm(max(0, (0.3, -0.2, -0.1))) = (1, 0, 0): every draw is token 0
    for u in [0.0, 0.5, 0.99]:
        tok, lo, hi, S = bracket([0.6, 0.3, 0.1], [0.3, 0.5, 0.2], 0, u=u)
        assert tok == 0 and lo == pytest.approx(0.0, abs=TOL) and hi == pytest.approx(1.0, abs=TOL)
        assert S == pytest.approx(0.3, abs=TOL)


def test_point_mass_residual_removes_the_draft_token():
    # q = point mass at x = 2: max(0, p - q) = p without token 2, S = 0.7
    p = [0.1, 0.2, 0.3, 0.4]
    want = [(0.0, 1 / 7), (1 / 7, 3 / 7), (3 / 7, 3 / 7), (3 / 7, 1.0)]
    for k in range(4):
        tok, lo, hi, S = bracket(p, None, k, u=0.2, x_excl=2)
        assert tok == 1 and S == pytest.approx(0.7, abs=TOL)
        assert (lo, hi) == (pytest.approx(want[k][0], abs=TOL), pytest.approx(want[k][1], abs=TOL))
    for u in np.linspace(0, 1 - 1e-9, 101):
        assert bracket(p, None, 0, u=u, x_excl=2)[0] != 2  # a removed token is never drawn


def test_zero_residual_falls_back_to_p():
    p = [0.25, 0.25, 0.5]
    tok, lo, hi, S = bracket(p, p, 2, u=0.6)
    assert tok == 2 and lo == pytest.approx(0.5, abs=TOL) and hi == pytest.approx(1.0, abs=TOL)
    assert S == pytest.approx(1.0, abs=TOL)


@pytest.mark.parametrize("V", [2, 3, 5])
def test_brackets_tile_the_unit_interval_and_contain_the_draw(V):
    rng = np.random.default_rng(V)
    for trial in range(50):
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V)) if trial % 3 else None
        xe = int(rng.integers(0, V)) if trial % 3 == 0 and trial % 2 else -1
        u = float(rng.random())
        br = [bracket(p, q, k, u=u, x_excl=xe) for k in range(V)]
        assert br[0][1] == 0.0 and br[-1][2] == pytest.approx(1.0, abs=1e-12)
        for k in range(V - 1):
            assert br[k][2] == br[k + 1][1]  # C_k / S is both the upper end of k and the lower end of k + 1
        tok = br[0][0]
        assert all(b[0] == tok for b in br)
        assert br[tok][1] <= u < br[tok][2]


def test_beta_hand_case_and_residual_mass():
    # velog §2-3: beta = 0.3 + 0.3 + 0.1 = 0.7 for the printed p and q
    p, q = [0.6, 0.3, 0.1], [0.3, 0.5, 0.2]
    target = np.stack([logits_of(p), logits_of(p)])
    draft = logits_of(q)[None]
    for x in range(3):
        r = oracle.verify(target, draft, [x], [0, 1], [1], 3, 1.0, 1, 0)
        assert r.beta[0] == pytest.approx(0.7, abs=TOL)
    rng = np.random.default_rng(4)
    for _ in range(20):
        V = int(rng.integers(2, 40))
        lt = rng.normal(0, 2, size=(2, V)).astype(np.float32)
        ld = rng.normal(0, 2, size=(1, V)).astype(np.float32)
        T = float(np.float32(rng.uniform(0.3, 2.0)))
        pe = np.exp(lt[0].astype(np.float64) / T); pe /= pe.sum()
        qe = np.exp(ld[0].astype(np.float64) / T); qe /= qe.sum()
        r = oracle.verify(lt, ld, [0], [0, 1], [1], V, T, 2, 0)
        assert r.beta[0] == pytest.approx(np.minimum(pe, qe).sum(), rel=1e-12)
        assert 1.0 - r.beta[0] == pytest.approx(np.maximum(pe - qe, 0).sum(), abs=1e-12)  # §2-3 item 2
        if r.num_accepted[0] == 0:  # rejected: the draw's normaliser is the residual mass 1 - beta
            assert r.seq_mass[0] == pytest.approx(1.0 - r.beta[0], abs=1e-12)


def test_beta_of_a_point_mass_draft_is_p_of_x():
    b = synth.make_batch("pointmass_b64_g5_v128256", B=3, V=500)
    r = oracle.verify(b.target, None, b.draft_tokens, b.seq_offsets, b.gammas, b.V, 1.0, 1, 0)
    assert np.allclose(r.beta, r.p_x, rtol=0, atol=0)


def test_beta_equals_the_acceptance_rate():
    # slot 0 accepted with probability beta when x ~ q (velog §2-3): 2e5 trials on V = 8
    rng = np.random.default_rng(11)
    V, N = 8, 200_000
    lt = rng.normal(0, 1, size=V).astype(np.float32)
    ld = rng.normal(0, 1, size=V).astype(np.float32)
    qe = np.exp(ld.astype(np.float64)); qe /= qe.sum()
    x = rng.choice(V, size=N, p=qe).astype(np.int32)
    target = np.tile(np.stack([lt, lt]), (N, 1))
    draft = np.tile(ld[None], (N, 1))
    offs = np.arange(N + 1, dtype=np.int32)
    r = oracle.verify(target, draft, x, offs, np.ones(N, np.int32), V, 1.0, 3, 0)
    beta = r.beta[0]
    assert np.allclose(r.beta, beta)
    rate = (r.num_accepted == 1).mean()
    assert abs(rate - beta) < 5 * np.sqrt(beta * (1 - beta) / N)


@pytest.mark.parametrize("name,B,V", [("b64_g5_v128256", 7, 3001), ("ragged_b128_v129280", 9, 2048),
                                      ("pointmass_b64_g5_v128256", 5, 999), ("b1_g4_v1024_f32", 1, 1024)])
def test_verify_steps_equals_one_call_per_step(name, B, V):
    b = synth.make_batch(name, B=B, V=V)
    toks, ns, st = oracle.verify_steps(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V,
                                       b.temperature, 77, 1000, 9)
    assert st == 0
    for s in range(9):
        r = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, b.temperature, 77,
                          1000 + s)
        assert np.array_equal(r.tokens, toks[s]) and np.array_equal(r.num_accepted, ns[s])


def test_verify_steps_reports_errors_like_verify():
    b = synth.make_batch("b8_g4_v32000_t0.7", B=4, V=300)
    b.draft_tokens[5] = 300  # sequence 1: bad token
    toks, ns, st = oracle.verify_steps(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, 0.7,
                                       1, 0, 3)
    r = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, 0.7, 1, 2)
    assert st == r.status == 1 << 3
    assert np.array_equal(ns[2], r.num_accepted) and np.array_equal(toks[2], r.tokens)
    assert np.all(ns[:, 1] == -1)
