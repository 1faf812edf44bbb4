"""Pins of the oracle's point-mass draft mode (drafts without a draft distribution, as an n-gram
drafter gives them: velog "6-1편. Speculative Decoding", §"drafter types", N-gram).

q_i is the point mass at x_i, so the rule of §2-1 accepts with probability min(1, p(x)/1) = p(x), and
the residual of §2-2 is max(0, p - q): p with x removed, renormalised. Pinned by hand-worked values and
by exact equality with the general path given draft logits that are 0 at x and -inf elsewhere (whose
softmax is exactly the point mass)."""
import numpy as np

import oracle
from speculative_decoding_verification_35_gb300 import synth


def test_hand_worked_point_mass():
    # [velog] §2-2 example p = (0.6, 0.3, 0.1); draft x = 1 with q = delta_1: accepted iff u < 0.3;
    # on rejection the token is drawn from (0.6, 0, 0.1) / 0.7
    p = np.array([[0.6, 0.3, 0.1], [0.2, 0.5, 0.3]])
    q = np.array([[0.0, 1.0, 0.0]])
    n, out, S, fb = oracle.verify_probs(p, q, [1], [0.29], [0.0, 0.0])
    assert n == 1 and out[0] == 1                       # u = 0.29 < p(x) = 0.3: accepted
    n, out, S, fb = oracle.verify_probs(p, q, [1], [0.31], [0.85, 0.0])
    assert n == 0 and abs(S - 0.7) < 1e-15 and not fb    # rejected: residual mass 1 - p(x)
    assert out[0] == 0                                   # u' S = 0.595 < 0.6
    n, out, S, fb = oracle.verify_probs(p, q, [1], [0.31], [0.86, 0.0])
    assert out[0] == 2                                   # u' S = 0.602 > 0.6: past token 0, token 1 has 0


def _onehot_logits(b):
    """Draft logits whose softmax is exactly the point mass at each draft token."""
    dt = np.full((b.R_d, b.V), -np.inf, dtype=np.float32)
    dt[np.arange(b.R_d), b.draft_tokens] = 0.0
    if b.target.dtype == np.uint16:  # raw bf16 bits: -inf is 0xFF80, 0.0 is 0
        bits = np.full((b.R_d, b.V), 0xFF80, dtype=np.uint16)
        bits[np.arange(b.R_d), b.draft_tokens] = 0
        return bits
    return dt


def test_point_mass_mode_equals_materialised_one_hot_logits():
    for name, B, V in [("ragged_b128_v129280", 16, 2000), ("b1_g4_v1024_f32", 1, 1024), ("b8_g4_v32000_t0.7", 8, 5000)]:
        b = synth.make_batch(name, B=B, V=V)
        T = float(np.float32(b.temperature))
        for step in range(4):
            r0 = oracle.verify(b.target, None, b.draft_tokens, b.seq_offsets, b.gammas, b.V, T, 77, step)
            r1 = oracle.verify(b.target, _onehot_logits(b), b.draft_tokens, b.seq_offsets, b.gammas, b.V, T, 77, step)
            assert r0.status == r1.status == 0
            assert np.array_equal(r0.num_accepted, r1.num_accepted) and np.array_equal(r0.tokens, r1.tokens)
            np.testing.assert_allclose(r0.p_x, r1.p_x, rtol=1e-15)
            assert np.all(r0.q_x == 1.0) and np.allclose(r1.q_x, 1.0)
            np.testing.assert_allclose(r0.seq_mass, r1.seq_mass, rtol=1e-13)


def test_point_mass_acceptance_rate_is_p_of_x():
    # 10^5 sequences, V = 6: slot 0 accepted with probability p(x); the residual draw ~ p without x
    V, N = 6, 100_000
    rng = np.random.default_rng(11)
    p = rng.dirichlet(np.ones(V)) * 0.98 + 0.02 / V
    lt = np.log(p).astype(np.float32)
    target = np.tile(np.stack([lt, lt]), (N, 1))
    x = np.full(N, 2, np.int32)
    offs = np.arange(N + 1, dtype=np.int32)
    r = oracle.verify(target, None, x, offs, np.ones(N, np.int32), V, 1.0, 5, 0)
    pe = np.exp(lt.astype(np.float64)); pe /= pe.sum()
    rate = (r.num_accepted == 1).mean()
    assert abs(rate - pe[2]) < 5 * np.sqrt(pe[2] * (1 - pe[2]) / N)
    rej = r.tokens[0::2][r.num_accepted == 0]
    assert not np.any(rej == 2)
    w = pe.copy(); w[2] = 0; w /= w.sum()
    cnt = np.bincount(rej, minlength=V)
    from scipy.stats import chi2
    m = w > 0
    stat = ((cnt[m] - w[m] * len(rej)) ** 2 / (w[m] * len(rej))).sum()
    assert chi2.sf(stat, m.sum() - 1) > 1e-4
