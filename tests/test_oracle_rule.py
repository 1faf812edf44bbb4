"""Pins of the oracle's accept rule, residual, greedy path, softmax and error handling (CPU).

Hand-worked cases follow the velog article "6-1편. Speculative Decoding":
  §2-1: q(x) <= p(x) is always accepted; otherwise accepted with probability p(x)/q(x).
  §2-2: the rejected slot draws from p' = norm(max(0, p - q)).
  §2-3: beta = sum_x min(p, q).
The greedy path follows "All About Transformer Inference", Appendix D steps 1-3.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_35_gb300 import synth

P = np.array([0.6, 0.3, 0.1])
Q = np.array([0.3, 0.5, 0.2])


def one_slot(x, u_acc, u_smp, p=P, q=Q, p_bonus=None):
    pb = P if p_bonus is None else p_bonus
    return oracle.verify_probs(np.stack([p, pb]), q[None], [x], [u_acc], [u_smp, 0.5])


def test_hand_case_q_le_p_always_accepted():
    # x = 0: q(0) = 0.3 <= p(0) = 0.6 -> accepted for every u (velog §2-1 case 1)
    for u in [0.0, 0.5, 0.999999]:
        n, out, _, _ = one_slot(0, u, 0.1)
        assert n == 1 and out[0] == 0


def test_hand_case_accept_probability_is_p_over_q():
    # x = 1: p/q = 0.6; x = 2: p/q = 0.5 (velog §2-1 case 2)
    assert one_slot(1, 0.5999, 0.1)[0] == 1
    assert one_slot(1, 0.6001, 0.1)[0] == 0
    assert one_slot(2, 0.4999, 0.1)[0] == 1
    assert one_slot(2, 0.5001, 0.1)[0] == 0


def test_hand_case_residual_is_norm_max_p_minus_q():
    # p' = norm(max(0, (0.3, -0.2, -0.1))) = (1, 0, 0): any rejected draw emits token 0 (velog §2-2)
    for us in [0.0, 0.3, 0.9999]:
        n, out, S, fb = one_slot(1, 0.9, us)
        assert n == 0 and out[0] == 0 and out[1] == -1 and not fb
        assert S == pytest.approx(0.3, abs=1e-15)          # 1 - beta
    assert np.minimum(P, Q).sum() == pytest.approx(0.7)    # beta (velog §2-3)


def test_identical_distributions_accept_every_draft():
    rng = np.random.default_rng(0)
    p = rng.dirichlet(np.ones(16), size=6)
    for t in range(200):
        x = rng.integers(0, 16, size=5)
        n, out, _, _ = oracle.verify_probs(p, p[:5], x, rng.random(5), rng.random(6))
        assert n == 5 and np.array_equal(out[:5], x)


def test_disjoint_supports_reject_at_slot0_and_draw_from_p():
    p = np.array([0.5, 0.5, 0.0, 0.0])
    q = np.array([0.0, 0.0, 0.25, 0.75])
    for u in [0.0, 0.4, 0.6, 0.99]:
        n, out, S, _ = oracle.verify_probs(np.stack([p, p]), q[None], [3], [0.0], [u, 0.0])
        assert n == 0 and out[0] == (0 if u < 0.5 else 1) and S == 1.0   # beta = 0, p' = p


def test_zero_draft_probability_accepts_and_zero_both_rejects():
    p = np.array([0.5, 0.5, 0.0])
    q = np.array([0.0, 0.5, 0.5])
    assert oracle.verify_probs(np.stack([p, p]), q[None], [0], [0.99], [0.1, 0.1])[0] == 1
    # x = 2 has p = 0 < q -> always rejected
    n, out, _, _ = oracle.verify_probs(np.stack([p, p]), q[None], [2], [0.0], [0.1, 0.1])
    assert n == 0 and out[0] == 0


def test_inverse_cdf_is_index_ordered_and_strict():
    p = np.array([0.25, 0.25, 0.25, 0.25])
    # u * S exactly on a boundary goes to the next token (C_k > u S strictly)
    assert oracle.verify_probs(p[None], np.zeros((0, 4)), [], [], [0.25])[1][0] == 1
    assert oracle.verify_probs(p[None], np.zeros((0, 4)), [], [], [0.2499])[1][0] == 0
    assert oracle.verify_probs(p[None], np.zeros((0, 4)), [], [], [0.0])[1][0] == 0
    # zero-weight tokens are never drawn, even at the boundaries around them
    p2 = np.array([0.5, 0.0, 0.0, 0.5])
    assert oracle.verify_probs(p2[None], np.zeros((0, 4)), [], [], [0.5])[1][0] == 3


def test_inverse_cdf_tail_rule_last_positive_weight():
    # parity unpinned convention: no crossing through rounding -> last k with w_k > 0
    p = np.array([0.1, 0.2, 0.3, 0.4 - 1e-12, 0.0])
    tok = oracle.verify_probs(p[None], np.zeros((0, 5)), [], [], [1.0])[1][0]
    assert tok == 3


def test_bonus_when_all_accepted_and_gamma_zero():
    rng = np.random.default_rng(1)
    p = rng.dirichlet(np.ones(8), size=1)
    n, out, S, _ = oracle.verify_probs(p, np.zeros((0, 8)), [], [], [0.3])
    c = np.cumsum(p[0])
    assert n == 0 and out[0] == int(np.argmax(c > 0.3 * c[-1]))


def _logits_batch(B, g, V, seed=0, dtype="f32"):
    rng = np.random.default_rng(seed)
    t = rng.normal(0, 2, size=((g + 1) * B, V)).astype(np.float32)
    d = (t[: g * B] + rng.normal(0, 1, size=(g * B, V))).astype(np.float32)
    offs = np.arange(B + 1, dtype=np.int32) * g
    toks = rng.integers(0, V, size=g * B).astype(np.int32)
    return t, d, toks, offs, np.full(B, g, np.int32)


@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_softmax_lse_matches_torch_log_softmax(T):
    t, d, toks, offs, gam = _logits_batch(4, 3, 257, seed=3)
    r = oracle.verify(t, d, toks, offs, gam, 257, T, 1, 0)
    assert r.status == 0
    # target rows of sequence b sit at offs[b] + b ..; draft rows at offs[b] ..
    tt = torch.from_numpy(t).double() / T
    dd = torch.from_numpy(d).double() / T
    lse_t = torch.logsumexp(tt, dim=1).numpy()
    lse_d = torch.logsumexp(dd, dim=1).numpy()
    np.testing.assert_allclose(r.row_lse[: len(t)], lse_t, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r.row_lse[len(t):], lse_d, rtol=1e-12, atol=1e-12)
    ls_t = torch.log_softmax(tt, dim=1).exp().numpy()
    ls_d = torch.log_softmax(dd, dim=1).exp().numpy()
    for b in range(4):
        for i in range(3):
            x = toks[offs[b] + i]
            assert r.p_x[offs[b] + i] == pytest.approx(ls_t[offs[b] + b + i, x], rel=1e-12)
            assert r.q_x[offs[b] + i] == pytest.approx(ls_d[offs[b] + i, x], rel=1e-12)


def test_bf16_logits_read_exactly():
    b = synth.make_batch("b8_g4_v32000_t0.7", B=2, V=300)
    r = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V,
                      b.temperature, 1234, 0)
    lse = torch.logsumexp(torch.from_numpy(b.logits_f32("target")).double() / 0.7, 1).numpy()
    np.testing.assert_allclose(r.row_lse[: b.R_t], lse, rtol=1e-12)


def test_greedy_matches_torch_argmax_and_appendix_d_rule():
    rng = np.random.default_rng(5)
    B, g, V = 50, 4, 40
    # coarse integer logits -> many ties, exercising the lowest-index rule
    t = rng.integers(-3, 4, size=((g + 1) * B, V)).astype(np.float32)
    offs = np.arange(B + 1, dtype=np.int32) * g
    am = torch.argmax(torch.from_numpy(t), dim=1).numpy()  # first maximal index
    toks = np.where(rng.random(g * B) < 0.7, am[np.arange(g * B) + np.repeat(np.arange(B), g)],
                    rng.integers(0, V, size=g * B)).astype(np.int32)
    r = oracle.verify(t, None, toks, offs, np.full(B, g, np.int32), V, 0.0, 1, 0)
    assert r.status == 0
    np.testing.assert_array_equal(r.row_argmax, am)
    for b in range(B):
        d0, t0 = offs[b], offs[b] + b
        n = next((i for i in range(g) if toks[d0 + i] != am[t0 + i]), g)
        assert r.num_accepted[b] == n
        exp = [int(toks[d0 + i]) for i in range(n)] + [int(am[t0 + n])] + [-1] * (g - n)
        assert list(r.tokens[t0: t0 + g + 1]) == exp


def test_error_paths():
    t, d, toks, offs, gam = _logits_batch(3, 2, 16, seed=9)
    bad = toks.copy(); bad[2] = 16
    r = oracle.verify(t, d, bad, offs, gam, 16, 1.0, 1, 0)
    assert r.status == 1 << 3 and r.num_accepted[1] == -1 and r.num_accepted[0] >= 0
    assert list(r.tokens[3:6]) == [-1, -1, -1]
    tn = t.copy(); tn[0, 5] = np.nan
    assert oracle.verify(tn, d, toks, offs, gam, 16, 1.0, 1, 0).status == 1 << 5
    ti = t.copy(); ti[4, :] = -np.inf
    r = oracle.verify(ti, d, toks, offs, gam, 16, 1.0, 1, 0)
    assert r.status == 1 << 6 and r.num_accepted[1] == -1
    tinf = t.copy(); tinf[0, :3] = -np.inf  # partial -inf is allowed: p = 0 there
    assert oracle.verify(tinf, d, toks, offs, gam, 16, 1.0, 1, 0).status == 0
    assert oracle.verify(t, d, toks, np.array([0, 2, 3, 6], np.int32), gam, 16, 1.0, 1, 0).status == 1 << 4
    assert oracle.verify(t, d, toks, offs, gam, 16, -1.0, 1, 0).status == 1 << 1
    assert oracle.verify(t, d, toks, offs, gam, 16, float("nan"), 1, 0).status == 1 << 1


def test_deterministic_and_thread_count_independent():
    b = synth.make_batch("ragged_b128_v129280", B=20, V=500)
    r1 = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, 1.0, 7, 3, nthreads=1)
    r2 = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, 1.0, 7, 3, nthreads=5)
    np.testing.assert_array_equal(r1.tokens, r2.tokens)
    np.testing.assert_array_equal(r1.num_accepted, r2.num_accepted)


def test_a_sequences_outputs_depend_only_on_its_own_rows():
    """A sequence's outputs depend only on its own rows (with the same uniforms): zeroing another
    sequence's target rows leaves every other sequence's outputs unchanged."""
    b = synth.make_batch("ragged_b128_v129280", B=12, V=300)
    full = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, 1.0, 11, 2)
    assert full.status == 0
    # the oracle has no shard API: checking sequence b alone means slicing its rows, which renumbers it
    # to 0 -- so compare per-sequence results only where the uniform does not depend on b: instead check
    # that the tokens emitted for b depend only on b's rows by perturbing another sequence
    t2 = b.target.copy(); t2[: b.gammas[0] + 1] = synth.to_bf16_bits(np.zeros((b.gammas[0] + 1, b.V)))
    r2 = oracle.verify(t2, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, 1.0, 11, 2)
    np.testing.assert_array_equal(r2.num_accepted[1:], full.num_accepted[1:])
    np.testing.assert_array_equal(r2.tokens[b.gammas[0] + 1:], full.tokens[b.gammas[0] + 1:])
