"""Pins of the post-verify update oracle (CPU): hand-worked cases, and the link to the verify rule
that the appended tokens before the drawn one are the accepted drafts themselves."""
import numpy as np

import oracle
from oracle.commit import commit, SV_ERR_BAD_OFFSETS, SV_ERR_CAPACITY
from speculative_decoding_verification_35_gb300 import synth


def test_hand_worked_append():
    # one sequence, gamma 3: two drafts accepted (7, 8), token 9 drawn at slot 2, slot 3 unused
    hist = np.array([[5, 6, 0, 0, 0, 0]], np.int32)
    h, lens, nxt, st = commit([7, 8, 9, -1], [2], [0, 3], hist, 6, [2])
    assert h.tolist() == [[5, 6, 7, 8, 9, 0]]
    assert lens.tolist() == [5] and nxt.tolist() == [9] and st == 0
    assert hist.tolist() == [[5, 6, 0, 0, 0, 0]]  # inputs untouched


def test_hand_worked_batch_with_failed_and_full_sequences():
    # b0: gamma 2, n 0 (first draft rejected, 4 drawn); b1: failed (n -1); b2: gamma 1, all accepted
    # (draft 3, bonus 2) but only 1 free slot; b3: gamma 0 (plain sampling), n 0, token 1
    out_tokens = [4, -1, -1, -1, -1, 3, 2, 1]
    offs = [0, 2, 3, 4, 4]
    hist = np.zeros((4, 3), np.int32)
    h, lens, nxt, st = commit(out_tokens, [0, -1, 1, 0], offs, hist, 3, [0, 1, 2, 2])
    assert h[0].tolist() == [4, 0, 0] and lens[0] == 1 and nxt[0] == 4
    assert h[1].tolist() == [0, 0, 0] and lens[1] == 1 and nxt[1] == -1
    assert h[2].tolist() == [0, 0, 0] and lens[2] == 2 and nxt[2] == -1
    assert h[3].tolist() == [0, 0, 1] and lens[3] == 3 and nxt[3] == 1
    assert st == 1 << SV_ERR_CAPACITY


def test_inconsistent_count_is_flagged():
    h, lens, nxt, st = commit([1, 2, 3], [3], [0, 2], np.zeros((1, 8), np.int32), 8, [0])
    assert st == 1 << SV_ERR_BAD_OFFSETS and lens.tolist() == [0] and nxt.tolist() == [-1]


def test_count_above_the_largest_gamma_is_flagged():
    # a gap of 40 slots with n = 35: no verify call reports n above 31, so the outputs are not a verify
    # call's and nothing is appended
    out = list(range(41))
    h, lens, nxt, st = commit(out, [35], [0, 40], np.zeros((1, 64), np.int32), 64, [0])
    assert st == 1 << SV_ERR_BAD_OFFSETS and lens.tolist() == [0] and nxt.tolist() == [-1]
    h, lens, nxt, st = commit(out, [31], [0, 40], np.zeros((1, 64), np.int32), 64, [0])
    assert st == 0 and lens.tolist() == [32] and h[0, :32].tolist() == list(range(32))


def test_appended_tokens_are_the_accepted_drafts():
    # a verify step of the oracle, then the update: the first n appended tokens equal the draft tokens,
    # the last one is the drawn token, and nothing outside the appended range changes
    b = synth.make_batch("ragged_b128_v129280", B=12, V=700)
    r = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V,
                      float(np.float32(b.temperature)), 1234, 3)
    cap = 64
    rng = np.random.default_rng(3)
    lens0 = rng.integers(0, 20, size=b.B).astype(np.int32)
    hist0 = rng.integers(0, b.V, size=(b.B, cap)).astype(np.int32)
    h, lens, nxt, st = commit(r.tokens, r.num_accepted, b.seq_offsets, hist0, cap, lens0)
    assert st == 0
    for s in range(b.B):
        n, L, d0 = int(r.num_accepted[s]), int(lens0[s]), int(b.seq_offsets[s])
        assert lens[s] == L + n + 1
        assert np.array_equal(h[s, L:L + n], b.draft_tokens[d0:d0 + n])
        assert h[s, L + n] == nxt[s] == r.tokens[d0 + s + n]
        assert np.array_equal(h[s, :L], hist0[s, :L]) and np.array_equal(h[s, L + n + 1:], hist0[s, L + n + 1:])
