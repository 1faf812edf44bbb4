"""Pins of the n-gram drafter oracle (CPU): hand-worked histories, and agreement with a second,
string-search formulation of the same rule on random histories."""
import numpy as np

from oracle.ngram import draft


def _one(h, n_min, n_max, gmax, cap=16):
    hist = np.zeros((1, cap), np.int32)
    hist[0, :len(h)] = h
    toks, g, offs, pos = draft(hist, [len(h)], n_min, n_max, gmax)
    return toks.tolist(), int(g[0]), int(pos[0])


def test_hand_worked_histories():
    # "5 6 7 8 5 6": the last bigram (5, 6) occurred at 0; the tokens after it are 7 8 5 6
    assert _one([5, 6, 7, 8, 5, 6], 2, 2, 3) == ([7, 8, 5], 3, 2)
    # the most recent earlier occurrence wins: (1, 2) at 0 and at 3; 8 1 2 follow the one at 3
    assert _one([1, 2, 9, 1, 2, 8, 1, 2], 2, 2, 5) == ([8, 1, 2], 3, 5)
    # n = 3 finds nothing (9 1 2 is new), n = 2 does
    assert _one([1, 2, 7, 9, 1, 2], 2, 3, 4) == ([7, 9, 1, 2], 4, 2)
    # a run: the last 4 follows an earlier 4; only one token is left after the latest earlier start
    assert _one([4, 4, 4, 4], 1, 1, 5) == ([4], 1, 3)
    # no earlier occurrence, too short a history, an empty one
    assert _one([1, 2, 3, 4], 1, 2, 5) == ([], 0, 4)
    assert _one([7], 1, 1, 5) == ([], 0, 1)
    assert _one([], 1, 3, 5) == ([], 0, 0)
    # gamma_max 0: no draft
    assert _one([5, 6, 5, 6], 1, 2, 0) == ([], 0, 4)


def test_csr_packing():
    hist = np.zeros((3, 8), np.int32)
    hist[0, :4] = [1, 2, 1, 2]   # bigram (1, 2) at 0 -> 1 2 (2 left)
    hist[1, :3] = [3, 4, 5]      # none
    hist[2, :5] = [6, 6, 6, 6, 6]  # unigram 6 at 3 -> 6
    toks, g, offs, pos = draft(hist, [4, 3, 5], 1, 2, 3)
    assert g.tolist() == [2, 0, 1] and offs.tolist() == [0, 2, 2, 3] and toks.tolist() == [1, 2, 6]
    assert pos.tolist() == [2, 3, 4]


def _by_string_search(h, n_min, n_max, gmax):
    """The same rule through str.rfind on a token string with separators (a different formulation)."""
    L = len(h)
    enc = "".join(f",{t}" for t in h) + ","
    for n in range(n_max, n_min - 1, -1):
        if gmax == 0 or L < n + 1:
            continue
        pat = "".join(f",{t}" for t in h[L - n:]) + ","
        # occurrences must end before the last token: search the prefix holding tokens 0 .. L-2
        pre = "".join(f",{t}" for t in h[:L - 1]) + ","
        i = pre.rfind(pat)
        if i >= 0:
            s = pre[:i].count(",")  # separators before the match = its token index
            p = s + n
            g = min(gmax, L - p)
            return h[p:p + g], g, p
    return [], 0, L


def test_agrees_with_string_search_on_random_histories():
    rng = np.random.default_rng(5)
    for trial in range(300):
        L = int(rng.integers(0, 40))
        h = rng.integers(0, 4, size=L).tolist()  # a small alphabet: many repeats
        n_min = int(rng.integers(1, 4))
        n_max = n_min + int(rng.integers(0, 3))
        gmax = int(rng.integers(0, 7))
        assert _one(h, n_min, n_max, gmax, cap=40) == tuple(_by_string_search(h, n_min, n_max, gmax)), (h, n_min, n_max, gmax)
