"""Oracle of the n-gram drafter (test infrastructure only; see ``oracle/__init__.py``).

velog "6-1편. Speculative Decoding", §"drafter types", N-gram: no draft model; look for the most recent n
consecutive tokens at an earlier place of the context and reuse the tokens that followed as the guess.
Plainest reading, written out in plain loops: for n from n_max down to n_min, the most recent earlier
occurrence (largest start s with s + n < L) of the last n tokens; the draft is up to gamma_max of the
tokens that followed it, within the history. No match: no draft.
"""
from __future__ import annotations

import numpy as np


def draft(history, lengths, n_min, n_max, gamma_max):
    """Returns (draft_tokens packed, gammas, seq_offsets, match_pos) for int32 history [B, capacity]."""
    hist = np.asarray(history)
    B, cap = hist.shape
    gammas = np.zeros(B, np.int32)
    pos = np.zeros(B, np.int32)
    drafts = []
    for b in range(B):
        L = int(lengths[b])
        if L < 0 or L > cap:
            pos[b] = 0 if L < 0 else cap
            drafts.append([])
            continue
        h = [int(v) for v in hist[b, :L]]
        g, p = 0, L
        for n in range(n_max, n_min - 1, -1):
            if gamma_max == 0 or L < n + 1:
                continue
            pattern = h[L - n:]
            for s in range(L - n - 1, -1, -1):  # most recent first
                if h[s:s + n] == pattern:
                    p = s + n
                    g = min(gamma_max, L - p)
                    break
            if g:
                break
        gammas[b], pos[b] = g, p
        drafts.append(h[p:p + g])
    offs = np.concatenate([[0], np.cumsum(gammas)]).astype(np.int32)
    flat = np.array([t for d in drafts for t in d], dtype=np.int32)
    return flat, gammas, offs, pos
