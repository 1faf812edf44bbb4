"""Oracle of the post-verify update (test infrastructure only; see ``oracle/__init__.py``).

"Accelerating Sonar through speculation", §"MTP scheduling": after verification, a kernel shifts the
target's input tokens and inserts the next target token, so the host does not wait for the accepted
length. Plainest reading, written out: for each sequence with n >= 0 accepted drafts, its n + 1
emitted tokens (the accepted drafts and the drawn token, slots 0..n of the verify output) are appended
to its token history at its current length, the length grows by n + 1, and the drawn token becomes the
next input token. Failed sequences (n < 0) are left as they are, with next token -1; so is a sequence
whose outputs are inconsistent (n above its gamma, or above 31, the largest gamma a verify call takes)
or whose history would overflow, which is flagged.
Plain Python loops: the function is the definition, nothing more.
"""
from __future__ import annotations

import numpy as np

SV_ERR_BAD_OFFSETS, SV_ERR_CAPACITY = 4, 9
MAX_GAMMA = 31  # a verify call takes gamma_b <= 31, so it never reports n above 31


def commit(out_tokens, out_num_accepted, seq_offsets, history, capacity, lengths):
    """Returns (history, lengths, next_tokens, status_bits) after the update; inputs are not modified.

    history is int32[B, capacity]; the rest as spec_verify_commit takes them.
    """
    out_tokens = [int(v) for v in np.asarray(out_tokens).ravel()]
    ns = [int(v) for v in np.asarray(out_num_accepted).ravel()]
    offs = [int(v) for v in np.asarray(seq_offsets).ravel()]
    hist = np.array(history, dtype=np.int32, copy=True).reshape(len(ns), capacity)
    lens = [int(v) for v in np.asarray(lengths).ravel()]
    nxt = [-1] * len(ns)
    status = 0
    for b, n in enumerate(ns):
        if n < 0:
            continue
        gamma = offs[b + 1] - offs[b]
        if n > gamma or n > MAX_GAMMA or offs[b] < 0:
            status |= 1 << SV_ERR_BAD_OFFSETS
            continue
        L = lens[b]
        if L < 0 or L + n + 1 > capacity:
            status |= 1 << SV_ERR_CAPACITY
            continue
        t0 = offs[b] + b
        for j in range(n + 1):
            hist[b, L + j] = out_tokens[t0 + j]
        lens[b] = L + n + 1
        nxt[b] = out_tokens[t0 + n]
    return hist, np.array(lens, dtype=np.int32), np.array(nxt, dtype=np.int32), status
