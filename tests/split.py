"""Contiguous sequence ranges of a CSR batch (multi-GPU by sequence): the sub-batch of sequences [s0, s1)
and the concatenation of the ranges' outputs."""
import numpy as np

from speculative_decoding_verification_35_gb300 import synth


def sub_batch(b, s0, s1):
    """Sequences [s0, s1) of batch b as a batch of their own (rows, tokens and offsets rebased)."""
    o = b.seq_offsets
    d0, d1 = int(o[s0]), int(o[s1])
    offs = (o[s0:s1 + 1] - d0).astype(np.int32)
    draft = None if b.draft is None else b.draft[d0:d1]
    return synth.Batch(b.workload, b.target[d0 + s0:d1 + s1], draft, b.draft_tokens[d0:d1].copy(), offs,
                       b.gammas[s0:s1].copy())


def ranges(B, parts):
    """`parts` contiguous ranges of nearly equal size covering 0 .. B."""
    cut = [B * j // parts for j in range(parts + 1)]
    return [(cut[j], cut[j + 1]) for j in range(parts) if cut[j + 1] > cut[j]]


def concat(outs):
    """Concatenate (tokens, n) of consecutive ranges."""
    return np.concatenate([t for t, _ in outs]), np.concatenate([n for _, n in outs])
