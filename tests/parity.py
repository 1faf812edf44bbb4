"""Helpers of the GPU parity tests: upload a synthetic batch, run the C ABI, compare with the oracle.

Comparison rule (tolerances of the verify step's contract): accepted counts and token ids must equal
the oracle's exactly, except on a draw whose uniform lies within 1e-6 of the oracle's decision boundary
(accept step: |u - p(x)/q(x)| < 1e-6; draw: u within 1e-6 of the oracle CDF bracket of the GPU's token).
Such band draws are counted; their number must stay below 1e-5 of the draws. Intermediates (row
log-normalisers, p(x_i), q(x_i), the draw's mass S) must agree within 1e-5 relative.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

BAND = 1e-6
REL = 1e-5


def to_device(b, dev="cuda"):
    def logits(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)
    return dict(target=logits(b.target), draft=logits(b.draft),
                draft_tokens=torch.from_numpy(b.draft_tokens).to(dev),
                seq_offsets=torch.from_numpy(b.seq_offsets).to(dev),
                gammas=torch.from_numpy(b.gammas).to(dev))


def run_gpu(b, seed, step, dev_in=None, debug=True, max_gamma=None):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    d = dev_in or to_device(b)
    mg = int(b.gammas.max()) if max_gamma is None else max_gamma
    call = sv.Call(b.B, b.V, mg, b.R_t, b.R_d, debug=debug)
    rc = call.run(d["target"], d["draft"], d["draft_tokens"], d["seq_offsets"], d["gammas"],
                  b.temperature, seed, step)
    assert rc == sv.SV_OK, sv.spec_verify_status_string(rc)
    torch.cuda.synchronize()
    out = dict(tokens=call.out_tokens.cpu().numpy(), n=call.out_n.cpu().numpy(), status=call.status_bits())
    if debug:
        out.update({k: v.cpu().numpy() for k, v in call.dbg.items()})
    return out


def t32(T):
    """The temperature the C ABI receives is a float32; the oracle is given that same value."""
    return float(np.float32(T))


def run_oracle(b, seed, step):
    return oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, t32(b.temperature),
                         seed, step)


def compare(b, g, r, seed, step):
    """Classify every sequence: exact, band (allowed, counted) or mismatch. Returns a report dict."""
    draws = 0
    band = []
    bad = []
    T = t32(b.temperature)
    for s in range(b.B):
        gm = int(b.gammas[s])
        d0 = int(b.seq_offsets[s])
        t0 = d0 + s
        nr, ng = int(r.num_accepted[s]), int(g["n"][s])
        if T > 0 and nr >= 0:  # accept tests up to the first rejection, plus one draw
            draws += (nr + 1 if nr < gm else gm) + 1
        if nr == ng and np.array_equal(r.tokens[t0:t0 + gm + 1], g["tokens"][t0:t0 + gm + 1]):
            continue
        if T == 0 or nr < 0 or ng < 0:
            bad.append((s, "greedy/err", nr, ng))
            continue
        if nr != ng:
            i = min(nr, ng)  # the slot whose accept decision differs
            u = oracle.uniform(seed, step, s, i, 0)
            px, qx = r.p_x[d0 + i], r.q_x[d0 + i]
            ratio = px / qx if qx > 0 else np.inf
            (band if abs(u - ratio) < BAND else bad).append((s, "accept", i, u, ratio))
            continue
        n = nr
        kg = int(g["tokens"][t0 + n])
        u = oracle.uniform(seed, step, s, n, 1)
        drow = b.draft[d0 + n] if n < gm and b.draft is not None else None
        x_excl = int(b.draft_tokens[d0 + n]) if n < gm and b.draft is None else -1  # point-mass draft
        tok, lo, hi, S = oracle.draw_bracket(b.target[t0 + n], drow, b.V, T, u, kg, x_excl)
        dist = 0.0 if lo <= u < hi else min(abs(u - lo), abs(u - hi))
        (band if dist < BAND else bad).append((s, "draw", n, u, kg, tok, lo, hi))
    return dict(draws=draws, band=band, bad=bad)


def assert_parity(b, seed, step, g=None, r=None, check_debug=True):
    g = g if g is not None else run_gpu(b, seed, step)
    r = r if r is not None else run_oracle(b, seed, step)
    assert g["status"] == r.status, (g["status"], r.status)
    rep = compare(b, g, r, seed, step)
    assert not rep["bad"], rep["bad"][:5]
    assert len(rep["band"]) <= 1e-5 * max(rep["draws"], 1) or len(rep["band"]) == 0, rep["band"]
    if check_debug and b.temperature > 0 and r.status == 0:
        np.testing.assert_allclose(g["row_lse"], r.row_lse, rtol=REL, atol=REL)
        m = r.p_x >= 1e-30
        np.testing.assert_allclose(g["p_x"][m], r.p_x[m], rtol=REL)
        m = r.q_x >= 1e-30
        np.testing.assert_allclose(g["q_x"][m], r.q_x[m], rtol=REL)
        np.testing.assert_allclose(g["seq_mass"], r.seq_mass, rtol=REL)
        m = r.beta >= 1e-30
        np.testing.assert_allclose(g["beta"][m], r.beta[m], rtol=REL)
        np.testing.assert_allclose(g["beta"][~m], r.beta[~m], rtol=0, atol=1e-30)
    if check_debug and b.temperature == 0 and r.status == 0:
        np.testing.assert_array_equal(g["row_argmax"], r.row_argmax)
    return rep


def compare_steps(b, g_tokens, g_n, r_tokens, r_n, r0, seed, step0):
    """``compare`` over many steps of one batch at once: g_* / r_* are [steps, R_t] tokens and [steps, B]
    counts from the GPU and from ``oracle.verify_steps``; r0 is the oracle's debug ``Result`` of the batch
    (p(x_i), q(x_i) do not depend on the step). Exact matches are found with array operations; only the
    disagreeing sequences are classified (band or mismatch) one by one. Returns counts: uniform draws
    (accept tests and draws), token draws, band and mismatch lists."""
    T = t32(b.temperature)
    S, B = r_n.shape
    gam = b.gammas.astype(np.int64)
    t0 = (b.seq_offsets[:-1] + np.arange(B)).astype(np.int64)
    # per sequence and step: do all gamma + 1 slots and the count agree
    same = g_n == r_n
    slot_ok = g_tokens == r_tokens  # [S, R_t]
    seq_of_slot = np.repeat(np.arange(B), gam + 1)
    bad_slot = np.zeros((S, B), dtype=bool)
    for s in range(S):
        bad_slot[s] = np.bincount(seq_of_slot, weights=~slot_ok[s], minlength=B) > 0
    agree = same & ~bad_slot
    ok = r_n >= 0
    uni = np.where(r_n < gam, r_n + 1, gam) + 1
    draws = int(uni[ok].sum())
    token_draws = int(ok.sum())
    band, bad = [], []
    for s, q in zip(*np.nonzero(~agree)):
        nr, ng = int(r_n[s, q]), int(g_n[s, q])
        if T == 0 or nr < 0 or ng < 0:
            bad.append((int(s), int(q), "greedy/err", nr, ng))
            continue
        d0 = int(b.seq_offsets[q])
        if nr != ng:
            i = min(nr, ng)
            u = oracle.uniform(seed, step0 + int(s), int(q), i, 0)
            px, qx = r0.p_x[d0 + i], r0.q_x[d0 + i]
            ratio = px / qx if qx > 0 else np.inf
            (band if abs(u - ratio) < BAND else bad).append((int(s), int(q), "accept", i, u, ratio))
            continue
        n = nr
        kg = int(g_tokens[s, t0[q] + n])
        u = oracle.uniform(seed, step0 + int(s), int(q), n, 1)
        gm = int(gam[q])
        drow = b.draft[d0 + n] if n < gm and b.draft is not None else None
        x_excl = int(b.draft_tokens[d0 + n]) if n < gm and b.draft is None else -1
        tok, lo, hi, Sm = oracle.draw_bracket(b.target[t0[q] + n], drow, b.V, T, u, kg, x_excl)
        dist = 0.0 if lo <= u < hi else min(abs(u - lo), abs(u - hi))
        (band if dist < BAND else bad).append((int(s), int(q), "draw", n, u, kg, tok, lo, hi))
    return dict(draws=draws, token_draws=token_draws, band=band, bad=bad)
