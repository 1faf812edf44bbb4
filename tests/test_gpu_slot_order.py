"""GPU parity of the slot-order verify path against the fp64 oracle, through the C ABI.

Calls without per-row debug outputs on bf16 rows with 16-byte alignment (sampled, linear drafts with draft
rows, row map in shared memory, enough statistics tasks) stream the statistics slot by slot and decide each
sequence at its first rejection; the rows after it are checked for NaN / +inf / empty by the sequence's find.
These tests force that path (sv_debug.order = 2, no debug arrays) on full-size and reduced batches, ragged gammas and gamma = 0, more sequences than
CTAs, a max_gamma above the batch's (empty slots), errors planted in rows before and after the first
rejection, and waits that run out. Point-mass batches keep sequence order; their cases here run that path
without debug arrays. Outputs and status must equal the oracle's under the usual rule.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import oracle  # noqa: E402
from speculative_decoding_verification_35_gb300 import synth  # noqa: E402
from tests import parity  # noqa: E402

NONFINITE, EMPTY, TIMEOUT = 1 << 5, 1 << 6, 1 << 7
NAN_BF16, NEG_INF_BF16 = 0x7FC0, 0xFF80


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_35_gb300 import _build
    _build.build()
    oracle.build()


def run_plain(b, seed, step, d=None, max_gamma=None, spin=0, order=2):
    """One call without debug arrays, through a debug struct that carries no arrays: the statistics in slot
    order wherever the call allows it (order 2; 0: the library's choice by size, 1: sequence order); spin > 0
    bounds every wait to that many polls."""
    from speculative_decoding_verification_35_gb300 import specverify as sv
    d = d or parity.to_device(b)
    mg = int(b.gammas.max()) if max_gamma is None else max_gamma
    call = sv.Call(b.B, b.V, mg, b.R_t, b.R_d)
    call.dbg_struct = sv.SvDebug(0, 0, 0, 0, 0, 0, spin, order, 1)  # the persistent launch (no cluster form)
    call.out_tokens.fill_(-9)
    call.out_n.fill_(-9)
    rc = call.run(d["target"], d["draft"], d["draft_tokens"], d["seq_offsets"], d["gammas"], b.temperature, seed, step)
    assert rc == sv.SV_OK, sv.spec_verify_status_string(rc)
    torch.cuda.synchronize()
    return dict(tokens=call.out_tokens.cpu().numpy(), n=call.out_n.cpu().numpy(), status=call.status_bits())


@pytest.mark.parametrize("name", ["b64_g5_v128256", "b256_g3_v152064_t0.8", "pointmass_b64_g5_v128256",
                                  "b8_g4_v32000_t0.7"])
@pytest.mark.parametrize("order", [0, 1, 2])
def test_slot_order_full_size(name, order):
    b = synth.make_batch(name)
    d = parity.to_device(b)
    tot = dict(draws=0, band=0)
    for step in range(4):
        g = run_plain(b, 1234, step, d=d, order=order)
        assert g["status"] == 0
        rep = parity.assert_parity(b, 1234, step, g=g, check_debug=False)
        tot["draws"] += rep["draws"]
        tot["band"] += len(rep["band"])
    print(name, tot)


@pytest.mark.parametrize("name,B,V", [("b64_g5_v128256", 5, 20000), ("ragged_b128_v129280", 17, 9000),
                                      ("pointmass_b64_g5_v128256", 9, 5000), ("b64_g5_v128256", 1, 8),
                                      ("b8_g4_v32000_t0.7", 6, 4096), ("b8_g4_v32000_t0.7", 3, 40000),
                                      ("b256_g3_v152064_t0.8", 200, 4096), ("pointmass_b64_g5_v128256", 350, 1024)])
def test_slot_order_reduced_and_ragged(name, B, V):
    b = synth.make_batch(name, B=B, V=V)
    d = parity.to_device(b)
    for step in range(4):
        g = run_plain(b, 99, step, d=d)
        parity.assert_parity(b, 99, step, g=g, check_debug=False)


def test_slot_order_gamma_zero_and_empty_slots():
    for name in ("b64_g5_v128256", "pointmass_b64_g5_v128256"):
        b = synth.make_batch(name, B=7, V=3000, gammas=[0, 3, 5, 0, 1, 5, 2])
        d = parity.to_device(b)
        for step in range(3):
            parity.assert_parity(b, 5, step, g=run_plain(b, 5, step, d=d), check_debug=False)
            # a max_gamma above the batch's: slots no sequence has (holes in the slot order)
            parity.assert_parity(b, 5, step, g=run_plain(b, 5, step, d=d, max_gamma=9), check_debug=False)


def _rows(b, s):
    """(first target row, first draft row) of sequence s."""
    o0 = int(b.seq_offsets[s])
    return o0 + s, o0


@pytest.mark.parametrize("pm", [False, True])
def test_errors_report_the_first_failure_in_order(pm):
    name = "pointmass_b64_g5_v128256" if pm else "b64_g5_v128256"
    cases = []
    # NaN in the last target row of sequence 2 (after most first rejections: the find's check)
    bb = synth.make_batch(name, B=5, V=704)
    t0, _ = _rows(bb, 2)
    bb.target[t0 + int(bb.gammas[2]), 17] = NAN_BF16
    cases.append(bb)
    # +inf in the last target row of sequence 4
    bb = synth.make_batch(name, B=5, V=704)
    t0, _ = _rows(bb, 4)
    bb.target[t0 + int(bb.gammas[4]), 700] = 0x7F80
    cases.append(bb)
    # an empty (all -inf) last target row of sequence 0, NaN in the one of sequence 1
    bb = synth.make_batch(name, B=5, V=704)
    t0, _ = _rows(bb, 0)
    bb.target[t0 + int(bb.gammas[0]), :] = NEG_INF_BF16
    t1, _ = _rows(bb, 1)
    bb.target[t1 + int(bb.gammas[1]), 3] = NAN_BF16
    cases.append(bb)
    if not pm:
        # an empty last draft row of sequence 0; in sequence 3, NaN in target row 1 and an empty draft row 3
        # (the first failing row in order decides the code); in sequence 1, an empty draft row 0 and NaN in
        # target row 4
        bb = synth.make_batch(name, B=5, V=704)
        _, d0 = _rows(bb, 0)
        bb.draft[d0 + int(bb.gammas[0]) - 1, :] = NEG_INF_BF16
        t3, d3 = _rows(bb, 3)
        bb.target[t3 + 1, 5] = NAN_BF16
        bb.draft[d3 + 3, :] = NEG_INF_BF16
        t1, d1 = _rows(bb, 1)
        bb.draft[d1, :] = NEG_INF_BF16
        bb.target[t1 + 4, 9] = NAN_BF16
        cases.append(bb)
    # a bad draft token with a NaN row in the same sequence: the token is reported, not the row
    bb = synth.make_batch(name, B=5, V=704)
    t4, _ = _rows(bb, 4)
    bb.draft_tokens[int(bb.seq_offsets[4]) + 1] = 704
    bb.target[t4, 0] = NAN_BF16
    cases.append(bb)
    for bb in cases:
        for step in range(3):
            r = parity.run_oracle(bb, 1, step)
            # both paths: without debug arrays (slot order for batches with draft rows) and with them
            # (sequence order); each reports the first failure in the rule's order, as the oracle does
            for g in (run_plain(bb, 1, step), parity.run_gpu(bb, 1, step)):
                assert g["status"] == r.status and r.status != 0, (g["status"], r.status)
                assert np.array_equal(g["n"], r.num_accepted), (g["n"], r.num_accepted)
                parity.assert_parity(bb, 1, step, g=g, r=r, check_debug=False)


@pytest.mark.parametrize("name,B,V", [("b64_g5_v128256", None, None), ("pointmass_b64_g5_v128256", None, None),
                                      ("b256_g3_v152064_t0.8", 200, 4096)])
def test_slot_order_waits_that_run_out(name, B, V):
    b = synth.make_batch(name, B=B, V=V)
    d = parity.to_device(b)
    r = parity.run_oracle(b, 1234, 3)
    for rep in range(2):
        g = run_plain(b, 1234, 3, d=d, spin=1)
        st = g["status"]
        assert st & ~TIMEOUT == 0, st
        failed = 0
        for s in range(b.B):
            t0, gm = int(b.seq_offsets[s]) + s, int(b.gammas[s])
            slots = g["tokens"][t0:t0 + gm + 1]
            if g["n"][s] == -1:
                assert np.all(slots == -1), (s, slots)
                failed += 1
            else:
                assert g["n"][s] == r.num_accepted[s] and np.array_equal(slots, r.tokens[t0:t0 + gm + 1]), s
        assert (failed > 0) == bool(st & TIMEOUT)
        if B is None:
            assert st & TIMEOUT and failed > 0
    g = run_plain(b, 1234, 3, d=d)
    parity.assert_parity(b, 1234, 3, g=g, r=r, check_debug=False)
