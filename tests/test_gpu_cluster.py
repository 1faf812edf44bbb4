"""GPU parity of the small-batch form (one CTA cluster per sequence, the vocabulary-sharded protocol inside the
cluster) against the fp64 oracle, through the C ABI. The form is forced (sv_debug.cluster = 2) on every
batch it can take: the small synthetic workloads at full size, reduced and ragged batches, vocabularies that
give 1 to 8 CTAs per cluster (and the largest slices), greedy, point-mass and fp32 batches, the error paths,
and many steps against the oracle's multi-step entry (the mismatch quota). Outputs and status must equal the
oracle's under the usual rule."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import oracle  # noqa: E402
from speculative_decoding_verification_35_gb300 import synth  # noqa: E402
from tests import parity  # noqa: E402

NAN_BF16, NEG_INF_BF16 = 0x7FC0, 0xFF80


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_35_gb300 import _build
    _build.build()
    oracle.build()


def make_call(b, max_gamma=None, cluster=2):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    mg = int(b.gammas.max()) if max_gamma is None else max_gamma
    call = sv.Call(b.B, b.V, mg, b.R_t, b.R_d)
    call.dbg_struct = sv.SvDebug(0, 0, 0, 0, 0, 0, 0, 0, cluster)
    return call


def run_cluster(b, seed, step, d=None, max_gamma=None, cluster=2):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    d = d or parity.to_device(b)
    call = make_call(b, max_gamma, cluster)
    call.out_tokens.fill_(-9)
    call.out_n.fill_(-9)
    rc = call.run(d["target"], d["draft"], d["draft_tokens"], d["seq_offsets"], d["gammas"], b.temperature, seed, step)
    assert rc == sv.SV_OK, sv.spec_verify_status_string(rc)
    torch.cuda.synchronize()
    return dict(tokens=call.out_tokens.cpu().numpy(), n=call.out_n.cpu().numpy(), status=call.status_bits())


@pytest.mark.parametrize("name,B,V,steps", [("b1_g4_v1024_f32", None, None, 40), ("b8_g4_v32000_t0.7", None, None, 20),
                                            ("b8_g4_v32000_greedy", None, None, 3),
                                            ("b64_g5_v128256", 5, 20000, 4), ("ragged_b128_v129280", 17, 9000, 4),
                                            ("pointmass_b64_g5_v128256", 9, 5000, 4),
                                            ("b8_g4_v32000_t0.7", 3, 131072, 3), ("b8_g4_v32000_t0.7", 4, 4097, 4),
                                            ("b8_g4_v32000_t0.7", 2, 1, 4), ("b1_g4_v1024_f32", 3, 777, 6),
                                            ("b8_g4_v32000_greedy", 9, 8193, 3)])
def test_cluster_form_matches_the_oracle(name, B, V, steps):
    b = synth.make_batch(name, B=B, V=V)
    d = parity.to_device(b)
    tot = dict(draws=0, band=0)
    for step in range(steps):
        g = run_cluster(b, 1234, step, d=d)
        assert g["status"] == 0
        rep = parity.assert_parity(b, 1234, step, g=g, check_debug=False)
        tot["draws"] += rep["draws"]
        tot["band"] += len(rep["band"])
    print(name, B, V, tot)


def test_cluster_form_gamma_zero_max_gamma_and_empty_slots():
    b = synth.make_batch("b64_g5_v128256", B=7, V=3000, gammas=[0, 3, 5, 0, 1, 5, 2])
    d = parity.to_device(b)
    for step in range(3):
        parity.assert_parity(b, 5, step, g=run_cluster(b, 5, step, d=d), check_debug=False)
        parity.assert_parity(b, 5, step, g=run_cluster(b, 5, step, d=d, max_gamma=9), check_debug=False)
    b31 = synth.make_batch("b8_g4_v32000_t0.7", B=2, V=2000, gammas=[31, 0])
    parity.assert_parity(b31, 3, 0, g=run_cluster(b31, 3, 0), check_debug=False)


def _rows(b, s):
    o0 = int(b.seq_offsets[s])
    return o0 + s, o0


@pytest.mark.parametrize("name", ["b8_g4_v32000_t0.7", "pointmass_b64_g5_v128256", "b8_g4_v32000_greedy"])
def test_cluster_form_error_paths(name):
    cases = []
    bb = synth.make_batch(name, B=5, V=700)
    bb.draft_tokens[int(bb.seq_offsets[1]) + 1] = 700          # sequence 1: bad token
    t1, _ = _rows(bb, 1)
    bb.target[t1, 3] = NAN_BF16                                 # ... and a NaN row: the token is reported
    cases.append(bb)
    bb = synth.make_batch(name, B=5, V=700)
    t2, _ = _rows(bb, 2)
    bb.target[t2 + int(bb.gammas[2]), 17] = NAN_BF16           # sequence 2: NaN in its last target row
    t0, _ = _rows(bb, 0)
    bb.target[t0 + 1, :] = NEG_INF_BF16                         # sequence 0: an empty target row
    cases.append(bb)
    if bb.draft is not None:
        bb = synth.make_batch(name, B=5, V=700)
        t3, d3 = _rows(bb, 3)
        bb.target[t3 + 1, 5] = NAN_BF16                         # sequence 3: NaN target row 1 ...
        bb.draft[d3, :] = NEG_INF_BF16                          # ... after an empty draft row 0: empty first
        cases.append(bb)
    for bb in cases:
        for step in range(2):
            r = parity.run_oracle(bb, 1, step)
            g = run_cluster(bb, 1, step)
            assert g["status"] == r.status and r.status != 0, (g["status"], r.status)
            assert np.array_equal(g["n"], r.num_accepted)
            parity.assert_parity(bb, 1, step, g=g, r=r, check_debug=False)
    off = synth.make_batch(name, B=4, V=500)
    off.seq_offsets[2] = 1000                                   # inconsistent offsets: every sequence fails
    g = run_cluster(off, 1, 0, max_gamma=4)
    assert g["status"] == 1 << 4 and np.all(g["n"] == -1)


@pytest.mark.parametrize("name", ["b8_g4_v32000_t0.7", "b1_g4_v1024_f32"])
def test_cluster_form_mismatch_quota_over_many_draws(name):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    b = synth.make_batch(name)
    d = parity.to_device(b)
    steps = -(-100_000 // b.B)
    seed, step0 = 4321, 10_000
    call = make_call(b)
    out_t = np.zeros((steps, b.R_t), np.int32)
    out_n = np.zeros((steps, b.B), np.int32)
    ts = torch.zeros((steps, b.R_t), dtype=torch.int32, device="cuda")
    ns = torch.zeros((steps, b.B), dtype=torch.int32, device="cuda")
    for s in range(steps):
        assert call.run(d["target"], d["draft"], d["draft_tokens"], d["seq_offsets"], d["gammas"], b.temperature,
                        seed, step0 + s, clear_status=False) == sv.SV_OK
        ts[s].copy_(call.out_tokens)
        ns[s].copy_(call.out_n)
    torch.cuda.synchronize()
    out_t, out_n = ts.cpu().numpy(), ns.cpu().numpy()
    assert call.status_bits() == 0
    r_t, r_n, r_st = oracle.verify_steps(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V,
                                         parity.t32(b.temperature), seed, step0, steps)
    r0 = parity.run_oracle(b, seed, step0)
    rep = parity.compare_steps(b, out_t, out_n, r_t, r_n, r0, seed, step0)
    print(f"{name}: steps {steps}, token draws {rep['token_draws']}, band {len(rep['band'])}, "
          f"mismatch {len(rep['bad'])}")
    assert not rep["bad"], rep["bad"][:5]
    assert len(rep["band"]) < 1e-5 * rep["draws"], rep["band"][:5]


def test_library_choice_takes_the_cluster_form_for_small_batches_only():
    # the library's choice (cluster = 0) gives the same outputs as either forced form
    for name in ("b8_g4_v32000_t0.7", "b64_g5_v128256"):
        b = synth.make_batch(name, B=None if name.startswith("b8") else 12, V=None if name.startswith("b8") else 40000)
        d = parity.to_device(b)
        g0 = run_cluster(b, 7, 1, d=d, cluster=0)
        parity.assert_parity(b, 7, 1, g=g0, check_debug=False)
