"""GPU parity of the post-verify update (spec_verify_commit) against its oracle, through the C ABI:
synthetic verify outputs with failed, full and inconsistent sequences, and verify -> commit chained on
one stream over several decode steps with no host synchronisation between them."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import oracle  # noqa: E402
from oracle.commit import commit  # noqa: E402
from speculative_decoding_verification_35_gb300 import synth  # noqa: E402
from tests import parity  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_35_gb300 import _build
    _build.build()
    oracle.build()


def _gpu_commit(out_tokens, out_n, offs, hist, cap, lens):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    d = {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.int32)).cuda()
         for k, v in dict(t=out_tokens, n=out_n, o=offs, h=hist, L=lens).items()}
    nxt = torch.full((len(out_n),), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = sv.spec_verify_commit(d["t"].data_ptr(), d["n"].data_ptr(), d["o"].data_ptr(), len(out_n), d["h"].data_ptr(),
                               cap, d["L"].data_ptr(), nxt.data_ptr(), st.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert rc == sv.SV_OK
    torch.cuda.synchronize()
    return d["h"].cpu().numpy(), d["L"].cpu().numpy(), nxt.cpu().numpy(), int(st.item()) & 0xFFFFFFFF


@pytest.mark.parametrize("B,cap", [(1, 8), (37, 40), (5000, 64)])
def test_commit_matches_oracle_on_synthetic_outputs(B, cap):
    rng = np.random.default_rng(B)
    gam = rng.integers(0, 32, size=B)
    offs = np.concatenate([[0], np.cumsum(gam)]).astype(np.int32)
    R_t = int(offs[-1]) + B
    out_tokens = rng.integers(0, 1 << 20, size=R_t).astype(np.int32)
    n = np.array([rng.integers(-1, g + 1) for g in gam], np.int32)
    n[:: 7] = -1
    n[3::11] = np.minimum(gam[3::11] + 1, 31)  # some inconsistent counts (n above gamma)
    lens = rng.integers(0, cap, size=B).astype(np.int32)
    lens[5::13] = -3
    hist = rng.integers(0, 1 << 20, size=(B, cap)).astype(np.int32)
    gh, gl, gn, gs = _gpu_commit(out_tokens, n, offs, hist, cap, lens)
    rh, rl, rn, rs = commit(out_tokens, n, offs, hist, cap, lens)
    assert np.array_equal(gh, rh) and np.array_equal(gl, rl) and np.array_equal(gn, rn)
    assert gs == rs


def test_commit_rejects_counts_above_the_largest_gamma():
    # gaps above 31 with n above 31: lanes 0..31 could not copy the slots, so nothing is appended
    out = np.arange(200, dtype=np.int32)
    offs = np.array([0, 40, 80, 120], np.int32)
    n = np.array([35, 31, 40], np.int32)
    hist = np.full((3, 100), 5, np.int32)
    lens = np.array([0, 1, 2], np.int32)
    gh, gl, gn, gs = _gpu_commit(out, n, offs, hist, 100, lens)
    rh, rl, rn, rs = commit(out, n, offs, hist, 100, lens)
    assert rs == 1 << 4 and gs == rs
    assert np.array_equal(gh, rh) and np.array_equal(gl, rl) and np.array_equal(gn, rn)
    assert gn.tolist() == [-1, int(out[40 + 1 + 31]), -1]


@pytest.mark.parametrize("name", ["b64_g5_v128256", "ragged_b128_v129280"])
def test_verify_then_commit_over_steps_without_host_sync(name):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    b = synth.make_batch(name)
    d = parity.to_device(b)
    cap = 64
    call = sv.Call(b.B, b.V, int(b.gammas.max()), b.R_t, b.R_d)
    hist = torch.zeros((b.B, cap), dtype=torch.int32, device="cuda")
    lens = torch.zeros(b.B, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b.B, dtype=torch.int32, device="cuda")
    steps = 3
    for step in range(steps):  # all enqueued on one stream; the host never waits in between
        assert call.run(d["target"], d["draft"], d["draft_tokens"], d["seq_offsets"], d["gammas"], b.temperature,
                        1234, step, clear_status=step == 0) == sv.SV_OK
        assert call.commit(d["seq_offsets"], hist, cap, lens, nxt) == sv.SV_OK
    torch.cuda.synchronize()
    assert call.status_bits() == 0
    rh, rl = np.zeros((b.B, cap), np.int32), np.zeros(b.B, np.int32)
    for step in range(steps):
        r = parity.run_oracle(b, 1234, step)
        rh, rl, rn, rs = commit(r.tokens, r.num_accepted, b.seq_offsets, rh, cap, rl)
        assert rs == 0
    assert np.array_equal(hist.cpu().numpy(), rh)
    assert np.array_equal(lens.cpu().numpy(), rl)
    assert np.array_equal(nxt.cpu().numpy(), rn)


@pytest.mark.parametrize("name", ["b64_g5_v128256", "b8_g4_v32000_greedy", "ragged_b128_v129280", "b1_g4_v1024_f32"])
def test_fused_update_matches_oracle_over_steps(name):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    b = synth.make_batch(name)
    d = parity.to_device(b)
    cap = 48
    call = sv.Call(b.B, b.V, int(b.gammas.max()), b.R_t, b.R_d)
    hist = torch.zeros((b.B, cap), dtype=torch.int32, device="cuda")
    lens = torch.zeros(b.B, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b.B, dtype=torch.int32, device="cuda")
    rh, rl = np.zeros((b.B, cap), np.int32), np.zeros(b.B, np.int32)
    for step in range(3):
        assert call.run_fused(d["target"], d["draft"], d["draft_tokens"], d["seq_offsets"], d["gammas"],
                              b.temperature, 1234, step, hist, cap, lens, nxt) == sv.SV_OK
        torch.cuda.synchronize()
        r = parity.run_oracle(b, 1234, step)
        assert np.array_equal(call.out_n.cpu().numpy(), r.num_accepted)
        assert np.array_equal(call.out_tokens.cpu().numpy(), r.tokens)
        rh, rl, rn, rs = commit(r.tokens, r.num_accepted, b.seq_offsets, rh, cap, rl)
        assert call.status_bits() == rs == 0
        assert np.array_equal(hist.cpu().numpy(), rh)
        assert np.array_equal(lens.cpu().numpy(), rl)
        assert np.array_equal(nxt.cpu().numpy(), rn)


def test_fused_update_overflow_and_failed_sequences():
    from speculative_decoding_verification_35_gb300 import specverify as sv
    b = synth.make_batch("ragged_b128_v129280", B=9, V=3001)
    b.draft_tokens[int(b.seq_offsets[2])] = b.V + 5  # sequence 2 fails verification (bad token)
    d = parity.to_device(b)
    cap = 8
    call = sv.Call(b.B, b.V, int(b.gammas.max()), b.R_t, b.R_d)
    lens0 = np.array([0, 7, 0, 3, 8, 1, 2, 6, 0], np.int32)  # some cannot take n + 1 more tokens
    hist = torch.full((b.B, cap), 77, dtype=torch.int32, device="cuda")
    lens = torch.from_numpy(lens0.copy()).cuda()
    nxt = torch.zeros(b.B, dtype=torch.int32, device="cuda")
    assert call.run_fused(d["target"], d["draft"], d["draft_tokens"], d["seq_offsets"], d["gammas"], b.temperature,
                          7, 0, hist, cap, lens, nxt) == sv.SV_OK
    torch.cuda.synchronize()
    r = parity.run_oracle(b, 7, 0)
    rh, rl, rn, rs = commit(r.tokens, r.num_accepted, b.seq_offsets, np.full((b.B, cap), 77, np.int32), cap, lens0)
    assert rn[2] == -1 and rs & (1 << sv.SV_ERR_CAPACITY)
    assert call.status_bits() == rs | r.status
    assert np.array_equal(hist.cpu().numpy(), rh)
    assert np.array_equal(lens.cpu().numpy(), rl)
    assert np.array_equal(nxt.cpu().numpy(), rn)


def test_fused_update_with_a_failure_in_rows_after_the_rejection():
    """Slot-order batches (bf16 rows with draft rows, no debug arrays): a NaN in a sequence's last target
    row, which most first rejections leave out of the draw, is found by the sequence's find before it writes;
    the sequence fails (n = -1, history and length kept, next token -1) like the oracle's."""
    from speculative_decoding_verification_35_gb300 import specverify as sv
    b = synth.make_batch("b64_g5_v128256", B=9, V=3000)
    t2 = int(b.seq_offsets[2]) + 2
    b.target[t2 + int(b.gammas[2]), 11] = 0x7FC0  # sequence 2: NaN in its last target row
    d = parity.to_device(b)
    cap = 40
    call = sv.Call(b.B, b.V, int(b.gammas.max()), b.R_t, b.R_d)
    lens0 = np.arange(b.B, dtype=np.int32)
    hist = torch.full((b.B, cap), 55, dtype=torch.int32, device="cuda")
    lens = torch.from_numpy(lens0.copy()).cuda()
    nxt = torch.zeros(b.B, dtype=torch.int32, device="cuda")
    for step in range(3):
        r = parity.run_oracle(b, 9, step)
        rh, rl, rn, rs = commit(r.tokens, r.num_accepted, b.seq_offsets, hist.cpu().numpy(), cap, lens.cpu().numpy())
        assert call.run_fused(d["target"], d["draft"], d["draft_tokens"], d["seq_offsets"], d["gammas"],
                              b.temperature, 9, step, hist, cap, lens, nxt) == sv.SV_OK
        torch.cuda.synchronize()
        assert r.num_accepted[2] == -1 and r.status == 1 << sv.SV_ERR_NONFINITE
        assert np.array_equal(call.out_n.cpu().numpy(), r.num_accepted)
        assert np.array_equal(call.out_tokens.cpu().numpy(), r.tokens)
        assert call.status_bits() == rs | r.status
        assert np.array_equal(hist.cpu().numpy(), rh)
        assert np.array_equal(lens.cpu().numpy(), rl)
        assert np.array_equal(nxt.cpu().numpy(), rn)
