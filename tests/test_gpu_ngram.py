"""GPU parity of the n-gram drafter (spec_draft_ngram) against its oracle, and the weights-free decode
loop on the device: n-gram drafts -> verify as point-mass drafts with the post-verify update fused ->
next drafts from the updated histories, over several steps, against the oracle chain."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import oracle  # noqa: E402
from oracle.commit import commit  # noqa: E402
from oracle.ngram import draft  # noqa: E402
from speculative_decoding_verification_35_gb300 import synth  # noqa: E402
from tests import parity  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_35_gb300 import _build
    _build.build()
    oracle.build()


def _histories(rng, B, cap, alphabet):
    """Token histories with planted repeats: random tokens, then copies of earlier spans."""
    hist = rng.integers(0, alphabet, size=(B, cap)).astype(np.int32)
    lens = rng.integers(0, cap + 1, size=B).astype(np.int32)
    for b in range(B):
        L = int(lens[b])
        if L > 20:
            for _ in range(3):
                a = int(rng.integers(0, L - 10)); c = int(rng.integers(a + 1, L)); w = int(rng.integers(2, 9))
                w = min(w, L - c, c - a)
                hist[b, c:c + w] = hist[b, a:a + w]
    return hist, lens


def _gpu_draft(hist, lens, n_min, n_max, gmax):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    B, cap = hist.shape
    h = torch.from_numpy(hist).cuda(); L = torch.from_numpy(lens).cuda()
    toks = torch.full((max(B * gmax, 1),), -7, dtype=torch.int32, device="cuda")
    gam = torch.full((max(B, 1),), -7, dtype=torch.int32, device="cuda")
    offs = torch.full((B + 1,), -7, dtype=torch.int32, device="cuda")
    pos = torch.full((max(B, 1),), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = sv.spec_draft_ngram(h.data_ptr(), cap, L.data_ptr(), B, n_min, n_max, gmax, toks.data_ptr(), gam.data_ptr(),
                             offs.data_ptr(), pos.data_ptr(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == sv.SV_OK
    torch.cuda.synchronize()
    o = offs.cpu().numpy()
    return toks.cpu().numpy()[:o[-1]], gam.cpu().numpy()[:B], o, pos.cpu().numpy()[:B], int(st.item())


@pytest.mark.parametrize("B,cap,alphabet,n_min,n_max,gmax", [(64, 2048, 50, 1, 3, 5), (7, 300, 3, 2, 4, 31),
                                                             (3000, 64, 8, 1, 2, 4), (1, 12288, 1000, 1, 5, 8), (2, 32768, 100, 1, 3, 6),
                                                             (5, 100, 5, 1, 1, 0)])
def test_drafter_matches_oracle(B, cap, alphabet, n_min, n_max, gmax):
    rng = np.random.default_rng(B + cap)
    hist, lens = _histories(rng, B, cap, alphabet)
    if B >= 3:
        lens[:3] = [0, 1, 2]  # empty and too-short histories
    t, g, o, p, st = _gpu_draft(hist, lens, n_min, n_max, gmax)
    rt, rg, ro, rp = draft(hist, lens, n_min, n_max, gmax)
    assert st == 0
    assert np.array_equal(g, rg) and np.array_equal(o, ro) and np.array_equal(p, rp) and np.array_equal(t, rt)


def test_drafter_flags_inconsistent_lengths_and_empty_batch():
    from speculative_decoding_verification_35_gb300 import specverify as sv
    hist = np.zeros((3, 16), np.int32); lens = np.array([4, -2, 17], np.int32)
    t, g, o, p, st = _gpu_draft(hist, lens, 1, 2, 3)
    assert st == 1 << sv.SV_ERR_INVALID_ARG and g.tolist()[1:] == [0, 0] and o[-1] == g[0]
    t, g, o, p, st = _gpu_draft(np.zeros((0, 16), np.int32), np.zeros(0, np.int32), 1, 2, 3)
    assert o.tolist() == [0]


def test_weights_free_decode_loop_on_device():
    """Three decode steps with no draft model: drafts from the histories, target logits for the CSR
    layout those drafts give (a stand-in for the target model), point-mass verification with the
    update fused, all on the device; compared with the oracle's drafter, verify and update."""
    from speculative_decoding_verification_35_gb300 import specverify as sv
    B, cap, V, gmax, T = 16, 512, 4096, 5, 1.0
    rng = np.random.default_rng(21)
    hist0, _ = _histories(rng, B, cap, 40)
    lens0 = np.full(B, 200, np.int32)
    h = torch.from_numpy(hist0).cuda(); L = torch.from_numpy(lens0).cuda()
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    toks = torch.zeros(B * gmax, dtype=torch.int32, device="cuda")
    gam = torch.zeros(B, dtype=torch.int32, device="cuda")
    offs = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rh, rl = hist0.copy(), lens0.copy()
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(3):
        assert sv.spec_draft_ngram(h.data_ptr(), cap, L.data_ptr(), B, 1, 3, gmax, toks.data_ptr(), gam.data_ptr(),
                                   offs.data_ptr(), pos.data_ptr(), st.data_ptr(), stream) == sv.SV_OK
        # the target model's stand-in needs the layout on the host (a real target runs on the device)
        o = offs.cpu().numpy(); g_np = gam.cpu().numpy()
        rt, rg, ro, rp = draft(rh, rl, 1, 3, gmax)
        assert np.array_equal(o, ro) and np.array_equal(g_np, rg)
        assert np.array_equal(toks.cpu().numpy()[:o[-1]], rt)
        R_t = int(o[-1]) + B
        trng = np.random.default_rng(100 + step)
        target = synth.to_bf16_bits(trng.normal(0, 2.5, size=(R_t, V)) - 1.1 * np.log(np.arange(1, V + 1)))
        tgt = torch.from_numpy(target.view(np.int16)).view(torch.bfloat16).cuda()
        call = sv.Call(B, V, gmax, R_t, max(int(o[-1]), 1))
        assert call.run_fused(tgt, None, toks, offs, gam, T, 1234, step, h, cap, L, nxt) == sv.SV_OK
        torch.cuda.synchronize()
        r = oracle.verify(target, None, rt, ro, rg, V, T, 1234, step)
        assert r.status == 0 and call.status_bits() == 0
        assert np.array_equal(call.out_n.cpu().numpy(), r.num_accepted)
        assert np.array_equal(call.out_tokens.cpu().numpy(), r.tokens)
        rh, rl, rn, rs = commit(r.tokens, r.num_accepted, ro, rh, cap, rl)
        assert np.array_equal(h.cpu().numpy(), rh) and np.array_equal(L.cpu().numpy(), rl)
        assert np.array_equal(nxt.cpu().numpy(), rn)
