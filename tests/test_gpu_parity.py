"""GPU parity of the CUDA verify step against the fp64 oracle, through the C ABI.

Workloads: every synthetic workload at full size (the launch configuration bench.py times), several
steps each, plus reduced and ragged cases (V not a multiple of the tiles, unaligned rows, gamma = 0 and
gamma = 31, B = 1), degenerate distributions and the device error paths.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import oracle  # noqa: E402
from speculative_decoding_verification_35_gb300 import synth  # noqa: E402
from tests import parity  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_35_gb300 import _build
    _build.build()
    oracle.build()


FULL = ["b1_g4_v1024_f32", "b8_g4_v32000_t0.7", "b8_g4_v32000_greedy", "b64_g5_v128256",
        "b256_g3_v152064_t0.8", "ragged_b128_v129280"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads(name):
    b = synth.make_batch(name)
    d = parity.to_device(b)
    steps = {"b1_g4_v1024_f32": 40, "b8_g4_v32000_t0.7": 20, "b8_g4_v32000_greedy": 1}.get(name, 3)
    tot = dict(draws=0, band=0)
    for step in range(steps):
        g = parity.run_gpu(b, 1234, step, dev_in=d)
        rep = parity.assert_parity(b, 1234, step, g=g)
        tot["draws"] += rep["draws"]
        tot["band"] += len(rep["band"])
    print(name, tot)


@pytest.mark.parametrize("name,B,V", [("b64_g5_v128256", 5, 20000), ("ragged_b128_v129280", 17, 9001),
                                      ("b8_g4_v32000_t0.7", 3, 1001), ("b1_g4_v1024_f32", 3, 777),
                                      ("b8_g4_v32000_greedy", 9, 8193), ("b256_g3_v152064_t0.8", 2, 1)])
def test_ragged_tiles_and_unaligned_rows(name, B, V):
    b = synth.make_batch(name, B=B, V=V)
    for step in range(4):
        parity.assert_parity(b, 99, step)


def test_more_sequences_than_ctas():
    # bf16 rows with V * 2 a multiple of 16 take the bulk-copy path; with more sequences than CTAs (304
    # on a GB300) each decision is made by one warp instead of by a CTA's deciding warps together
    b = synth.make_batch("b64_g5_v128256", B=400, V=2048)
    parity.assert_parity(b, 77, 0)
    bp = synth.make_batch("pointmass_b64_g5_v128256", B=350, V=1024)
    parity.assert_parity(bp, 77, 1)


@pytest.mark.parametrize("name,B,V", [("b64_g5_v128256", 64, 128256), ("pointmass_b64_g5_v128256", 9, 5000),
                                      ("b1_g4_v1024_f32", 3, 777)])
def test_host_buffer_form_matches_device_form(name, B, V):
    # spec_verify_host copies page-locked host inputs into staging buffers, runs the step and copies the
    # outputs back: the same tokens and counts as spec_verify_ex on device inputs, and oracle parity
    from speculative_decoding_verification_35_gb300 import specverify as sv
    b = synth.make_batch(name, B=B, V=V)
    d = parity.to_device(b)
    host = {k: (None if v is None else v.cpu().pin_memory()) for k, v in d.items()}
    staging = {k: (None if v is None else torch.empty_like(v)) for k, v in d.items()}
    mg = int(b.gammas.max())
    call = sv.Call(b.B, b.V, mg, b.R_t, b.R_d)
    out_t = torch.full((b.R_t,), -9, dtype=torch.int32).pin_memory()
    out_n = torch.full((b.B,), -9, dtype=torch.int32).pin_memory()
    rc = call.run_host(host["target"], host["draft"], host["draft_tokens"], host["seq_offsets"], host["gammas"],
                       b.temperature, 31, 2, out_t, out_n, staging)
    assert rc == sv.SV_OK, sv.spec_verify_status_string(rc)
    torch.cuda.synchronize()
    assert call.status_bits() == 0
    g = parity.run_gpu(b, 31, 2, dev_in=d, debug=False)
    assert np.array_equal(out_t.numpy(), g["tokens"]) and np.array_equal(out_n.numpy(), g["n"])
    parity.assert_parity(b, 31, 2, g=g, check_debug=False)


def test_gamma_zero_and_max_gamma():
    b = synth.make_batch("ragged_b128_v129280", B=6, V=3000, gammas=[0, 31, 1, 0, 7, 31])
    for step in range(3):
        parity.assert_parity(b, 5, step)
    bg = synth.make_batch("b8_g4_v32000_greedy", B=4, V=3000, gammas=[0, 31, 2, 5])
    parity.assert_parity(bg, 5, 0)


def test_max_gamma_above_batch_gammas():
    b = synth.make_batch("b8_g4_v32000_t0.7", B=4, V=5000)
    g = parity.run_gpu(b, 3, 0, max_gamma=31)
    parity.assert_parity(b, 3, 0, g=g)


def _custom(target, draft, tokens, gammas, T):
    offs = np.zeros(len(gammas) + 1, np.int32)
    offs[1:] = np.cumsum(gammas)
    w = synth.Workload("custom", len(gammas), target.shape[1], synth.F32, T, None, 1.0, 0.0, 1.0, (1.0,))
    return synth.Batch(w, target.astype(np.float32), None if draft is None else draft.astype(np.float32),
                       np.asarray(tokens, np.int32), offs, np.asarray(gammas, np.int32))


def test_identical_rows_accept_everything():
    rng = np.random.default_rng(0)
    t = rng.normal(0, 2, size=(3 * 5, 300))
    d = np.concatenate([t[s * 5: s * 5 + 4] for s in range(3)])
    toks = rng.integers(0, 300, size=12)
    b = _custom(t, d, toks, [4, 4, 4], 1.0)
    g = parity.run_gpu(b, 1, 0)
    assert np.array_equal(g["n"], [4, 4, 4])
    parity.assert_parity(b, 1, 0, g=g)


def test_disjoint_supports_and_neg_inf():
    V = 64
    t = np.full((2, V), -np.inf)
    t[:, :8] = np.linspace(0, 1, 8)
    d = np.full((1, V), -np.inf)
    d[0, 32:40] = 0.5
    b = _custom(t, d, [35], [1], 0.9)
    for step in range(20):
        g = parity.run_gpu(b, 7, step)
        assert g["n"][0] == 0 and 0 <= g["tokens"][0] < 8  # beta = 0: rejected, residual = p
        parity.assert_parity(b, 7, step, g=g)


def test_error_paths_match_oracle_and_do_not_disturb_others():
    b = synth.make_batch("b8_g4_v32000_t0.7", B=5, V=700)
    cases = []
    bt = synth.make_batch("b8_g4_v32000_t0.7", B=5, V=700)
    bt.draft_tokens[6] = 700                      # sequence 1: bad token
    cases.append((bt, 1 << 3))
    bn = synth.make_batch("b8_g4_v32000_t0.7", B=5, V=700)
    bn.target[12, 3] = 0x7FC0                     # sequence 2: NaN (target rows 10..14)
    cases.append((bn, 1 << 5))
    bi = synth.make_batch("b8_g4_v32000_t0.7", B=5, V=700)
    bi.draft[0, :] = 0xFF80                       # sequence 0: all -inf draft row
    cases.append((bi, 1 << 6))
    for bb, bit in cases:
        g = parity.run_gpu(bb, 1, 0)
        r = parity.run_oracle(bb, 1, 0)
        assert g["status"] == bit and r.status == bit
        assert np.array_equal(g["n"], r.num_accepted)
        parity.assert_parity(bb, 1, 0, g=g, r=r, check_debug=False)
    assert b.B == 5


def test_bad_offsets_fail_the_whole_batch_without_reading_rows():
    """Inconsistent CSR offsets make row ownership ambiguous: like the oracle, the call fails every
    sequence (n = -1) and reads no logit row."""
    for mutate in (lambda o: o.__setitem__(2, 1000), lambda o: o.__setitem__(2, 2), lambda o: o.__setitem__(0, 1)):
        b = synth.make_batch("b8_g4_v32000_t0.7", B=4, V=500)
        mutate(b.seq_offsets)
        g = parity.run_gpu(b, 1, 0, max_gamma=4, debug=False)
        r = parity.run_oracle(b, 1, 0)
        assert g["status"] == 1 << 4 and r.status == 1 << 4
        assert np.all(g["n"] == -1)
    b = synth.make_batch("b8_g4_v32000_t0.7", B=4, V=500)
    b.gammas[1] = 5  # gamma disagrees with the offsets
    g = parity.run_gpu(b, 1, 0, max_gamma=5, debug=False)
    assert g["status"] == 1 << 4 and np.all(g["n"] == -1)
    b = synth.make_batch("b8_g4_v32000_t0.7", B=4, V=500)
    g = parity.run_gpu(b, 1, 0, max_gamma=3, debug=False)  # gamma = 4 above max_gamma
    assert g["status"] == 1 << 4 and np.all(g["n"] == -1)


def test_plain_blocking_form():
    from speculative_decoding_verification_35_gb300 import specverify as sv
    b = synth.make_batch("ragged_b128_v129280", B=9, V=4000)
    d = parity.to_device(b)
    out_t = torch.empty(b.R_t, dtype=torch.int32, device="cuda")
    out_n = torch.empty(b.B, dtype=torch.int32, device="cuda")
    rc = sv.spec_verify(d["target"].data_ptr(), d["draft"].data_ptr(), d["draft_tokens"].data_ptr(),
                        d["seq_offsets"].data_ptr(), d["gammas"].data_ptr(), b.B, b.V, 1.0, 77, 5,
                        out_t.data_ptr(), out_n.data_ptr())
    assert rc == sv.SV_OK
    r = parity.run_oracle(b, 77, 5)
    assert np.array_equal(out_n.cpu().numpy(), r.num_accepted)
    assert np.array_equal(out_t.cpu().numpy(), r.tokens)
    bb = synth.make_batch("ragged_b128_v129280", B=3, V=100)
    bb.draft_tokens[0] = -1
    d = parity.to_device(bb)
    rc = sv.spec_verify(d["target"].data_ptr(), d["draft"].data_ptr(), d["draft_tokens"].data_ptr(),
                        d["seq_offsets"].data_ptr(), d["gammas"].data_ptr(), bb.B, bb.V, 1.0, 1, 0,
                        out_t.data_ptr(), out_n.data_ptr())
    assert rc == sv.SV_ERR_BAD_TOKEN


def test_philox_against_curand_device_function(tmp_path):
    """The library's device Philox equals a call of curand_Philox4x32_10(counter, key) on every word."""
    import ctypes
    import os
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = os.path.join(root, "tests", "cuda", "philox_check.cu")
    so = str(tmp_path / "philox_check.so")
    subprocess.check_call(["/usr/local/cuda/bin/nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-Xcompiler", "-fPIC", "-shared", "-I", os.path.join(root, "include"), src, "-o", so])
    L = ctypes.CDLL(so)
    n = 1 << 16
    rng = np.random.default_rng(3)
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2**32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    ours = np.zeros((n, 4), np.uint32)
    ref = np.zeros((n, 4), np.uint32)
    rc = L.philox_check(ctypes.c_int(n), ctr.ctypes.data_as(ctypes.c_void_p), key.ctypes.data_as(ctypes.c_void_p),
                        ours.ctypes.data_as(ctypes.c_void_p), ref.ctypes.data_as(ctypes.c_void_p))
    assert rc == 0
    assert np.array_equal(ours, ref)
    for i in range(0, n, 4099):
        assert np.array_equal(oracle.philox4x32_10(ctr[i], key[i]), ours[i])


def test_statistical_losslessness_on_gpu():
    """10^6 sequences of V = 8 on the GPU: first emitted token ~ p_0 (chi-square), beta = acceptance rate."""
    from scipy.stats import chi2
    V, N = 8, 1_000_000
    rng = np.random.default_rng(8)
    p = rng.dirichlet(np.ones(V)) * 0.99 + 0.01 / V
    q = rng.dirichlet(np.ones(V)) * 0.99 + 0.01 / V
    lt = np.log(p).astype(np.float32)
    ld = np.log(q).astype(np.float32)
    target = np.tile(np.stack([lt, lt]), (N, 1))
    draft = np.tile(ld[None], (N, 1))
    toks = rng.choice(V, size=N, p=q / q.sum()).astype(np.int32)
    b = _custom(target, draft, toks, np.ones(N, np.int32), 1.0)
    g = parity.run_gpu(b, 2024, 0, debug=False)
    first = g["tokens"][0::2]
    pe = np.exp(lt.astype(np.float64)); pe /= pe.sum()
    qe = np.exp(ld.astype(np.float64)); qe /= qe.sum()
    cnt = np.bincount(first, minlength=V)
    stat = ((cnt - pe * N) ** 2 / (pe * N)).sum()
    assert chi2.sf(stat, V - 1) > 1e-4
    beta = np.minimum(pe, qe).sum()
    rate = (g["n"] == 1).mean()
    assert abs(rate - beta) < 5 * np.sqrt(beta * (1 - beta) / N)
    r = parity.run_oracle(b, 2024, 0)
    assert np.array_equal(g["n"], r.num_accepted) and np.array_equal(g["tokens"], r.tokens)


@pytest.mark.parametrize("name", ["b8_g4_v32000_t0.7", "b64_g5_v128256"])
def test_rows_with_maximum_near_zero(name):
    """Rows shifted so their maximum is -2^-20 (as log-probabilities of a confident model are): l - m
    rounds in float for nearly every column of such rows, so the sampler carries its rounding error."""
    b0 = synth.make_batch(name)

    def shifted_bf16(bits):
        x = synth.bf16_bits_to_f32(bits)
        return synth.to_bf16_bits((x - x.max(1, keepdims=True) - np.float32(2.0 ** -20)).astype(np.float32))

    b = synth.Batch(b0.workload, shifted_bf16(b0.target), shifted_bf16(b0.draft), b0.draft_tokens,
                    b0.seq_offsets, b0.gammas)
    m = synth.bf16_bits_to_f32(b.target).max(1)
    assert np.all(np.abs(m) < 2.0 ** -19)  # these rows take the carried-rounding path
    parity.assert_parity(b, 31, 2)


@pytest.mark.parametrize("name,B,V,f32", [("pointmass_b64_g5_v128256", None, None, False),
                                          ("pointmass_b64_g5_v128256", 7, 20001, False),
                                          ("pointmass_b64_g5_v128256", 5, 3000, True)])
def test_point_mass_drafts(name, B, V, f32):
    """Drafts without a draft distribution (an n-gram drafter's): no draft rows, q = point mass."""
    b = synth.make_batch(name, B=B, V=V)
    if f32:
        b.target = synth.bf16_bits_to_f32(b.target)
    assert b.draft is None
    d = parity.to_device(b)
    for step in range(3 if B is None else 5):
        g = parity.run_gpu(b, 1234, step, dev_in=d)
        parity.assert_parity(b, 1234, step, g=g)


def test_point_mass_gamma_zero_and_max():
    b = synth.make_batch("pointmass_b64_g5_v128256", B=5, V=4000, gammas=[0, 31, 3, 0, 31])
    for step in range(3):
        parity.assert_parity(b, 9, step)


@pytest.mark.parametrize("T", [0.3, 0.6, 1.7, 3.0])
def test_value_table_across_temperatures(T):
    """Batches large enough that the call builds the value table (>= 2048 sampler tasks), at temperatures
    that move its range (the largest row maximum it serves is min(63.75, 96 / K), K = log2(e) / T)."""
    w = synth.WORKLOADS["b64_g5_v128256"]
    wt = synth.Workload("b20_g5_v128256_t", 20, w.V, w.dtype, T, w.gamma, w.target_sigma, w.zipf_s, w.draft_scale,
                        w.draft_sigmas, seed=w.seed)
    b = synth.make_batch(wt)
    assert b.B * ((b.V + 1023) // 1024) >= 2048
    for step in range(3):
        parity.assert_parity(b, 42, step)


def test_value_table_and_exponential_draws_in_one_call():
    """Rows shifted so that some sequences' maxima lie above the value table's range (63.75) or below its
    floor (-63.75 + 60 / K): those draws take the precise exponential, the others the table, in one call."""
    b0 = synth.make_batch("b64_g5_v128256", B=24)

    def shifted(bits, shift):
        x = synth.bf16_bits_to_f32(bits) + np.float32(shift)
        return synth.to_bf16_bits(x.astype(np.float32))

    tgt, dft = b0.target.copy(), b0.draft.copy()
    for s in range(b0.B):
        shift = (70.0, -40.0, 0.0, 50.0)[s % 4]  # above the range, below the floor, inside, near the top
        t0, d0, g = int(b0.seq_offsets[s]) + s, int(b0.seq_offsets[s]), int(b0.gammas[s])
        tgt[t0:t0 + g + 1] = shifted(b0.target[t0:t0 + g + 1], shift)
        dft[d0:d0 + g] = shifted(b0.draft[d0:d0 + g], shift)
    b = synth.Batch(b0.workload, tgt, dft, b0.draft_tokens, b0.seq_offsets, b0.gammas)
    m = synth.bf16_bits_to_f32(b.target).max(1)
    assert m.max() > 63.75 and m.min() < -63.75 + 60 / 1.4426950408889634
    for step in range(3):
        parity.assert_parity(b, 8, step)
