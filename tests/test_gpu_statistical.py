"""The mismatch quota at full vocabulary size, on enough draws to bound it (GPU, through the C ABI).

The contract: token ids and accepted counts equal the oracle's, except on draws whose uniform lies within
1e-6 of an oracle decision boundary; such band draws are counted and must stay below 1e-5 of the draws.
Zero mismatches over N draws bounds the rate below about 3/N, so each workload here verifies at least
2 x 10^5 token draws (and about four times as many uniform draws, counting the accept tests): one batch
per workload at its full size, verified for many consecutive steps (each step a different set of uniforms),
against the oracle's multi-step entry (the same rule on the same probabilities, step by step).
The counts are printed for the record.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import oracle  # noqa: E402
from speculative_decoding_verification_35_gb300 import synth  # noqa: E402
from tests import parity  # noqa: E402

TOKEN_DRAWS = 200_000


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_35_gb300 import _build
    _build.build()
    oracle.build()


def gpu_steps(b, d, seed, step0, steps):
    """`steps` consecutive verify calls on one batch, each writing its own output rows."""
    from speculative_decoding_verification_35_gb300 import specverify as sv
    mg = int(b.gammas.max())
    ws_bytes = sv.spec_verify_workspace_size(b.B, b.V, mg)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_t = torch.full((steps, b.R_t), -9, dtype=torch.int32, device="cuda")
    out_n = torch.full((steps, b.B), -9, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    dt = sv.dtype_code(d["target"])
    for s in range(steps):
        rc = sv.spec_verify_ex(d["target"].data_ptr(), d["draft"].data_ptr() if d["draft"] is not None else None,
                               dt, d["draft_tokens"].data_ptr(), d["seq_offsets"].data_ptr(), d["gammas"].data_ptr(),
                               b.B, b.V, mg, b.temperature, seed, step0 + s, out_t[s].data_ptr(), out_n[s].data_ptr(),
                               st.data_ptr(), ws.data_ptr(), ws_bytes, None, stream)
        assert rc == sv.SV_OK
    torch.cuda.synchronize()
    return out_t.cpu().numpy(), out_n.cpu().numpy(), int(st.item()) & 0xFFFFFFFF


@pytest.mark.parametrize("name", ["b64_g5_v128256", "b256_g3_v152064_t0.8", "ragged_b128_v129280",
                                  "pointmass_b64_g5_v128256"])
def test_mismatch_quota_over_many_draws(name):
    b = synth.make_batch(name)
    d = parity.to_device(b)
    steps = -(-TOKEN_DRAWS // b.B)
    seed, step0 = 4321, 10_000
    g_t, g_n, g_st = gpu_steps(b, d, seed, step0, steps)
    r_t, r_n, r_st = oracle.verify_steps(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V,
                                         parity.t32(b.temperature), seed, step0, steps)
    r0 = parity.run_oracle(b, seed, step0)
    assert g_st == r_st == 0
    rep = parity.compare_steps(b, g_t, g_n, r_t, r_n, r0, seed, step0)
    print(f"{name}: steps {steps}, token draws {rep['token_draws']}, uniform draws {rep['draws']}, "
          f"band {len(rep['band'])}, mismatch {len(rep['bad'])}")
    assert rep["token_draws"] >= TOKEN_DRAWS
    assert not rep["bad"], rep["bad"][:5]
    assert len(rep["band"]) < 1e-5 * rep["draws"], rep["band"][:5]
