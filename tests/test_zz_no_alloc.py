"""The allocation-free entry point (spec_verify_noalloc) against the workspace entry point (GPU).

Callers that cannot allocate device memory use spec_verify_noalloc, whose scratch is a fixed array
inside the library. Through the C ABI, two consecutive calls must give exactly the tokens and counts
that spec_verify_ex gives for the same arguments (the parity tolerance of the token path is exact
equality), and a batch larger than the fixed scratch must be refused before anything runs.
This file is collected last so that a failure here never hides the other GPU tests.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_35_gb300 import _build
    _build.build()
    from speculative_decoding_verification_35_gb300 import specverify
    return specverify


def _args(b, d, out_t, out_n, status, stream):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    return dict(target_logits=d["target"].data_ptr(),
                draft_logits=d["draft"].data_ptr() if d["draft"] is not None else None,
                dtype=sv.dtype_code(d["target"]), draft_tokens=d["draft_tokens"].data_ptr(),
                seq_offsets=d["seq_offsets"].data_ptr(), gammas=d["gammas"].data_ptr(), B=b.B, V=b.V,
                max_gamma=int(b.gammas.max()), temperature=b.temperature, out_tokens=out_t.data_ptr(),
                out_num_accepted=out_n.data_ptr(), device_status=status.data_ptr(), debug=None,
                cuda_stream=stream.cuda_stream)


@pytest.mark.parametrize("name", ["b64_g5_v128256", "ragged_b128_v129280", "b8_g4_v32000_greedy"])
def test_noalloc_matches_workspace_entry_point_twice(sv, name):
    from speculative_decoding_verification_35_gb300 import synth
    from tests import parity
    b = synth.make_batch(name)
    d = parity.to_device(b)
    stream = torch.cuda.current_stream()
    ws_bytes = sv.spec_verify_workspace_size(b.B, b.V, int(b.gammas.max()))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for step in (3, 4):  # two calls in a row, each checked against the workspace form
        ref_t = torch.full((b.R_t,), -9, dtype=torch.int32, device="cuda")
        ref_n = torch.full((b.B,), -9, dtype=torch.int32, device="cuda")
        ref_s = torch.zeros(1, dtype=torch.int32, device="cuda")
        a = _args(b, d, ref_t, ref_n, ref_s, stream)
        rc = sv.spec_verify_ex(seed=1234, step=step, workspace=ws.data_ptr(), workspace_bytes=ws_bytes, **a)
        assert rc == sv.SV_OK
        got_t = torch.full((b.R_t,), -9, dtype=torch.int32, device="cuda")
        got_n = torch.full((b.B,), -9, dtype=torch.int32, device="cuda")
        got_s = torch.zeros(1, dtype=torch.int32, device="cuda")
        a = _args(b, d, got_t, got_n, got_s, stream)
        rc = sv.spec_verify_noalloc(seed=1234, step=step, **a)
        assert rc == sv.SV_OK, sv.spec_verify_status_string(rc)
        torch.cuda.synchronize()
        assert int(ref_s.item()) == 0 and int(got_s.item()) == 0
        np.testing.assert_array_equal(got_n.cpu().numpy(), ref_n.cpu().numpy())
        np.testing.assert_array_equal(got_t.cpu().numpy(), ref_t.cpu().numpy())


def test_noalloc_refuses_batches_beyond_its_scratch(sv):
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = sv.spec_verify_noalloc(fake, fake, sv.SV_BF16, fake, fake, fake, 4096, 152064, 31, 1.0, 1, 0, fake, fake,
                                None, None, None)
    assert rc == sv.SV_ERR_WORKSPACE
