"""GPU: a batch verified as contiguous sequence ranges (spec_verify_range, each range with the global index
of its first sequence) gives, concatenated, the whole batch's outputs: tokens and counts equal the fp64
oracle's on the whole batch under the parity rule, as the whole-batch GPU call's do."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import oracle  # noqa: E402
from speculative_decoding_verification_35_gb300 import synth  # noqa: E402
from tests import parity  # noqa: E402
from tests.split import concat, ranges, sub_batch  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_35_gb300 import _build
    _build.build()
    oracle.build()


def run_range(b, seed, step, seq_base):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    d = parity.to_device(b)
    call = sv.Call(b.B, b.V, int(b.gammas.max()), b.R_t, b.R_d)
    rc = call.run(d["target"], d["draft"], d["draft_tokens"], d["seq_offsets"], d["gammas"], b.temperature, seed,
                  step, seq_base=seq_base)
    assert rc == sv.SV_OK
    torch.cuda.synchronize()
    return call.out_tokens.cpu().numpy(), call.out_n.cpu().numpy(), call.status_bits()


@pytest.mark.parametrize("name,B,V,parts", [("b64_g5_v128256", None, None, 2), ("b64_g5_v128256", 13, 20000, 3),
                                            ("ragged_b128_v129280", 17, 9000, 3),
                                            ("pointmass_b64_g5_v128256", 11, 5000, 2),
                                            ("b8_g4_v32000_greedy", None, None, 3), ("b1_g4_v1024_f32", 3, 777, 3)])
def test_ranges_equal_the_whole_batch(name, B, V, parts):
    b = synth.make_batch(name, B=B, V=V)
    for step in range(2):
        outs, st = [], 0
        for s0, s1 in ranges(b.B, parts):
            t, n, s = run_range(sub_batch(b, s0, s1), 1234, step, s0)
            outs.append((t, n))
            st |= s
        toks, n = concat(outs)
        g = dict(tokens=toks, n=n, status=st)
        parity.assert_parity(b, 1234, step, g=g, check_debug=False)
        whole = parity.run_gpu(b, 1234, step, debug=False)
        parity.assert_parity(b, 1234, step, g=whole, check_debug=False)
