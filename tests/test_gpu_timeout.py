"""The bounded waits between warps give up cleanly (GPU, through the C ABI).

Every wait of one warp on another's word inside the verify launch is bounded. A call whose debug struct
asks for a spin limit of one poll makes nearly every such wait run out while the launch is under way:
the kernel must still return (no hang), set SV_ERR_TIMEOUT, and leave every sequence either failed the
documented way (n = -1, every slot -1) or exactly as the oracle verifies it (a sequence none of whose
waits ran out). The context stays usable: a normal call right after gives oracle parity. No fault is
injected: the waits simply stop early.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import oracle  # noqa: E402
from speculative_decoding_verification_35_gb300 import synth  # noqa: E402
from tests import parity  # noqa: E402

TIMEOUT_BIT = 1 << 7


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_35_gb300 import _build
    _build.build()
    oracle.build()


@pytest.mark.parametrize("name,B,V", [("b64_g5_v128256", None, None), ("pointmass_b64_g5_v128256", None, None),
                                      ("ragged_b128_v129280", 9, 20000), ("b8_g4_v32000_greedy", None, None),
                                      ("b1_g4_v1024_f32", None, None), ("b64_g5_v128256", 400, 2048)])
def test_waits_that_run_out_fail_their_sequences(name, B, V):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    b = synth.make_batch(name, B=B, V=V)
    d = parity.to_device(b)
    call = sv.Call(b.B, b.V, int(b.gammas.max()), b.R_t, b.R_d, debug=True)
    call.dbg_struct.spin_limit = 1
    r = parity.run_oracle(b, 1234, 3)
    for rep in range(2):
        call.out_tokens.fill_(-9)
        call.out_n.fill_(-9)
        rc = call.run(d["target"], d["draft"], d["draft_tokens"], d["seq_offsets"], d["gammas"], b.temperature,
                      1234, 3)
        assert rc == sv.SV_OK
        torch.cuda.synchronize()  # the launch returned
        st = call.status_bits()
        assert st & ~TIMEOUT_BIT == 0, st
        g_t, g_n = call.out_tokens.cpu().numpy(), call.out_n.cpu().numpy()
        failed = 0
        for s in range(b.B):
            t0, gm = int(b.seq_offsets[s]) + s, int(b.gammas[s])
            slots = g_t[t0:t0 + gm + 1]
            if g_n[s] == -1:
                assert np.all(slots == -1), (s, slots)
                failed += 1
            else:
                assert g_n[s] == r.num_accepted[s] and np.array_equal(slots, r.tokens[t0:t0 + gm + 1]), s
        assert (failed > 0) == bool(st & TIMEOUT_BIT)
        if name in ("b64_g5_v128256", "pointmass_b64_g5_v128256") and B is None:
            # full-size sampled batches: decisions and sampler tasks start while the statistics stream, so
            # one-poll waits surely run out (greedy and fp32 batches decide after streaming their own tasks,
            # when their words may all be in)
            assert st & TIMEOUT_BIT and failed > 0
    # a normal call right after, with the library's own bound: parity, status clean
    call.dbg_struct.spin_limit = 0
    g = parity.run_gpu(b, 1234, 3, dev_in=d, debug=True)
    parity.assert_parity(b, 1234, 3, g=g, r=r)
