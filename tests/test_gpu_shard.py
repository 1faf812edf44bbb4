"""GPU parity of the vocabulary-sharded verify step (spec_shard_*) against the unsharded fp64 oracle.

The shards of one batch run on one GPU as separate shard objects, each holding its own contiguous slice of
every row; the three exchanges are stacks of the shards' records (the protocol a tensor-parallel group runs
over NCCL, exercised across processes by the gloo test of the sharded oracle). Tokens and counts must equal
the unsharded oracle's under the usual rule (exact except draws within 1e-6 of a boundary, counted).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import oracle  # noqa: E402
from oracle.shard import bounds_for  # noqa: E402
from speculative_decoding_verification_35_gb300 import synth  # noqa: E402
from tests import parity  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_35_gb300 import _build
    _build.build()
    oracle.build()


def cuda_shards(b, bounds):
    from speculative_decoding_verification_35_gb300.shard import CudaShard
    d = parity.to_device(b)
    T = float(np.float32(b.temperature))
    out = []
    for j in range(len(bounds) - 1):
        lo, hi = bounds[j], bounds[j + 1]
        tgt = d["target"][:, lo:hi].contiguous()
        dft = None if d["draft"] is None or T == 0 else d["draft"][:, lo:hi].contiguous()
        out.append(CudaShard(j, bounds, tgt, dft, d["draft_tokens"], d["seq_offsets"], d["gammas"], b.B, b.V,
                             int(b.gammas.max()), b.R_t, b.R_d, T))
    return out


def check(b, bounds, seed, steps):
    from speculative_decoding_verification_35_gb300.shard import local_steps
    shards = cuda_shards(b, bounds)
    tot = dict(draws=0, band=0)
    for step in range(steps):
        toks, n = local_steps(shards, seed, step)
        torch.cuda.synchronize()
        st = int(shards[0].status.item()) & 0xFFFFFFFF
        assert all(int(s.status.item()) & 0xFFFFFFFF == st for s in shards)
        g = dict(tokens=toks.cpu().numpy(), n=n.cpu().numpy(), status=st)
        rep = parity.assert_parity(b, seed, step, g=g, check_debug=False)
        tot["draws"] += rep["draws"]
        tot["band"] += len(rep["band"])
    return tot


@pytest.mark.parametrize("S", [2, 4])
@pytest.mark.parametrize("name,B,V", [("b64_g5_v128256", None, None), ("ragged_b128_v129280", 17, 20000),
                                      ("b8_g4_v32000_t0.7", None, None), ("b8_g4_v32000_greedy", None, None),
                                      ("b1_g4_v1024_f32", None, None), ("pointmass_b64_g5_v128256", 9, 30001)])
def test_sharded_verify_matches_unsharded_oracle(name, B, V, S):
    b = synth.make_batch(name, B=B, V=V)
    tot = check(b, bounds_for(b.V, S), 77, 3)
    print(name, S, tot)


def test_uneven_shards_and_error_paths():
    b = synth.make_batch("b8_g4_v32000_t0.7", B=5, V=3001)
    check(b, [0, 17, 1500, 2999, 3001], 3, 2)
    bad = synth.make_batch("b8_g4_v32000_t0.7", B=5, V=3001)
    bad.draft_tokens[6] = 3001                   # sequence 1: bad token
    bad.target[12, 2000] = 0x7FC0                # sequence 2: NaN in the third shard's slice
    check(bad, bounds_for(3001, 3), 3, 1)
    off = synth.make_batch("b8_g4_v32000_t0.7", B=4, V=500)
    off.seq_offsets[2] = 1000                    # inconsistent offsets: every sequence fails, no row read
    from speculative_decoding_verification_35_gb300.shard import local_steps
    shards = cuda_shards(off, bounds_for(500, 2))
    toks, n = local_steps(shards, 1, 0)
    torch.cuda.synchronize()
    assert np.all(n.cpu().numpy() == -1) and int(shards[0].status.item()) == 1 << 4


def test_one_shard_equals_the_unsharded_library():
    b = synth.make_batch("b64_g5_v128256", B=8, V=20000)
    tot = check(b, [0, b.V], 5, 3)
    assert tot["band"] == 0
