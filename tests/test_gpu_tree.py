"""GPU parity of token-tree verification (spec_verify_tree) against the oracle: random trees with
repeated candidates, chains (equal to linear point-mass verification), greedy trees, full-size rows and
a bad parent."""
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


def _trees(B, V, gmax, seed, f32=False, chain=False):
    t = synth.make_tree_batch(B, V, gmax, seed, f32=f32, chain=chain)
    return t.target, t.draft_tokens, t.parents, t.seq_offsets, t.gammas


def _gpu_tree(target, tokens, parents, offs, gam, V, T, seed, step):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    B = len(gam)
    R_d, R_t = int(offs[-1]), int(offs[-1]) + B
    mg = int(gam.max()) if B else 0
    if target.dtype == np.uint16:
        tg = torch.from_numpy(target.view(np.int16)).view(torch.bfloat16).cuda(); dt = sv.SV_BF16
    else:
        tg = torch.from_numpy(target).cuda(); dt = sv.SV_F32
    d = {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.int32)).cuda()
         for k, v in dict(t=tokens if R_d else np.zeros(1), p=parents if R_d else np.zeros(1), o=offs, g=gam).items()}
    ws_bytes = sv.spec_verify_workspace_size(B, V, mg)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    out = torch.full((R_t,), -7, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    path = torch.full((max(R_d, 1),), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = sv.spec_verify_tree(tg.data_ptr(), dt, d["t"].data_ptr(), d["p"].data_ptr(), d["o"].data_ptr(), d["g"].data_ptr(),
                             B, V, mg, T, seed, step, out.data_ptr(), n.data_ptr(), path.data_ptr(), st.data_ptr(),
                             ws.data_ptr(), ws_bytes, torch.cuda.current_stream().cuda_stream)
    assert rc == sv.SV_OK, sv.spec_verify_status_string(rc)
    torch.cuda.synchronize()
    return out.cpu().numpy(), n.cpu().numpy(), path.cpu().numpy()[:R_d], int(st.item()) & 0xFFFFFFFF


@pytest.mark.parametrize("B,V,gmax,T,f32", [(16, 3000, 31, 1.0, False), (40, 1001, 12, 0.7, False),
                                             (9, 777, 20, 1.0, True), (64, 128256, 15, 1.0, False)])
def test_random_trees_match_oracle(B, V, gmax, T, f32):
    target, tokens, parents, offs, gam = _trees(B, V, gmax, seed=B * 7 + gmax, f32=f32)
    for step in range(4 if B < 64 else 2):
        g = _gpu_tree(target, tokens, parents, offs, gam, V, T, 77, step)
        r = oracle.verify_tree(target, tokens, offs, gam, parents, V, float(np.float32(T)), 77, step)
        assert g[3] == r[3] == 0
        assert np.array_equal(g[1], r[1]), (g[1], r[1])
        assert np.array_equal(g[0], r[0])
        assert np.array_equal(g[2], r[2])


def test_chain_trees_equal_linear_point_mass_verify():
    from speculative_decoding_verification_35_gb300 import specverify as sv
    target, tokens, parents, offs, gam = _trees(12, 5000, 8, seed=5, chain=True)
    B, V = len(gam), 5000
    for step in range(3):
        out, n, path, st = _gpu_tree(target, tokens, parents, offs, gam, V, 1.0, 11, step)
        b = synth.Batch(synth.WORKLOADS["pointmass_b64_g5_v128256"], target, None, tokens, offs, gam)
        g = parity.run_gpu(b, 11, step, debug=False)
        assert st == 0 and np.array_equal(n, g["n"]) and np.array_equal(out, g["tokens"])


def test_greedy_trees_match_oracle():
    target, tokens, parents, offs, gam = _trees(20, 2000, 10, seed=9)
    g = _gpu_tree(target, tokens, parents, offs, gam, 2000, 0.0, 0, 0)
    r = oracle.verify_tree(target, tokens, offs, gam, parents, 2000, 0.0, 0, 0)
    assert g[3] == r[3] == 0
    assert np.array_equal(g[0], r[0]) and np.array_equal(g[1], r[1]) and np.array_equal(g[2], r[2])
    assert (r[1] > 0).any()  # some candidates are accepted


def test_bad_parent_fails_only_its_tree():
    from speculative_decoding_verification_35_gb300 import specverify as sv
    target, tokens, parents, offs, gam = _trees(6, 900, 6, seed=13)
    b_bad = int(np.argmax(gam >= 2))
    parents = parents.copy()
    parents[int(offs[b_bad]) + 1] = 5  # node 2's parent must lie in [0, 2)
    g = _gpu_tree(target, tokens, parents, offs, gam, 900, 1.0, 3, 0)
    r = oracle.verify_tree(target, tokens, offs, gam, parents, 900, 1.0, 3, 0)
    assert g[3] == r[3] == 1 << sv.SV_ERR_BAD_OFFSETS
    assert g[1][b_bad] == -1 and np.array_equal(g[1], r[1]) and np.array_equal(g[0], r[0])
