"""Pins of the token-tree verification oracle (CPU).

Candidates without a draft distribution (EAGLE-style top-K tokens, "Accelerating Sonar through
speculation", §"EAGLE") are point masses; the children of the current node are tried in order with
velog "6-1편. Speculative Decoding" §2-1's rule on p restricted to the tokens not yet rejected. Pinned by
hand-worked probabilities, by exact equality with the linear point-mass verify on chain trees, and by
the law that makes it lossless: the first emitted token is distributed as p_root (10^6 trials)."""
import numpy as np
from scipy.stats import chi2

import oracle
from speculative_decoding_verification_35_gb300 import synth


def test_hand_worked_two_children():
    # p_root = (0.6, 0.3, 0.1); children: node 1 (token 1), node 2 (token 0); both leaves
    p = [[0.6, 0.3, 0.1], [0.2, 0.5, 0.3], [0.3, 0.3, 0.4]]
    par, x = [0, 0], [1, 0]
    # u_1 < 0.3: token 1 accepted, then the leaf's row draws (u' = 0.5: 0.2 < 0.5 < 0.7 -> token 1)
    n, out, path = oracle.tree_probs(p, par, x, [0.29, 0.99], [0.0, 0.5, 0.0])
    assert (n, out.tolist(), path.tolist()) == (1, [1, 1, -1], [1, -1])
    # u_1 >= 0.3: token 1 removed; token 0 accepted iff u_2 * 0.7 < 0.6
    n, out, path = oracle.tree_probs(p, par, x, [0.31, 0.857], [0.0, 0.0, 0.0])
    assert (n, out.tolist(), path.tolist()) == (1, [0, 0, -1], [2, -1])
    # both rejected: drawn from p_root without tokens 1 and 0 -> token 2 (whatever u')
    n, out, path = oracle.tree_probs(p, par, x, [0.31, 0.858], [0.3, 0.0, 0.0])
    assert (n, out.tolist(), path.tolist()) == (0, [2, -1, -1], [-1, -1])


def test_duplicate_candidate_is_rejected_and_leaf_draws_from_p():
    p = [[0.5, 0.5], [0.9, 0.1], [0.1, 0.9]]
    # two children with the same token 1: the second is never accepted after the first is rejected
    n, out, path = oracle.tree_probs(p, [0, 0], [1, 1], [0.6, 0.0], [0.0, 0.0, 0.0])
    assert n == 0 and out[0] == 0  # token 1 removed: only token 0 remains


def test_chain_equals_linear_point_mass_verify():
    for name, B, V in [("pointmass_b64_g5_v128256", 12, 3000), ("ragged_b128_v129280", 9, 2000)]:
        b = synth.make_batch(name, B=B, V=V)
        parents = np.concatenate([np.arange(g, dtype=np.int32) for g in b.gammas])  # node j's parent j - 1
        for step in range(4):
            r = oracle.verify(b.target, None, b.draft_tokens, b.seq_offsets, b.gammas, b.V, 1.0, 42, step)
            t, n, path, st = oracle.verify_tree(b.target, b.draft_tokens, b.seq_offsets, b.gammas, parents, b.V,
                                                1.0, 42, step)
            assert st == r.status == 0
            assert np.array_equal(n, r.num_accepted) and np.array_equal(t, r.tokens)
            for s in range(b.B):  # the path of a chain is nodes 1..n
                d0 = int(b.seq_offsets[s])
                assert path[d0:d0 + n[s]].tolist() == list(range(1, n[s] + 1))


def test_tree_is_lossless_first_and_second_token():
    # 10^6 trees over V = 6: root with children (token 2, token 0, token 2, token 4), node 1 has children
    # (token 3, token 5); the first emitted token must follow p_root, and given that node 1 was accepted
    # the second must follow p_node1
    V, N = 6, 1_000_000
    rng = np.random.default_rng(17)
    ps = rng.dirichlet(np.ones(V), size=7) * 0.97 + 0.03 / V
    lg = np.log(ps).astype(np.float32)
    gam = 6
    tokens = np.array([2, 0, 2, 4, 3, 5], np.int32)
    parents = np.array([0, 0, 0, 0, 1, 1], np.int32)
    target = np.tile(lg, (N, 1))
    offs = (np.arange(N + 1) * gam).astype(np.int32)
    t, n, path, st = oracle.verify_tree(target, np.tile(tokens, N), offs, np.full(N, gam, np.int32),
                                        np.tile(parents, N), V, 1.0, 3, 0)
    assert st == 0
    pe = np.exp(lg.astype(np.float64)); pe /= pe.sum(axis=1, keepdims=True)
    first = t[0::gam + 1]
    cnt = np.bincount(first, minlength=V)
    stat = ((cnt - pe[0] * N) ** 2 / (pe[0] * N)).sum()
    assert chi2.sf(stat, V - 1) > 1e-4
    via1 = path[0::gam] == 1
    second = t[1::gam + 1][via1]
    c2 = np.bincount(second, minlength=V)
    stat2 = ((c2 - pe[1] * len(second)) ** 2 / (pe[1] * len(second))).sum()
    assert chi2.sf(stat2, V - 1) > 1e-4


def test_greedy_tree_and_bad_parent():
    V = 5
    lg = np.array([[0, 3, 1, 0, 0], [4, 0, 0, 0, 0], [0, 0, 0, 0, 9], [0, 2, 0, 0, 0]], np.float32)
    # root children: node 1 (token 0), node 2 (token 1 = argmax of the root); node 3 child of node 2 with
    # token 4 = argmax of node 2's row -> accepted; node 3 is a leaf: its argmax (1) is emitted
    t, n, path, st = oracle.verify_tree(lg, [0, 1, 4], [0, 3], [3], [0, 0, 2], V, 0.0, 0, 0)
    assert st == 0 and n.tolist() == [2] and t.tolist() == [1, 4, 1, -1] and path.tolist() == [2, 3, -1]
    t, n, path, st = oracle.verify_tree(lg, [0, 1, 4], [0, 3], [3], [0, 0, 3], V, 1.0, 0, 0)
    assert st == 1 << 4 and n.tolist() == [-1] and t.tolist() == [-1] * 4
