"""Pins of the sharded oracle (CPU): over 1 to 4 vocabulary shards, the protocol of stats, decisions, sums and
the owner's scan gives exactly the unsharded oracle's outputs ("All About Transformer Inference", the
model-parallel sections: logits sharded over the vocabulary; the rule of velog "6-1편. Speculative
Decoding" §2-1/§2-2 unchanged); and the same protocol across two processes over a gloo group (exchange 1
and 2 all-gathers, exchange 3 a max all-reduce) gives the same outputs on both ranks."""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.shard import OracleShard, bounds_for
from speculative_decoding_verification_35_gb300 import synth
from speculative_decoding_verification_35_gb300.shard import local_steps


def shards_of(b, bounds):
    T = float(np.float32(b.temperature))
    return [OracleShard(j, bounds, b.target[:, bounds[j]:bounds[j + 1]],
                        None if b.draft is None or T == 0 else b.draft[:, bounds[j]:bounds[j + 1]],
                        b.draft_tokens, b.seq_offsets, b.gammas, b.V, T) for j in range(len(bounds) - 1)]


def unsharded(b, seed, step):
    return oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V,
                         float(np.float32(b.temperature)), seed, step)


CASES = [("b64_g5_v128256", 6, 2001), ("ragged_b128_v129280", 7, 1500), ("b8_g4_v32000_t0.7", 4, 999),
         ("b8_g4_v32000_greedy", 5, 777), ("b1_g4_v1024_f32", 1, 1024), ("pointmass_b64_g5_v128256", 5, 900)]


@pytest.mark.parametrize("name,B,V", CASES)
@pytest.mark.parametrize("S", [1, 2, 3, 4])
def test_sharded_protocol_equals_unsharded(name, B, V, S):
    b = synth.make_batch(name, B=B, V=V)
    bounds = bounds_for(V, S) if S != 3 else [0, V // 5, V // 2, V]  # uneven widths too
    for step in range(3):
        toks, n = local_steps(shards_of(b, bounds), 11, step)
        r = unsharded(b, 11, step)
        assert np.array_equal(n.numpy(), r.num_accepted), (step, n, r.num_accepted)
        assert np.array_equal(toks.numpy(), r.tokens), step


def test_sharded_errors_equal_unsharded():
    b = synth.make_batch("b8_g4_v32000_t0.7", B=4, V=600)
    b.draft_tokens[5] = 600       # sequence 1: bad token
    b.target[12, 400] = 0x7FC0    # sequence 2: NaN in the third shard's columns
    sh = shards_of(b, bounds_for(600, 3))
    toks, n = local_steps(sh, 1, 0)
    r = unsharded(b, 1, 0)
    assert np.array_equal(n.numpy(), r.num_accepted) and np.array_equal(toks.numpy(), r.tokens)
    assert all(s.status == r.status for s in sh) and r.status == (1 << 3) | (1 << 5)


def _gloo_rank(rank, world, path, name, B, V):
    import torch.distributed as dist
    from speculative_decoding_verification_35_gb300.shard import dist_exchange, step
    dist.init_process_group("gloo", init_method=f"file://{path}.store", rank=rank, world_size=world)
    b = synth.make_batch(name, B=B, V=V)
    bounds = bounds_for(V, world)
    sh = shards_of(b, bounds)[rank]
    gather, allmax = dist_exchange()
    outs = []
    for s in range(3):
        toks, n = step(sh, gather, allmax, 5, s)
        outs.append((toks.numpy().copy(), n.numpy().copy()))
    np.save(f"{path}.rank{rank}.npy", np.array(outs, dtype=object), allow_pickle=True)
    dist.destroy_process_group()


@pytest.mark.parametrize("name,B,V", [("b64_g5_v128256", 5, 3000), ("b8_g4_v32000_greedy", 4, 1000),
                                      ("pointmass_b64_g5_v128256", 3, 800)])
def test_sharded_protocol_over_gloo_world_size_2(tmp_path, name, B, V):
    import torch.multiprocessing as mp
    path = str(tmp_path / "shard")
    mp.start_processes(_gloo_rank, args=(2, path, name, B, V), nprocs=2, join=True, start_method="spawn")
    b = synth.make_batch(name, B=B, V=V)
    for rank in range(2):
        outs = np.load(f"{path}.rank{rank}.npy", allow_pickle=True)
        for s in range(3):
            r = unsharded(b, 5, s)
            assert np.array_equal(outs[s][1], r.num_accepted) and np.array_equal(outs[s][0], r.tokens), (rank, s)
