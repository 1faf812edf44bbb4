"""Sequence ranges of one batch (multi-GPU by sequence): verifying contiguous ranges
separately, each with the global index of its first sequence (oracle seq_base), and concatenating the
outputs equals verifying the whole batch, since a sequence's draws depend only on its own rows and on its
global index. In one process, and across two gloo processes exchanging the ranges' outputs."""
import os

import numpy as np
import pytest

import oracle
from speculative_decoding_verification_35_gb300 import synth
from tests.split import concat, ranges, sub_batch

CASES = [("ragged_b128_v129280", 13, 300), ("b8_g4_v32000_greedy", 7, 256),
         ("pointmass_b64_g5_v128256", 9, 300), ("b1_g4_v1024_f32", 1, 64)]


def run(b, seed, step, seq_base=0):
    r = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, b.temperature, seed, step,
                      nthreads=2, seq_base=seq_base)
    return r


@pytest.mark.parametrize("name,B,V", CASES)
@pytest.mark.parametrize("parts", [2, 3])
def test_ranges_with_their_global_index_equal_the_batch(name, B, V, parts):
    b = synth.make_batch(name, B=B, V=V)
    for step in range(3):
        whole = run(b, 21, step)
        outs = []
        for s0, s1 in ranges(b.B, parts):
            r = run(sub_batch(b, s0, s1), 21, step, seq_base=s0)
            assert r.status == whole.status == 0
            outs.append((r.tokens, r.num_accepted))
        toks, n = concat(outs)
        np.testing.assert_array_equal(toks, whole.tokens)
        np.testing.assert_array_equal(n, whole.num_accepted)


def test_the_global_index_keys_the_draws():
    # the same rows verified as the batch's sequence 5 draw other uniforms than as its sequence 0
    b = synth.make_batch("b8_g4_v32000_t0.7", B=1, V=300)
    diff = 0
    for step in range(40):
        r0, r5 = run(b, 3, step), run(b, 3, step, seq_base=5)
        diff += int(not (np.array_equal(r0.tokens, r5.tokens) and np.array_equal(r0.num_accepted, r5.num_accepted)))
    assert diff > 0


def _gloo_rank(rank, world, path, name, B, V):
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"file://{path}.store", rank=rank, world_size=world)
    b = synth.make_batch(name, B=B, V=V)
    s0, s1 = ranges(b.B, world)[rank]
    r = run(sub_batch(b, s0, s1), 21, 1, seq_base=s0)
    mine = torch.from_numpy(np.concatenate([r.tokens, r.num_accepted]).astype(np.int64))
    sizes = [None] * world
    dist.all_gather_object(sizes, int(mine.numel()))
    parts = [torch.zeros(n, dtype=torch.int64) for n in sizes]
    if len(set(sizes)) == 1:
        dist.all_gather(parts, mine)
    else:
        objs = [None] * world
        dist.all_gather_object(objs, mine.numpy())
        parts = [torch.from_numpy(o) for o in objs]
    if rank == 0:
        outs = []
        for (a, c), p in zip(ranges(b.B, world), parts):
            rt = int(b.seq_offsets[c] - b.seq_offsets[a]) + (c - a)
            outs.append((p[:rt].numpy(), p[rt:].numpy()))
        toks, n = concat(outs)
        whole = run(b, 21, 1)
        np.save(f"{path}.ok.npy", np.array([np.array_equal(toks, whole.tokens) and
                                            np.array_equal(n, whole.num_accepted)]))
    dist.destroy_process_group()


def test_ranges_over_gloo_world_size_2(tmp_path):
    import torch.multiprocessing as mp
    path = str(tmp_path / "range")
    mp.start_processes(_gloo_rank, args=(2, path, "ragged_b128_v129280", 11, 300), nprocs=2, join=True,
                       start_method="spawn")
    assert bool(np.load(f"{path}.ok.npy")[0])
