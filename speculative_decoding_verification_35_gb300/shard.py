"""The vocabulary-sharded verify step: one shard's device state and the exchange protocol.

A tensor-parallel model's unembedding leaves every logit row sharded over the vocabulary ("All About
Transformer Inference", the model-parallel sections; "Accelerating Sonar through speculation", the
tensor-parallel scheduling section). ``CudaShard`` holds one shard's slices and runs the four C-ABI calls
(``spec_shard_stats``, ``_decide``, ``_sums``, ``_finish``); ``step`` strings them together with the three
exchanges between shards, taken as two functions so that the same protocol runs over a process group
(``dist_exchange``: all-gathers and one max all-reduce, NCCL for device tensors) or over shards
held by one process (``local_steps``). Marshalling only: every step of the verify rule runs in the
library's kernels.
"""
from __future__ import annotations

from . import specverify as sv

PARTIAL_WORDS = 4  # sv_shard_partial: 16 bytes
DRAW_WORDS = 8     # sv_shard_draw: 32 bytes
SUM_WORDS = 8      # four float pairs per sequence and chunk


class CudaShard:
    """Shard `shard` of `bounds` (S + 1 columns): its slices target [R_t, Vs] and draft [R_d, Vs] (None in greedy
    mode or for point-mass drafts), the batch's draft tokens / offsets / gammas, and its output buffers."""

    def __init__(self, shard, bounds, target, draft, draft_tokens, seq_offsets, gammas, B, V, max_gamma, R_t, R_d,
                 temperature, device=None):
        import torch
        self.torch = torch
        self.shard, self.bounds, self.S = shard, list(bounds), len(bounds) - 1
        self.v0, self.Vs = int(bounds[shard]), int(bounds[shard + 1] - bounds[shard])
        assert target.shape[1] == self.Vs and (draft is None or draft.shape[1] == self.Vs)
        self.target, self.draft = target, draft
        self.tokens, self.offs, self.gammas = draft_tokens, seq_offsets, gammas
        self.B, self.V, self.max_gamma, self.R_t, self.R_d = B, V, max_gamma, R_t, R_d
        self.T = temperature
        self.point_mass = temperature > 0 and draft is None
        self.rows = R_t if temperature == 0 or draft is None else R_t + R_d
        dev = target.device if device is None else device
        i32 = torch.int32
        self.partials = torch.zeros((self.rows, PARTIAL_WORDS), dtype=i32, device=dev)
        self.draws = torch.zeros((B, DRAW_WORDS), dtype=i32, device=dev)
        self.nc = sv.spec_shard_chunks(self.S, self.bounds)
        if self.nc < 1:
            raise ValueError(f"invalid shard bounds {self.bounds}")
        self.sums = torch.zeros((B, self.nc * SUM_WORDS), dtype=torch.float32, device=dev)
        self.out_tokens = torch.full((R_t,), -1, dtype=i32, device=dev)
        self.out_n = torch.full((B,), -1, dtype=i32, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)
        self.dtype = sv.dtype_code(target)

    def _st(self, stream):
        return (stream if stream is not None else self.torch.cuda.current_stream()).cuda_stream

    def stats(self, stream=None):
        p = sv._ptr
        rc = sv.spec_shard_stats(p(self.target), p(self.draft) if self.T > 0 else None, self.dtype, p(self.tokens),
                                 p(self.offs), p(self.gammas), self.B, self.V, self.v0, self.Vs, self.max_gamma,
                                 self.T, p(self.partials), p(self.status), self._st(stream))
        if rc != sv.SV_OK:
            raise RuntimeError(sv.spec_verify_status_string(rc))
        return self.partials

    def decide(self, all_partials, seed, step, stream=None):
        p = sv._ptr
        rc = sv.spec_shard_decide(p(all_partials), self.S, self.bounds, p(self.tokens), p(self.offs), p(self.gammas),
                                  self.B, self.V, self.max_gamma, self.T, self.point_mass, seed, step,
                                  p(self.out_tokens), p(self.out_n), p(self.draws), p(self.status), self._st(stream))
        if rc != sv.SV_OK:
            raise RuntimeError(sv.spec_verify_status_string(rc))

    def draw_sums(self, stream=None):
        p = sv._ptr
        rc = sv.spec_shard_sums(self.shard, self.S, self.bounds, p(self.target), p(self.draft), self.dtype,
                                p(self.draws), p(self.offs), self.B, self.V, self.T, p(self.sums), self._st(stream))
        if rc != sv.SV_OK:
            raise RuntimeError(sv.spec_verify_status_string(rc))
        return self.sums

    def finish(self, all_sums, stream=None):
        p = sv._ptr
        rc = sv.spec_shard_finish(self.shard, self.S, self.bounds, p(self.target), p(self.draft), self.dtype,
                                  p(self.draws), p(all_sums), p(self.offs), self.B, self.V, self.T, p(self.out_tokens),
                                  self._st(stream))
        if rc != sv.SV_OK:
            raise RuntimeError(sv.spec_verify_status_string(rc))
        return self.out_tokens


def step(shard, gather, allmax, seed, step_index):
    """One verify step of one shard: statistics, exchange 1 (gather), decisions, sums, exchange 2 (gather),
    finish, exchange 3 (max of the drawn slot). gather(t) -> [S, *t.shape]; allmax(t) -> the element-wise max
    over the shards. Returns (out_tokens, out_num_accepted) after the last exchange."""
    all_partials = gather(shard.stats())
    shard.decide(all_partials, seed, step_index)
    all_sums = gather(shard.draw_sums())
    tokens = allmax(shard.finish(all_sums))
    return tokens, shard.out_n


def dist_exchange(group=None):
    """(gather, allmax) over a torch.distributed process group (rank j holds shard j)."""
    import torch
    import torch.distributed as dist

    def gather(t):
        parts = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
        dist.all_gather(parts, t.contiguous(), group=group)
        return torch.stack(parts)

    def allmax(t):
        t = t.clone()
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
        return t

    return gather, allmax


def local_steps(shards, seed, step_index):
    """The protocol for shards held by one process (all on one device): each exchange is a stack of the
    shards' records. Returns (out_tokens, out_num_accepted) (identical on every shard)."""
    import torch
    allp = torch.stack([sh.stats() for sh in shards])
    for sh in shards:
        sh.decide(allp, seed, step_index)
    alls = torch.stack([sh.draw_sums() for sh in shards])
    toks = torch.stack([sh.finish(alls) for sh in shards]).max(0).values
    return toks, shards[0].out_n
