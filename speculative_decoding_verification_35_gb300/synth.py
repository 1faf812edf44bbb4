"""Seeded synthetic logit batches shaped like the verify-step workloads.

This module is the one piece shared by the CUDA path's tests/bench and the CPU oracle. It holds none
of the verify step's arithmetic: it draws logits (Gaussian noise plus a Zipf log-prior over the
vocabulary index), rounds them once to the kernel dtype, and draws the draft tokens from the draft
distribution with the Gumbel-max trick (argmax of l/T + Gumbel noise), which samples softmax(l/T)
exactly by a different route than the verify step's inverse CDF. Greedy workloads take the draft's
argmax as its token. All randomness comes from numpy's PCG64 with per-workload seeds.

Point-mass workloads stand in for a drafter without a draft distribution (an n-gram drafter, velog
"6-1편. Speculative Decoding", §"drafter types": it proposes the tokens that followed an earlier occurrence
of the last n tokens). Each draft slot gets a planted next token whose target logit is raised by `boost`;
the drafter proposes it with probability `hit`, else a uniform token. No draft rows exist.

No dataset is used: the pages measure nothing on the verify step itself, and these synthetic batches
stand in for the decode batches the pages describe (draft model proposes gamma tokens, target scores
gamma + 1 positions; "Accelerating Sonar through speculation", §"Speculative decoding" steps 2-4).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32, BF16 = "f32", "bf16"


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    V: int
    dtype: str
    temperature: float
    gamma: int | None            # fixed gamma, or None for the ragged U{gamma_lo..gamma_hi} draw
    target_sigma: float
    zipf_s: float                # 0: no prior
    draft_scale: float           # draft = draft_scale * target + N(0, draft_sigma^2)
    draft_sigmas: tuple          # per-sequence sigma cycle (b mod len)
    gamma_lo: int = 1
    gamma_hi: int = 8
    seed: int = 0
    tags: tuple = field(default_factory=tuple)
    point_mass: bool = False     # drafts without a draft distribution (q = point mass), no draft rows
    boost: float = 0.0           # point mass: raise of the planted token's target logit
    hit: float = 0.0             # point mass: probability that the draft is the planted token

    @property
    def greedy(self) -> bool:
        return self.temperature == 0.0


# Workloads named by what they are. The seeds only make each workload's draw distinct.
WORKLOADS = {
    w.name: w for w in [
        Workload("b1_g4_v1024_f32", 1, 1024, F32, 1.0, 4, 2.0, 0.0, 1.0, (0.5,), seed=1000),
        Workload("b8_g4_v32000_t0.7", 8, 32000, BF16, 0.7, 4, 3.0, 1.1, 0.9, (1.0,), seed=2000),
        Workload("b8_g4_v32000_greedy", 8, 32000, BF16, 0.0, 4, 3.0, 1.1, 0.9, (1.0,), seed=2000),
        Workload("b64_g5_v128256", 64, 128256, BF16, 1.0, 5, 2.5, 1.1, 1.0, (0.3, 1.0, 2.0), seed=3000),
        Workload("b256_g3_v152064_t0.8", 256, 152064, BF16, 0.8, 3, 2.0, 1.05, 1.0, (0.8,), seed=4000),
        Workload("ragged_b128_v129280", 128, 129280, BF16, 1.0, None, 2.0, 1.1, 1.0, (1.0,), seed=5000),
        Workload("pointmass_b64_g5_v128256", 64, 128256, BF16, 1.0, 5, 2.5, 1.1, 0.0, (0.0,), seed=6000,
                 point_mass=True, boost=9.0, hit=0.8),
    ]
}

# The workload the headline throughput is quoted on.
HEADLINE = "b64_g5_v128256"


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (round to nearest even, via float32) and return the raw 16-bit codes."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Batch:
    workload: Workload
    target: np.ndarray           # [R_t, V] float32, or uint16 raw bf16 codes
    draft: np.ndarray | None     # [R_d, V], same dtype as target (None only when R_d == 0)
    draft_tokens: np.ndarray     # [R_d] int32
    seq_offsets: np.ndarray      # [B+1] int32, prefix sum of gammas over draft rows
    gammas: np.ndarray           # [B] int32

    @property
    def B(self):
        return len(self.gammas)

    @property
    def V(self):
        return int(self.target.shape[1])

    @property
    def R_t(self):
        return int(self.seq_offsets[-1]) + self.B

    @property
    def R_d(self):
        return int(self.seq_offsets[-1])

    @property
    def temperature(self):
        return self.workload.temperature

    @property
    def elem_bytes(self):
        return 2 if self.workload.dtype == BF16 else 4

    def logits_f32(self, which: str) -> np.ndarray:
        a = self.target if which == "target" else self.draft
        return bf16_bits_to_f32(a) if self.workload.dtype == BF16 else a

    def algorithmic_bytes(self) -> int:
        """Bytes the verify step must move at least: every logit it needs read once, plus the
        small index arrays and outputs."""
        rows = self.verified_rows()
        return (rows * self.V * self.elem_bytes + 4 * self.R_d + 4 * (self.B + 1) + 4 * self.B
                + 4 * self.R_t + 4 * self.B)

    def verified_rows(self) -> int:
        return self.R_t if self.workload.greedy or self.draft is None else self.R_t + self.R_d


def _rows(rng, n, V, sigma, zipf_s):
    prior = -zipf_s * np.log(np.arange(1, V + 1, dtype=np.float64)) if zipf_s else 0.0
    return rng.normal(0.0, sigma, size=(n, V)) + prior


def make_batch(name_or_w, B: int | None = None, V: int | None = None, gammas=None,
               seed_offset: int = 0) -> Batch:
    """Draw one batch. ``B``/``V``/``gammas`` override the workload's sizes (smaller parity cases
    with the same value distributions); ``seed_offset`` selects another independent draw."""
    w = WORKLOADS[name_or_w] if isinstance(name_or_w, str) else name_or_w
    B = w.B if B is None else B
    V = w.V if V is None else V
    rng = np.random.Generator(np.random.PCG64(w.seed + seed_offset))
    if gammas is None:
        if w.gamma is None:
            gammas = rng.integers(w.gamma_lo, w.gamma_hi + 1, size=B)
        else:
            gammas = np.full(B, w.gamma)
    gammas = np.asarray(gammas, dtype=np.int32)
    offs = np.zeros(B + 1, dtype=np.int32)
    offs[1:] = np.cumsum(gammas)
    R_d = int(offs[-1])
    R_t = R_d + B
    out_dtype = np.uint16 if w.dtype == BF16 else np.float32
    target = np.empty((R_t, V), dtype=out_dtype)
    draft = np.empty((R_d, V), dtype=out_dtype)
    tokens = np.zeros(R_d, dtype=np.int32)
    tok_rng = np.random.Generator(np.random.PCG64(w.seed + seed_offset + 7))
    for b in range(B):
        g = int(gammas[b])
        d0 = int(offs[b])
        t0 = d0 + b
        t64 = _rows(rng, g + 1, V, w.target_sigma, w.zipf_s)
        if w.point_mass:
            planted = tok_rng.integers(0, min(V, 1024), size=g)
            t64[np.arange(g), planted] += w.boost
            guess = np.where(tok_rng.random(size=g) < w.hit, planted, tok_rng.integers(0, V, size=g))
            tokens[d0:d0 + g] = guess
            target[t0:t0 + g + 1] = to_bf16_bits(t64) if w.dtype == BF16 else t64.astype(np.float32)
            continue
        sig = w.draft_sigmas[b % len(w.draft_sigmas)]
        d64 = w.draft_scale * t64[:g] + rng.normal(0.0, sig, size=(g, V))
        if w.dtype == BF16:
            target[t0:t0 + g + 1] = to_bf16_bits(t64)
            draft[d0:d0 + g] = to_bf16_bits(d64)
            dl = bf16_bits_to_f32(draft[d0:d0 + g]).astype(np.float64)
        else:
            target[t0:t0 + g + 1] = t64.astype(np.float32)
            draft[d0:d0 + g] = d64.astype(np.float32)
            dl = draft[d0:d0 + g].astype(np.float64)
        if g:
            if w.greedy:
                tokens[d0:d0 + g] = np.argmax(dl, axis=1)
            else:
                gum = -np.log(-np.log(tok_rng.random(size=(g, V)) + 1e-300) + 1e-300)
                tokens[d0:d0 + g] = np.argmax(dl / w.temperature + gum, axis=1)
    return Batch(w, target, draft if R_d and not w.point_mass else None, tokens, offs, gammas)


@dataclass
class TreeBatch:
    """Token trees for spec_verify_tree: gamma_b non-root nodes per tree (CSR like Batch), node j >= 1 is
    draft slot seq_offsets[b] + j - 1 with token draft_tokens[.] and parent parents[.] in [0, j); target row
    seq_offsets[b] + b + j holds the logits after the path to node j."""
    target: np.ndarray
    draft_tokens: np.ndarray
    parents: np.ndarray
    seq_offsets: np.ndarray
    gammas: np.ndarray
    temperature: float

    @property
    def B(self):
        return len(self.gammas)

    @property
    def V(self):
        return int(self.target.shape[1])

    @property
    def R_t(self):
        return int(self.seq_offsets[-1]) + self.B


def make_tree_batch(B: int, V: int, gamma_max: int, seed: int, temperature: float = 1.0, f32: bool = False,
                    chain: bool = False) -> TreeBatch:
    """Random token trees (EAGLE-style top-K candidates stand-in): node j's parent uniform in [0, j) (or
    j - 1 for a chain); a candidate is a planted token of its parent's row (raised by 6 nats) with
    probability 0.6, else one of 6 common tokens (so siblings repeat tokens); logits N(0, 2^2) plus a
    Zipf(1.1) prior, rounded once to bf16 (or kept fp32)."""
    rng = np.random.Generator(np.random.PCG64(9000 + seed))
    gam = rng.integers(0, gamma_max + 1, size=B).astype(np.int32)
    offs = np.concatenate([[0], np.cumsum(gam)]).astype(np.int32)
    R_d, R_t = int(offs[-1]), int(offs[-1]) + B
    logits = rng.normal(0, 2.0, size=(R_t, V)) - 1.1 * np.log(np.arange(1, V + 1))
    parents = np.zeros(R_d, np.int32)
    tokens = np.zeros(R_d, np.int32)
    for b in range(B):
        d0, t0 = int(offs[b]), int(offs[b]) + b
        planted = rng.integers(0, min(V, 64), size=gam[b] + 1)
        logits[t0 + np.arange(gam[b] + 1), planted] += 6.0
        for j in range(1, gam[b] + 1):
            par = j - 1 if chain else int(rng.integers(0, j))
            parents[d0 + j - 1] = par
            tokens[d0 + j - 1] = planted[par] if rng.random() < 0.6 else int(rng.integers(0, 6))
    target = logits.astype(np.float32) if f32 else to_bf16_bits(logits)
    return TreeBatch(target, tokens, parents, offs, gam, temperature)
