"""Oracle of the vocabulary-sharded verify step (test infrastructure only; see ``oracle/__init__.py``).

When the logits are sharded over the vocabulary (a tensor-parallel unembedding: "All About Transformer
Inference", the model-parallel sections), the verify rule of velog "6-1편. Speculative Decoding" §2-1/§2-2
is unchanged; only where its sums are taken changes. Written out in fp64, one shard's view:
  stats     per row, over the shard's columns: the raw maximum m_j, s_j = sum exp((l - m_j) / T), the
            first argmax (global column) and the logit at the row's draft token if the shard holds it;
  decide    merged rows: m = max_j m_j, s = sum_j s_j exp((m_j - m) / T), argmax = the first shard's
            argmax among those attaining m; p(x) = exp((l_x - m) / T) / s from the shard holding x; the
            accept rule u q(x) < p(x) (greedy: x == argmax) and the first rejection n, as unsharded;
  sums      per sequence, over the shard's columns: W_j = sum of the draw's weights (max(0, p - q) for a
            residual, p for a bonus, p without x for a point-mass draft) and P_j = sum of p;
  finish    S = sum_j W_j (S = 0: P_j, draw from p); target u S; the owner is the first shard whose running
            total exceeds it (rounding: the last shard of positive weight), and it runs the inverse CDF over
            its columns with the remainder (no crossing by rounding: its last column of positive weight).
The shards exchange only these records, so the outputs equal the unsharded oracle's up to the order in
which the fp64 sums are taken. Pinned by tests against ``oracle.verify`` (unsharded) on the same batches.
``OracleShard`` has the interface the sharded protocol driver calls (stats, decide, draw_sums, finish).
"""
from __future__ import annotations

import numpy as np

from . import uniform

NONE, RESIDUAL, BONUS, RESIDUAL_PM = 0, 1, 2, 3
ERR_BAD_TOKEN, ERR_NONFINITE, ERR_EMPTY_ROW = 3, 5, 6


def _f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:  # raw bf16 codes
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


class OracleShard:
    """Shard `shard` of `bounds` (S + 1 columns). target/draft: this shard's columns of the batch's rows
    (numpy, raw bf16 codes or float32); draft None: greedy or point-mass drafts."""

    def __init__(self, shard, bounds, target, draft, draft_tokens, seq_offsets, gammas, V, temperature):
        import torch
        self.torch = torch
        self.shard, self.bounds, self.S = shard, [int(b) for b in bounds], len(bounds) - 1
        self.v0 = self.bounds[shard]
        self.lt = _f64(target)
        self.ld = None if draft is None else _f64(draft)
        self.tok = np.asarray(draft_tokens, dtype=np.int64)
        self.offs = np.asarray(seq_offsets, dtype=np.int64)
        self.gam = np.asarray(gammas, dtype=np.int64)
        self.B, self.V, self.T = len(self.gam), V, float(temperature)
        self.R_t = int(self.offs[-1]) + self.B
        self.pm = self.T > 0 and draft is None
        self.status = 0

    # rows: targets first, then drafts (sampling with draft rows)
    def _rows(self):
        n = self.R_t + (len(self.ld) if self.ld is not None and self.T > 0 else 0)
        for r in range(n):
            if r < self.R_t:
                b = int(np.searchsorted(self.offs + np.arange(self.B + 1), r, side="right") - 1)
                slot = r - int(self.offs[b]) - b
                yield r, self.lt[r], b, slot
            else:
                rr = r - self.R_t
                b = int(np.searchsorted(self.offs, rr, side="right") - 1)
                yield r, self.ld[rr], b, rr - int(self.offs[b])

    def stats(self):
        out = []
        for r, l, b, slot in self._rows():
            x = int(self.tok[self.offs[b] + slot]) if slot < self.gam[b] else -1
            g = l[x - self.v0] if self.v0 <= x < self.v0 + len(l) else 0.0
            if np.any(np.isnan(l)) or np.any(l == np.inf):
                out.append((np.nan, np.nan, -1, g))
                continue
            m = float(l.max())
            arg = self.v0 + int(np.argmax(l)) if m > -np.inf else -1
            s = float(np.exp((l - m) / self.T).sum()) if self.T > 0 and m > -np.inf else 0.0
            out.append((m, s, arg, g))
        return self.torch.tensor(out, dtype=self.torch.float64).reshape(-1, 4)

    def _merge(self, allp, r):
        ps = allp[:, r, :].numpy()
        if np.any(np.isnan(ps[:, 0])):
            return np.nan, np.nan, -1
        m = ps[:, 0].max()
        arg = int(ps[int(np.argmax(ps[:, 0])), 2])  # the first shard attaining the maximum
        if m == -np.inf or self.T == 0:
            return m, 0.0, arg
        s = sum(p[1] * np.exp((p[0] - m) / self.T) for p in ps if p[0] > -np.inf)
        return m, s, arg

    def _owner(self, x):
        return max(j for j in range(self.S) if self.bounds[j] <= x)

    def decide(self, allp, seed, step):
        self.seed, self.step = seed, step
        self.out_tokens = self.torch.full((self.R_t,), -1, dtype=self.torch.int64)
        self.out_n = self.torch.full((self.B,), -1, dtype=self.torch.int64)
        self.draws = []
        for b in range(self.B):
            g, d0 = int(self.gam[b]), int(self.offs[b])
            t0 = d0 + b
            x = self.tok[d0:d0 + g]
            code = ERR_BAD_TOKEN if np.any((x < 0) | (x >= self.V)) else 0
            T_ = [self._merge(allp, t0 + i) for i in range(g + 1)]
            D_ = [self._merge(allp, self.R_t + d0 + i) for i in range(g)] if self.T > 0 and not self.pm else []
            # the first failing row in the unsharded order: target row i, then draft row i
            order = [T_[i // 2] if i % 2 == 0 else D_[i // 2] for i in range(2 * g + 1) if i % 2 == 0 or D_]
            for m, _, _ in order:
                if not code and m != m:
                    code = ERR_NONFINITE
                if not code and m == -np.inf:
                    code = ERR_EMPTY_ROW
            if code:
                self.status |= 1 << code
                self.draws.append((NONE,))
                continue
            if self.T == 0:
                n = next((i for i in range(g) if x[i] != T_[i][2]), g)
                for j in range(g + 1):
                    self.out_tokens[t0 + j] = int(x[j]) if j < n else (T_[j][2] if j == n else -1)
                self.out_n[b] = n
                self.draws.append((NONE,))
                continue
            n = g
            for i in range(g):
                jo = self._owner(int(x[i]))
                mt, st, _ = T_[i]
                px = np.exp((allp[jo, t0 + i, 3].item() - mt) / self.T) / st
                if self.pm:
                    qx = 1.0
                else:
                    md, sd, _ = D_[i]
                    qx = np.exp((allp[jo, self.R_t + d0 + i, 3].item() - md) / self.T) / sd
                if not (uniform(seed, step, b, i, 0) * qx < px):
                    n = i
                    break
            for j in range(g + 1):
                if j != n:
                    self.out_tokens[t0 + j] = int(x[j]) if j < n else -1
            self.out_n[b] = n
            mode = BONUS if n == g else (RESIDUAL_PM if self.pm else RESIDUAL)
            self.draws.append((mode, n, T_[n], D_[n] if mode == RESIDUAL else None,
                               int(x[n]) if mode == RESIDUAL_PM else -1, uniform(seed, step, b, n, 1)))

    def _weights(self, b):
        """The draw's weights over this shard's columns, and p there."""
        dw = self.draws[b]
        n, (mp, sp, _) = dw[1], dw[2]
        d0 = int(self.offs[b])
        p = np.exp((self.lt[d0 + b + n] - mp) / self.T) / sp
        if dw[0] == RESIDUAL:
            mq, sq, _ = dw[3]
            q = np.exp((self.ld[d0 + n] - mq) / self.T) / sq
            w = np.where(p > q, p - q, 0.0)
        elif dw[0] == RESIDUAL_PM:
            w = p.copy()
            if self.v0 <= dw[4] < self.v0 + len(p):
                w[dw[4] - self.v0] = 0.0
        else:
            w = p
        return w, p

    def draw_sums(self):
        out = np.zeros((self.B, 2))
        for b in range(self.B):
            if self.draws[b][0] != NONE:
                w, p = self._weights(b)
                out[b] = (w.sum(), p.sum())
        return self.torch.tensor(out, dtype=self.torch.float64)

    def finish(self, alls):
        a = alls.numpy()
        for b in range(self.B):
            dw = self.draws[b]
            if dw[0] == NONE:
                continue
            k = 0
            if a[:, b, 0].sum() > 0.0:
                W = a[:, b, 0]
            else:  # a residual of mass 0: draw from p
                W, k = a[:, b, 1], 1
            S = W.sum()
            target = dw[5] * S
            c, jo, before = 0.0, -1, 0.0
            for j in range(self.S):
                if W[j] > 0.0 and jo < 0 and c + W[j] > target:
                    jo, before = j, c
                c += W[j]
            tail = jo < 0
            if tail:
                jo = max(j for j in range(self.S) if W[j] > 0.0)
                before = sum(W[:jo])
            t = int(self.offs[b]) + b + dw[1]
            if jo != self.shard:
                self.out_tokens[t] = -1
                continue
            w, p = self._weights(b)
            w = p if k else w
            col = -1
            if not tail:
                cum = before
                for i in range(len(w)):
                    cum += w[i]
                    if w[i] > 0.0 and cum > target:
                        col = i
                        break
            if col < 0:  # no crossing (rounding or the tail rule): the last column of positive weight
                col = int(np.nonzero(w > 0.0)[0][-1])
            self.out_tokens[t] = self.v0 + col
        return self.out_tokens


def bounds_for(V, S):
    """S contiguous shards of nearly equal width."""
    return [V * j // S for j in range(S + 1)]
