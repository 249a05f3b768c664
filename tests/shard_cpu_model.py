"""A plain fp64 CPU model of the vocabulary-split verify (test infrastructure).

Each model rank sees only its columns [v_begin, v_begin + V_q) of the target
and draft logits and runs the same five steps as the library's split path
(include/spec_verify_shard.h), exchanging the same three kinds of buffer
through the same protocol drivers (``sharded.run_distributed`` over gloo,
``sharded.run_local`` in one process):

  stats   per row and rank: max z, sum exp(z - max) over the rank's columns,
          lowest argmax id, and z at the drafted token if the rank holds it;
  merge   the ranks' partials merged in rank order; the accept test
          u * p_d(x) < p_t(x) (greedy: x == argmax) and the first rejection;
  masses  per row and rank: sum min(p_t, p_d), sum max(0, p_t - p_d), sum p_t;
  draw    labels = the ranks' min-shares summed; the owning rank (the first
          whose running share passes u * total) walks its columns;
  finish  the owner's token.

Comparing its results with the oracle over the whole rows checks the split
algorithm itself -- merging partial statistics, choosing the owner, walking
inside it -- independently of the CUDA kernels.  Plain numpy in float64, one
row at a time.
"""

from types import SimpleNamespace

import numpy as np
import torch

import oracle
from speculative_decoding_verification_16_gb300 import workloads

# columns of the stats record and of the merged row
_M_T, _Z_T, _A_T, _M_D, _Z_D, _A_D, _X_T, _X_D, _HAS = range(9)


def _partial(z, v_begin):
    """(max, sum exp(z - max), lowest argmax id) of one row's columns."""
    m = z.max()
    if m == -np.inf:
        return -np.inf, 0.0, -1
    return m, float(np.exp(z - m).sum()), v_begin + int(np.argmax(z))


class CpuShardRank:
    def __init__(self, rank, world, v_begin, V, target_shard, draft_shard, draft_tokens,
                 uniforms, verify_lens, row_offsets, *, temperature, mode, want_conf):
        dt = workloads.dtype_name(target_shard)
        vq = target_shard.shape[1]
        self.t = oracle.decode_logits(workloads.bits_of(target_shard), dt).reshape(-1, vq)
        self.d = oracle.decode_logits(workloads.bits_of(draft_shard), dt).reshape(-1, vq)
        self.t = self.t / temperature
        self.d = self.d / temperature
        self.rank, self.world, self.v_begin, self.V = rank, world, v_begin, V
        self.x = draft_tokens.numpy().astype(np.int64)
        self.u = uniforms.double().numpy()
        self.lens = verify_lens.numpy().astype(np.int64)
        self.offs = row_offsets.numpy().astype(np.int64)
        self.mode, self.want_conf = mode, want_conf
        B, n_t, n_d = len(self.lens), self.t.shape[0], self.d.shape[0]
        self.out = SimpleNamespace(tokens=torch.full((n_t,), -1, dtype=torch.int32),
                                   accept_len=torch.zeros(B, dtype=torch.int32),
                                   conf=torch.zeros(n_d, dtype=torch.float32) if want_conf
                                   else None, row_stats=None)

    sample = property(lambda self: self.mode == oracle.SV_SAMPLE)
    needs_masses = property(lambda self: self.sample or self.want_conf)

    def rows(self):
        """(r, j, g, gd, drafted) for every target row g of every request."""
        for r in range(len(self.lens)):
            off, ell = int(self.offs[r]), int(self.lens[r])
            for j in range(ell):
                yield r, j, off + j, off - r + j, j < ell - 1

    def stats(self):
        rec = np.zeros((self.t.shape[0], 9))
        for r, j, g, gd, drafted in self.rows():
            rec[g, _M_T:_A_T + 1] = _partial(self.t[g], self.v_begin)
            rec[g, _M_D:_A_D + 1] = (-np.inf, 0.0, -1)
            if drafted:
                rec[g, _M_D:_A_D + 1] = _partial(self.d[gd], self.v_begin)
                c = int(self.x[gd]) - self.v_begin
                if 0 <= c < self.t.shape[1]:
                    rec[g, _X_T], rec[g, _X_D], rec[g, _HAS] = self.t[g, c], self.d[gd, c], 1
        return torch.from_numpy(rec)

    @staticmethod
    def _merge_stat(ms, zs, ids):
        m = ms.max()
        Z = sum(z * np.exp(mq - m) for mq, z in zip(ms, zs) if mq > -np.inf)
        return m, Z, min(int(i) for mq, i in zip(ms, ids) if mq == m)

    def merge(self, recs):
        recs = recs.numpy()
        n_t = recs.shape[1]
        self.norm = np.zeros((n_t, 4))  # m_t, Z_t, m_d, Z_d
        self.argt = np.zeros(n_t, dtype=np.int64)
        acc = np.zeros(n_t, dtype=bool)
        for r, j, g, gd, drafted in self.rows():
            mt, zt, at = self._merge_stat(recs[:, g, _M_T], recs[:, g, _Z_T], recs[:, g, _A_T])
            self.norm[g, :2] = (mt, zt)
            self.argt[g] = at
            if drafted:
                md, zd, _ = self._merge_stat(recs[:, g, _M_D], recs[:, g, _Z_D], recs[:, g, _A_D])
                self.norm[g, 2:] = (md, zd)
                q = int(np.nonzero(recs[:, g, _HAS])[0][0])  # the rank holding x
                if self.mode == oracle.SV_GREEDY:
                    acc[g] = int(self.x[gd]) == at
                else:
                    pt = np.exp(recs[q, g, _X_T] - mt) / zt
                    pd = np.exp(recs[q, g, _X_D] - md) / zd
                    acc[g] = self.u[g] * pd < pt
        self.a = np.zeros(len(self.lens), dtype=np.int64)
        for r in range(len(self.lens)):
            off, ell = int(self.offs[r]), int(self.lens[r])
            a = ell - 1
            for j in range(ell - 1):
                if not acc[off + j]:
                    a = j
                    break
            self.a[r] = a
            self.out.accept_len[r] = a
            for j in range(a):
                self.out.tokens[off + j] = int(self.x[off - r + j])
            if self.mode == oracle.SV_GREEDY:
                self.out.tokens[off + a] = int(self.argt[off + a])

    def _probs(self, g, gd, drafted):
        mt, zt, md, zd = self.norm[g]
        pt = np.exp(self.t[g] - mt) / zt
        pd = np.exp(self.d[gd] - md) / zd if drafted else None
        return pt, pd

    def masses(self):
        out = np.zeros((self.t.shape[0], 3))
        for r, j, g, gd, drafted in self.rows():
            pt, pd = self._probs(g, gd, drafted)
            out[g, 2] = pt.sum()
            if drafted:
                out[g, 0] = np.minimum(pt, pd).sum()
                out[g, 1] = np.maximum(0.0, pt - pd).sum()
        return torch.from_numpy(out)

    def draw(self, masses):
        masses = masses.numpy()
        if self.want_conf:
            for r, j, g, gd, drafted in self.rows():
                if drafted:
                    self.out.conf[gd] = float(sum(masses[q, g, 0] for q in range(self.world)))
        if not self.sample:
            return None
        cand = torch.full((len(self.lens),), -1, dtype=torch.int32)
        for r in range(len(self.lens)):
            off, ell, a = int(self.offs[r]), int(self.lens[r]), int(self.a[r])
            g, gd = off + a, off - r + a
            resid = a < ell - 1
            if resid and sum(masses[q, g, 1] for q in range(self.world)) == 0.0:
                resid = False  # no residual mass: the draw uses p_t
            k = 1 if resid else 2
            target = self.u[off + ell - 1] * sum(masses[q, g, k] for q in range(self.world))
            owner, need, run = -1, 0.0, 0.0
            for q in range(self.world):
                w = masses[q, g, k]
                if w > 0:
                    owner, need = q, target - run
                    if target < run + w:
                        break
                run += w
            if owner != self.rank:
                continue
            pt, pd = self._probs(g, gd, resid)
            wts = np.maximum(0.0, pt - pd) if resid else pt
            cum = np.cumsum(wts)
            hit = np.nonzero((cum > need) & (wts > 0))[0]
            v = int(hit[0]) if hit.size else int(np.nonzero(wts > 0)[0][-1])
            cand[r] = self.v_begin + v
        return cand

    def finish(self, cands):
        cands = cands.numpy()
        for r in range(len(self.lens)):
            off, a = int(self.offs[r]), int(self.a[r])
            owners = [int(c) for c in cands[:, r] if c >= 0]
            self.out.tokens[off + a] = owners[0]
