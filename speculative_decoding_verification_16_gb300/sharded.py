"""The verify step over a vocabulary split across ranks: one rank's steps and
the exchange protocol between them.

A tensor-parallel LM head (the DFlash/Spec V2 page serves at TP=8, section
"A4 实验环境与运行配置") leaves rank q the columns [v_q, v_q + V_q) of every
target and draft logits row.  ``ShardRank`` runs that rank's steps through
the C ABI of ``include/spec_verify_shard.h``; ``protocol`` orders the steps
and names the three buffers the ranks all-gather between them:

  1. stats -> records [N_t, 12]   -> merge     (statistics, accept decisions)
  2. masses -> shares [N_t, 4]    -> draw      (labels; labels or sampling only)
  3. draw  -> candidates [B]      -> finish    (the final token; sampling only)

Two drivers run the protocol: ``run_distributed`` on one rank of a
``torch.distributed`` group (``all_gather``, rank order), and ``run_local``,
which drives every rank in lockstep in one process -- all shards on one
device, the all-gather a stack of the ranks' buffers in rank order.  The
drivers only move buffers; every step of the verify runs in the library's
kernels.
"""

from __future__ import annotations

import torch

from . import binding as L


def split_columns(V: int, world: int):
    """Even split of ids [0, V) over ``world`` ranks in rank order: a list of
    (v_begin, V_q), the first V % world ranks one column longer."""
    if world < 1 or world > L.SV_SHARD_MAX_WORLD or V < world:
        raise ValueError(f"cannot split {V} columns over {world} ranks")
    base, extra = divmod(V, world)
    out, v = [], 0
    for q in range(world):
        n = base + (1 if q < extra else 0)
        out.append((v, n))
        v += n
    return out


class ShardRank:
    """One rank's side of the split verify: its columns of the logits, the
    full (replicated) per-row inputs, and the buffers of its steps."""

    def __init__(self, rank, world, v_begin, V, target_shard, draft_shard, draft_tokens,
                 uniforms, verify_lens, row_offsets, *, max_len=16, temperature=1.0,
                 mode=L.SV_SAMPLE, want_conf=True, want_stats=False, stream=None):
        for t in (target_shard, draft_shard, draft_tokens, uniforms, verify_lens, row_offsets):
            if not t.is_contiguous():
                raise ValueError("inputs must be contiguous")
        if target_shard.dim() != 2 or draft_shard.dim() != 2:
            raise ValueError("shard logits must be [rows, V_q]")
        vq = target_shard.shape[1]
        if draft_shard.dtype != target_shard.dtype or \
                (draft_shard.shape[0] and draft_shard.shape[1] != vq):
            raise ValueError("draft columns must match the target columns (dtype and V_q)")
        if not (0 <= v_begin and v_begin + vq <= V):
            raise ValueError(f"columns [{v_begin}, {v_begin + vq}) outside [0, {V})")
        if not 0 <= rank < world:
            raise ValueError(f"rank {rank} outside a world of {world}")
        for name, t, dt in (("draft_tokens", draft_tokens, torch.int32),
                            ("uniforms", uniforms, torch.float32),
                            ("verify_lens", verify_lens, torch.int32),
                            ("row_offsets", row_offsets, torch.int32)):
            if t.dtype != dt:
                raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        self.rank, self.world, self.v_begin, self.V = rank, world, v_begin, V
        self.tgt, self.drf = target_shard, draft_shard
        self.draft_tokens, self.uniforms = draft_tokens, uniforms
        self.lens, self.offs = verify_lens, row_offsets
        self.max_len, self.T, self.mode = max_len, temperature, mode
        self.want_conf = want_conf
        self.stream = stream
        n_t = target_shard.shape[0]
        B = verify_lens.numel()
        dev = target_shard.device
        self.out = L.alloc_outputs(n_t, B, dev, want_conf, want_stats)
        self.rec = torch.empty((n_t, L.SV_SHARD_REC_WORDS), dtype=torch.int32, device=dev)
        self.merged = torch.empty((n_t, L.SV_SHARD_ROW_WORDS), dtype=torch.int32, device=dev)
        self.mass = torch.zeros((n_t, L.SV_SHARD_MASS_WORDS), dtype=torch.float32, device=dev)
        self.cand = torch.empty(B, dtype=torch.int32, device=dev)

    @property
    def sample(self) -> bool:
        return self.mode == L.SV_SAMPLE

    @property
    def needs_masses(self) -> bool:
        return self.sample or self.want_conf

    def stats(self):
        L.spec_verify_shard_stats(self.tgt, self.drf, self.v_begin, self.V, self.draft_tokens,
                                  self.lens, self.offs, max_len=self.max_len,
                                  temperature=self.T, out_rec=self.rec, stream=self.stream)
        return self.rec

    def merge(self, recs):
        L.spec_verify_shard_merge(recs, self.draft_tokens, self.uniforms, self.lens, self.offs,
                                  self.V, max_len=self.max_len, temperature=self.T,
                                  mode=self.mode, out_merged=self.merged, out=self.out,
                                  stream=self.stream)

    def masses(self):
        L.spec_verify_shard_masses(self.tgt, self.drf, self.merged, self.lens, self.offs,
                                   self.out.accept_len, max_len=self.max_len,
                                   temperature=self.T, all_rows=self.want_conf,
                                   out_mass=self.mass, stream=self.stream)
        return self.mass

    def draw(self, masses):
        L.spec_verify_shard_draw(masses, self.rank, self.tgt, self.drf, self.v_begin,
                                 self.merged, self.uniforms, self.lens, self.offs,
                                 max_len=self.max_len, temperature=self.T, mode=self.mode,
                                 out=self.out, out_cand=self.cand if self.sample else None,
                                 stream=self.stream)
        return self.cand if self.sample else None

    def finish(self, cands):
        L.spec_verify_shard_finish(cands, self.merged, self.lens, self.offs, out=self.out,
                                   stream=self.stream)


def protocol(r):
    """The steps of one rank as a generator: it yields each buffer to be
    all-gathered and receives the gathered [world, ...] array; it returns
    the rank's outputs.  ``r`` is a ``ShardRank`` (or any object with the
    same five steps and flags)."""
    recs = yield r.stats()
    r.merge(recs)
    if r.needs_masses:
        masses = yield r.masses()
        cand = r.draw(masses)
        if cand is not None:
            cands = yield cand
            r.finish(cands)
    return r.out


def run_distributed(r, group=None):
    """Run one rank's protocol over a ``torch.distributed`` process group
    (``all_gather`` in rank order; NCCL for device buffers, gloo for host
    ones).  Every rank of the group calls this with its own ``r``."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    gen = protocol(r)
    try:
        buf = next(gen)
        while True:
            parts = [torch.empty_like(buf) for _ in range(world)]
            dist.all_gather(parts, buf, group=group)
            buf = gen.send(torch.stack(parts))
    except StopIteration as stop:
        return stop.value


def run_local(ranks):
    """Run the protocol of every rank in ``ranks`` (rank order) in lockstep in
    this process; the all-gather is a stack of the ranks' buffers.  Returns
    the ranks' outputs.  With all shards on one device and one stream, each
    stack is ordered after the steps that wrote its parts."""
    gens = [protocol(r) for r in ranks]
    bufs = [next(g) for g in gens]
    while True:
        gathered = torch.stack(bufs)
        nxt, done = [], []
        for g in gens:
            try:
                nxt.append(g.send(gathered))
            except StopIteration as stop:
                done.append(stop.value)
        if done:
            if nxt:
                raise RuntimeError("ranks left the protocol at different rounds")
            return done
        bufs = nxt


def verify_sharded_local(target, draft, draft_tokens, uniforms, verify_lens, row_offsets, world,
                         **kw):
    """Split the columns of ``target`` and ``draft`` over ``world`` ranks on
    their own device and run the split verify in lockstep; returns every
    rank's outputs.  (Each shard is a copy of its columns, as a
    tensor-parallel LM head would have written it.)"""
    V = target.shape[1]
    ranks = []
    for q, (v0, vq) in enumerate(split_columns(V, world)):
        ranks.append(ShardRank(q, world, v0, V, target[:, v0:v0 + vq].contiguous(),
                               draft[:, v0:v0 + vq].contiguous(), draft_tokens, uniforms,
                               verify_lens, row_offsets, **kw))
    return run_local(ranks)
