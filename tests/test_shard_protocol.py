"""The split-vocabulary verify on CPU: host argument checks of its C entry
points (nothing is enqueued), the column split, and the exchange protocol
-- which buffer each round all-gathers, in which order, and when the rounds
stop -- driven in one process and over gloo ranks (world sizes 2 and 3)."""

import ctypes
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 1 << 20  # aligned, never dereferenced: every call below fails its host checks


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_16_gb300 import build
    return ctypes.CDLL(build.build())


vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float


def _stats(lib, **over):
    a = dict(t=FAKE, d=FAKE, Vq=100, v0=0, V=300, tok=FAKE, lens=FAKE, offs=FAKE, B=2, Nt=8,
             max_len=4, dtype=0, T=1.0, rec=FAKE)
    a.update(over)
    f = lib.spec_verify_shard_stats
    f.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, i32, i32, i32, i32, f32, vp, vp]
    return f(a["t"], a["d"], a["Vq"], a["v0"], a["V"], a["tok"], a["lens"], a["offs"], a["B"],
             a["Nt"], a["max_len"], a["dtype"], a["T"], a["rec"], None)


@pytest.mark.parametrize("over,code", [
    (dict(dtype=7), -2),
    (dict(Vq=0), -1),
    (dict(v0=-1), -1),
    (dict(v0=250), -1),               # columns past the vocabulary
    (dict(T=0.0), -1),
    (dict(T=float("inf")), -1),
    (dict(t=FAKE + 1), -1),           # bf16 logits need 2-byte alignment
    (dict(d=None), -1),               # N_d = 6 > 0 needs draft logits
    (dict(tok=None), -1),
    (dict(rec=None), -1),
    (dict(rec=FAKE + 2), -1),
    (dict(B=0), -1),
    (dict(max_len=257), -1),
    (dict(Nt=9), -1),                 # more rows than B * max_len
])
def test_stats_host_checks(lib, over, code):
    assert _stats(lib, **over) == code


def _merge(lib, **over):
    a = dict(recs=FAKE, world=2, tok=FAKE, u=FAKE, lens=FAKE, offs=FAKE, B=2, V=300, Nt=8,
             max_len=4, T=1.0, mode=1, merged=FAKE, toks=FAKE, acc=FAKE, stats=None, err=None)
    a.update(over)
    f = lib.spec_verify_shard_merge
    f.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp, vp, vp, vp, vp, vp]
    return f(a["recs"], a["world"], a["tok"], a["u"], a["lens"], a["offs"], a["B"], a["V"],
             a["Nt"], a["max_len"], a["T"], a["mode"], a["merged"], a["toks"], a["acc"],
             a["stats"], a["err"], None)


@pytest.mark.parametrize("over,code", [
    (dict(world=0), -1),
    (dict(world=33), -1),
    (dict(mode=3), -1),
    (dict(T=-1.0), -1),
    (dict(recs=None), -1),
    (dict(u=None), -1),
    (dict(merged=None), -1),
    (dict(acc=None), -1),
    (dict(err=FAKE + 1), -1),
    (dict(V=0), -1),
])
def test_merge_host_checks(lib, over, code):
    assert _merge(lib, **over) == code


def test_masses_draw_finish_host_checks(lib):
    fm = lib.spec_verify_shard_masses
    fm.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp, vp]
    ok = (FAKE, FAKE, 100, FAKE, FAKE, FAKE, FAKE, 2, 8, 4, 0, 1.0)
    assert fm(*ok, 2, FAKE, None) == -1          # all_rows is 0 or 1
    assert fm(*ok[:11], 0.0, 1, FAKE, None) == -1  # T > 0
    assert fm(*ok, 1, None, None) == -1          # no output
    assert fm(*ok[:10], 5, 1.0, 1, FAKE, None) == -2  # dtype

    fd = lib.spec_verify_shard_draw
    fd.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32,
                   i32, vp, vp, vp, vp]

    def draw(world=2, rank=0, mode=1, cand=FAKE, masses=FAKE, v0=0):
        return fd(masses, world, rank, FAKE, FAKE, 100, v0, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8,
                  4, 0, 1.0, mode, None, cand, None, None)
    assert draw(rank=2) == -1                    # rank outside the world
    assert draw(rank=-1) == -1
    assert draw(world=40) == -1
    assert draw(cand=None) == -1                 # sampling needs the candidate buffer
    assert draw(masses=None) == -1
    assert draw(v0=-5) == -1

    ff = lib.spec_verify_shard_finish
    ff.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, vp, vp, vp]
    assert ff(FAKE, 0, FAKE, FAKE, FAKE, FAKE, 2, 8, FAKE, None, None) == -1
    assert ff(None, 2, FAKE, FAKE, FAKE, FAKE, 2, 8, FAKE, None, None) == -1
    assert ff(FAKE, 2, FAKE, FAKE, FAKE, FAKE, 2, 1, FAKE, None, None) == -1  # N_t < B


def test_split_columns():
    from speculative_decoding_verification_16_gb300.sharded import split_columns
    for V, world in [(1000, 1), (1000, 3), (151936, 8), (7, 7), (129280, 5), (33, 32)]:
        parts = split_columns(V, world)
        assert len(parts) == world
        v = 0
        for v0, n in parts:
            assert v0 == v and n >= 1
            v += n
        assert v == V
        assert max(n for _, n in parts) - min(n for _, n in parts) <= 1
    for V, world in [(3, 4), (100, 0), (100, 33)]:
        with pytest.raises(ValueError):
            split_columns(V, world)


class FakeRank:
    """Stands in for ShardRank on the host: each step returns a buffer that
    names its rank and step, and the receiving steps log what they got."""

    def __init__(self, rank, world, sample, want_conf, n_t=4, B=3):
        self.rank, self.world = rank, world
        self.sample, self.want_conf = sample, want_conf
        self.n_t, self.B = n_t, B
        self.out = []

    @property
    def needs_masses(self):
        return self.sample or self.want_conf

    def stats(self):
        return (torch.arange(self.n_t * 12, dtype=torch.int32).reshape(self.n_t, 12)
                + 1000 * self.rank)

    def merge(self, recs):
        self.out.append(("merge", recs.tolist()))

    def masses(self):
        return torch.arange(self.n_t * 4, dtype=torch.float32).reshape(self.n_t, 4) * 0.5 \
            + self.rank

    def draw(self, masses):
        self.out.append(("draw", masses.tolist()))
        if not self.sample:
            return None
        ids = torch.arange(self.B, dtype=torch.int32)
        return torch.where(ids % self.world == self.rank, 100 * self.rank + ids,
                           torch.full_like(ids, -1))

    def finish(self, cands):
        self.out.append(("finish", cands.tolist()))


def expected_log(world, sample, want_conf):
    ranks = [FakeRank(q, world, sample, want_conf) for q in range(world)]
    log = [("merge", torch.stack([r.stats() for r in ranks]).tolist())]
    if sample or want_conf:
        log.append(("draw", torch.stack([r.masses() for r in ranks]).tolist()))
        if sample:
            ms = torch.stack([r.masses() for r in ranks])
            log.append(("finish", torch.stack([r.draw(ms) for r in ranks]).tolist()))
    return log


MODES = [(True, True), (True, False), (False, True), (False, False)]


@pytest.mark.parametrize("sample,want_conf", MODES)
@pytest.mark.parametrize("world", [1, 2, 5])
def test_protocol_rounds_in_one_process(world, sample, want_conf):
    from speculative_decoding_verification_16_gb300.sharded import run_local
    outs = run_local([FakeRank(q, world, sample, want_conf) for q in range(world)])
    want = expected_log(world, sample, want_conf)
    assert len(outs) == world
    for o in outs:
        assert o == want
    # rounds: records always; shares for labels or sampling; candidates for sampling
    assert len(want) == 1 + (sample or want_conf) + sample


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    from speculative_decoding_verification_16_gb300.sharded import run_distributed
    from test_shard_protocol import MODES, FakeRank
    dist.init_process_group("gloo", rank=rank, world_size=world)
    logs = []
    for sample, want_conf in MODES:
        logs.append(run_distributed(FakeRank(rank, world, sample, want_conf)))
    dist.barrier()
    q.put((rank, logs))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_protocol_over_gloo_ranks(world):
    """Every rank of a gloo group receives each gathered buffer in rank
    order, the rounds end together, and the result equals the one-process
    driver's."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    for rank in range(world):
        for (sample, want_conf), log in zip(MODES, got[rank]):
            assert log == expected_log(world, sample, want_conf)


def test_shard_rank_rejects_inconsistent_inputs():
    """ShardRank checks shapes, dtypes and the column range on the host
    before any call reaches the library."""
    from speculative_decoding_verification_16_gb300.sharded import ShardRank
    B, n_t, vq = 2, 6, 10
    ok = dict(target_shard=torch.zeros((n_t, vq), dtype=torch.bfloat16),
              draft_shard=torch.zeros((n_t - B, vq), dtype=torch.bfloat16),
              draft_tokens=torch.zeros(n_t - B, dtype=torch.int32),
              uniforms=torch.zeros(n_t, dtype=torch.float32),
              verify_lens=torch.tensor([3, 3], dtype=torch.int32),
              row_offsets=torch.tensor([0, 3, 6], dtype=torch.int32))

    def make(rank=0, world=2, v_begin=0, V=20, **over):
        kw = dict(ok)
        kw.update(over)
        return ShardRank(rank, world, v_begin, V, **kw)

    make()  # consistent: accepted
    with pytest.raises(ValueError):
        make(draft_shard=torch.zeros((n_t - B, vq), dtype=torch.float32))
    with pytest.raises(ValueError):
        make(draft_shard=torch.zeros((n_t - B, vq + 1), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        make(v_begin=15)                       # columns 15..24 of a vocabulary of 20
    with pytest.raises(ValueError):
        make(rank=2)
    with pytest.raises(ValueError):
        make(target_shard=torch.zeros((vq, n_t), dtype=torch.bfloat16).t())  # not contiguous
    with pytest.raises(TypeError):
        make(draft_tokens=torch.zeros(n_t - B, dtype=torch.int64))
    with pytest.raises(TypeError):
        make(uniforms=torch.zeros(n_t, dtype=torch.float64))
