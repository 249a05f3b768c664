"""The split algorithm on CPU ranks: the fp64 model of the vocabulary-split
verify (``shard_cpu_model``), driven by the library's own protocol drivers
-- in one process and over gloo ranks -- against the oracle on the whole
rows, under the same comparison rules as the GPU parity tests."""

import os
import socket
import sys
from types import SimpleNamespace

import pytest
import torch
import torch.multiprocessing as mp

from parity_helpers import compare, oracle_requests
from shard_cpu_model import CpuShardRank
from speculative_decoding_verification_16_gb300 import workloads as W
from speculative_decoding_verification_16_gb300.sharded import (run_distributed, run_local,
                                                                split_columns)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    # (workload index, V, B, lens)
    (0, None, None, None),             # fp32, V 1000, l 5
    (2, 3001, 4, None),                # bf16, block 16
    (3, 777, None, [1, 16, 2, 1, 9]),  # ragged, a request without drafts
    (3, 2003, 12, None),
]


def model_ranks(w, world, mode, want_conf, only=None):
    V = w.target.shape[1]
    ranks = []
    for q, (v0, vq) in enumerate(split_columns(V, world)):
        if only is not None and q != only:
            continue
        ranks.append(CpuShardRank(q, world, v0, V, w.target[:, v0:v0 + vq].contiguous(),
                                  w.draft[:, v0:v0 + vq].contiguous(), w.draft_tokens,
                                  w.uniforms, w.verify_lens, w.row_offsets,
                                  temperature=w.spec.temperature, mode=mode,
                                  want_conf=want_conf))
    return ranks


def check_against_oracle(w, out, mode, want_conf):
    ref = oracle_requests(w, range(w.B), mode=mode, temperature=w.spec.temperature, top_k=0,
                          top_p=1.0, want_conf=want_conf)
    return compare(w, out, ref, check_stats=False, check_conf=want_conf)


@pytest.mark.parametrize("want_conf", [True, False])
@pytest.mark.parametrize("mode", [W.SAMPLE, W.GREEDY])
@pytest.mark.parametrize("world", [1, 2, 3, 7])
@pytest.mark.parametrize("idx,V,B,lens", CASES)
def test_split_model_in_one_process(idx, V, B, lens, world, mode, want_conf):
    w = W.make_workload(W.WORKLOADS[idx], mode, seed=200 + idx, device="cpu", V=V, B=B,
                        lens=lens)
    outs = run_local(model_ranks(w, world, mode, want_conf))
    for o in outs[1:]:  # every rank ends with the same outputs
        assert torch.equal(o.tokens, outs[0].tokens)
        assert torch.equal(o.accept_len, outs[0].accept_len)
        if want_conf:
            assert torch.equal(o.conf, outs[0].conf)
    counts = check_against_oracle(w, outs[0], mode, want_conf)
    assert counts["checked"] >= 1


def test_split_model_zero_residual():
    """Identical rows with the drafted token of position 2 masked in both:
    every rank's residual share is exactly zero and the draw falls back to
    p_t across the ranks."""
    base = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=5, device="cpu", V=1501, B=3)
    offs = base.row_offsets.numpy()
    t = base.target.clone()
    d = torch.cat([t[offs[r]:offs[r + 1] - 1] for r in range(base.B)]).clone()
    x = base.draft_tokens.clone()
    for r in range(base.B):
        j = int(offs[r]) + 2
        t[j, x[j - r]] = float("-inf")
        d[j - r, x[j - r]] = float("-inf")
    w = W.Workload(base.spec, W.SAMPLE, t, d, x, base.uniforms, base.verify_lens,
                   base.row_offsets)
    outs = run_local(model_ranks(w, 4, W.SAMPLE, True))
    assert (outs[0].accept_len <= 2).all()
    check_against_oracle(w, outs[0], W.SAMPLE, True)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    from test_shard_cpu_model import CASES, model_ranks
    dist.init_process_group("gloo", rank=rank, world_size=world)
    res = []
    for idx, V, B, lens in CASES:
        for mode in (W.SAMPLE, W.GREEDY):
            w = W.make_workload(W.WORKLOADS[idx], mode, seed=300 + idx, device="cpu", V=V, B=B,
                                lens=lens)
            out = run_distributed(model_ranks(w, world, mode, True, only=rank)[0])
            res.append((out.tokens.tolist(), out.accept_len.tolist(), out.conf.tolist()))
    dist.barrier()
    q.put((rank, res))
    dist.destroy_process_group()


def test_split_model_over_gloo_ranks():
    """Three gloo ranks, each holding only its columns, exchange through
    ``run_distributed``; every rank ends with the same outputs, and they
    match the oracle."""
    world = 3
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    for rank in range(1, world):
        assert got[rank] == got[0]
    k = 0
    for idx, V, B, lens in CASES:
        for mode in (W.SAMPLE, W.GREEDY):
            w = W.make_workload(W.WORKLOADS[idx], mode, seed=300 + idx, device="cpu", V=V, B=B,
                                lens=lens)
            toks, acc, conf = got[0][k]
            out = SimpleNamespace(tokens=torch.tensor(toks, dtype=torch.int32),
                                  accept_len=torch.tensor(acc, dtype=torch.int32),
                                  conf=torch.tensor(conf, dtype=torch.float32), row_stats=None)
            check_against_oracle(w, out, mode, True)
            k += 1
