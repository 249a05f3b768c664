"""GPU parity of the split-vocabulary verify (include/spec_verify_shard.h):
the columns of every row split over W ranks, the ranks' steps run in
lockstep on one device (the all-gather a stack in rank order), compared with
the fp64 oracle on the whole rows under the same rules as the unsplit path,
and every rank's outputs compared with every other rank's bit for bit."""

import pytest
import torch

from parity_helpers import compare, oracle_requests
from speculative_decoding_verification_16_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def run_split(w, world, *, mode=None, want_conf=True, want_stats=True, max_len=None):
    from speculative_decoding_verification_16_gb300.sharded import verify_sharded_local
    mode = w.mode if mode is None else mode
    outs = verify_sharded_local(w.target, w.draft, w.draft_tokens, w.uniforms, w.verify_lens,
                                w.row_offsets, world,
                                max_len=w.spec.max_len if max_len is None else max_len,
                                temperature=w.spec.temperature, mode=mode, want_conf=want_conf,
                                want_stats=want_stats)
    torch.cuda.synchronize()
    return outs


def same_on_every_rank(outs):
    o0 = outs[0]
    for o in outs[1:]:
        assert torch.equal(o.tokens, o0.tokens)
        assert torch.equal(o.accept_len, o0.accept_len)
        assert torch.equal(o.dev_error, o0.dev_error)
        if o0.conf is not None:
            assert torch.equal(o.conf.view(torch.int32), o0.conf.view(torch.int32))
        if o0.row_stats is not None:
            assert torch.equal(o.row_stats.view(torch.int32), o0.row_stats.view(torch.int32))


def check_split(w, world, *, mode=None, requests=None, want_conf=True, want_stats=True,
                max_len=None, min_checked=1):
    mode = w.mode if mode is None else mode
    outs = run_split(w, world, mode=mode, want_conf=want_conf, want_stats=want_stats,
                     max_len=max_len)
    for o in outs:
        assert int(o.dev_error.item()) == 0
    same_on_every_rank(outs)
    requests = range(w.B) if requests is None else requests
    ref = oracle_requests(w, requests, mode=mode, temperature=w.spec.temperature, top_k=0,
                          top_p=1.0, want_conf=want_conf or want_stats)
    counts = compare(w, outs[0], ref, check_stats=want_stats, check_conf=want_conf)
    assert counts["checked"] >= min_checked
    return outs


SMALL = [
    # (workload index, V, B, lens)
    (0, None, None, None),          # fp32 rows of 1000
    (1, 20000, None, None),
    (2, 8191, 6, None),             # odd V: shard rows start at every 2-byte offset
    (3, 5003, 40, None),            # ragged lengths
    (3, 777, None, [1, 16, 2, 1, 9]),
]


@pytest.mark.parametrize("mode", [W.SAMPLE, W.GREEDY])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("idx,V,B,lens", SMALL)
def test_small_workloads_every_request(cuda_lib, idx, V, B, lens, world, mode):
    w = W.make_workload(W.WORKLOADS[idx], mode, seed=100 + idx, device=DEV, V=V, B=B, lens=lens)
    check_split(w, world, mode=mode)


@pytest.mark.parametrize("world", [4, 8])
def test_conc32_full_size(cuda_lib, world):
    """B 32, block 16, V 151,936 bf16, sampling with labels: every request."""
    w = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=2, device=DEV)
    check_split(w, world)


def test_ragged_full_size_sample(cuda_lib):
    """B 256 ragged, V 129,280 bf16 over 8 ranks: 40 requests compared."""
    w = W.make_workload(W.WORKLOADS[3], W.SAMPLE, seed=3, device=DEV)
    check_split(w, 8, requests=range(0, 256, 7))


@pytest.mark.parametrize("world", [2, 5])
def test_sampling_without_labels(cuda_lib, world):
    """Without labels the second round visits only each request's stopping
    row."""
    w = W.make_workload(W.WORKLOADS[3], W.SAMPLE, seed=7, device=DEV, V=30011, B=24)
    check_split(w, world, want_conf=False, want_stats=False)


def test_greedy_without_labels_takes_one_round(cuda_lib):
    w = W.make_workload(W.WORKLOADS[2], W.GREEDY, seed=8, device=DEV, V=30011, B=8)
    check_split(w, 3, mode=W.GREEDY, want_conf=False, want_stats=False)


@pytest.mark.parametrize("V,world", [(3, 3), (17, 5), (40, 32)])
def test_one_or_few_columns_per_rank(cuda_lib, V, world):
    for dtype_idx in (0, 2):  # fp32, bf16
        w = W.make_workload(W.WORKLOADS[dtype_idx], W.SAMPLE, seed=V, device=DEV, V=V, B=4,
                            lens=[5, 1, 3, 4] if dtype_idx == 0 else None)
        check_split(w, world, mode=W.SAMPLE, max_len=max(5, w.spec.max_len))


@pytest.mark.parametrize("mode", [W.SAMPLE, W.GREEDY])
def test_maximum_request_length(cuda_lib, mode):
    """Requests of the maximum 256 rows next to short ones."""
    w = W.make_workload(W.WORKLOADS[3], mode, seed=47, device=DEV, V=3001,
                        lens=[256, 1, 200, 256])
    check_split(w, 3, mode=mode, max_len=256)


def _pair_workload(t, d, x, lens, u, spec=W.WORKLOADS[2], mode=W.SAMPLE):
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    offs = torch.zeros(len(lens) + 1, dtype=torch.int32, device=DEV)
    offs[1:] = torch.cumsum(lens_t, 0)
    return W.Workload(spec, mode, t.contiguous(), d.contiguous(),
                      x.to(torch.int32).contiguous(), u.to(torch.float32).contiguous(), lens_t,
                      offs)


def test_zero_residual_draws_from_target(cuda_lib):
    """Identical target and draft rows, the drafted token of position 5
    masked in both: it is rejected, every rank's residual share is zero and
    the final token is drawn from p_t over all ranks."""
    base = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=41, device=DEV, B=5, V=12007)
    offs = base.row_offsets.cpu().numpy()
    t = base.target.clone()
    d = torch.cat([t[offs[r]:offs[r + 1] - 1] for r in range(base.B)]).clone()
    g = torch.Generator(device=DEV).manual_seed(3)
    x = torch.multinomial(torch.softmax(d.float(), 1), 1, generator=g).flatten()
    for r in range(base.B):
        j = int(offs[r]) + 5
        t[j, x[j - r]] = float("-inf")
        d[j - r, x[j - r]] = float("-inf")
    w = _pair_workload(t, d, x, [16] * base.B, base.uniforms)
    for world in (3, 7):
        outs = check_split(w, world)
        assert (outs[0].accept_len.cpu() == 5).all()


def test_identical_rows_accept_all(cuda_lib):
    base = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=4, device=DEV, B=6, V=30011)
    offs = base.row_offsets.cpu().numpy()
    d = torch.cat([base.target[offs[r]:offs[r + 1] - 1] for r in range(base.B)])
    g = torch.Generator(device=DEV).manual_seed(1)
    x = torch.multinomial(torch.softmax(d.float(), 1), 1, generator=g).flatten()
    w = _pair_workload(base.target, d, x, [16] * 6, base.uniforms)
    outs = check_split(w, 4)
    assert (outs[0].accept_len.cpu() == 15).all()


def test_matches_the_unsplit_path(cuda_lib):
    """The split and the unsplit calls agree on accept lengths and tokens
    (up to near ties, which the oracle comparison of each covers)."""
    w = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=12, device=DEV, V=50021, B=16)
    outs = run_split(w, 6)
    one = cuda_lib.verify_workload(w, want_conf=True, want_stats=True)
    torch.cuda.synchronize()
    agree = (outs[0].accept_len == one.accept_len).float().mean().item()
    assert agree >= 0.9
    # each label is within 1e-5 of the oracle's, so the two within 2e-5
    assert torch.allclose(outs[0].conf, one.conf, rtol=0, atol=2e-5)


def test_data_errors_reach_every_rank(cuda_lib):
    """A NaN in one rank's columns and a drafted token outside the
    vocabulary raise their flags on every rank."""
    w = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=13, device=DEV, V=9000, B=3)
    t = w.target.clone()
    t[0, 8500] = float("nan")  # in the last of 3 ranks' columns
    w_nan = _pair_workload(t, w.draft, w.draft_tokens, w.verify_lens.tolist(), w.uniforms)
    for o in run_split(w_nan, 3):
        assert int(o.dev_error.item()) & 1
    x = w.draft_tokens.clone()
    x[0] = 9000  # == V
    w_tok = _pair_workload(w.target, w.draft, x, w.verify_lens.tolist(), w.uniforms)
    for o in run_split(w_tok, 3):
        assert int(o.dev_error.item()) & 2
