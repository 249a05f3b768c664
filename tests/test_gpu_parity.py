"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, element by element, under the stated tolerance rules."""

import json
import math
import os
from contextlib import contextmanager

import numpy as np
import pytest
import torch

from parity_helpers import compare, oracle_requests
from speculative_decoding_verification_16_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@contextmanager
def tuning(**knobs):
    """Set rows-kernel knobs (SV_TUNE_<NAME>=value) for the duration, then
    restore their defaults."""
    from speculative_decoding_verification_16_gb300 import binding as L
    names = [k.upper() for k, v in knobs.items() if v is not None]
    try:
        for k, v in knobs.items():
            if v is not None:
                L.spec_verify_set_tuning(getattr(L, "SV_TUNE_" + k.upper()), v)
        yield
    finally:
        for k in names:
            L.spec_verify_set_tuning(getattr(L, "SV_TUNE_" + k), -1)


def slice_len(L):
    """Force the rows kernel's slice length (elements): several slices per
    row exercise the cross-CTA exchange even at small V."""
    return tuning(slice=L)


def run_and_compare(cuda_lib, w, *, requests=None, T=None, top_k=None, top_p=None,
                    want_conf=True, want_stats=True, mode=None, min_checked=1, max_len=None):
    spec = w.spec
    T = spec.temperature if T is None else T
    top_k = spec.top_k if top_k is None else top_k
    top_p = spec.top_p if top_p is None else top_p
    mode = w.mode if mode is None else mode
    max_len = spec.max_len if max_len is None else max_len
    out = cuda_lib.verify_workload(w, want_conf=want_conf, want_stats=want_stats,
                                   temperature=T, top_k=top_k, top_p=top_p, mode=mode,
                                   max_len=max_len)
    torch.cuda.synchronize()
    assert int(out.dev_error.item()) == 0
    requests = range(w.B) if requests is None else requests
    ref = oracle_requests(w, requests, mode=mode, temperature=T, top_k=top_k, top_p=top_p,
                          want_conf=want_conf or want_stats)
    counts = compare(w, out, ref, check_stats=want_stats, check_conf=want_conf)
    assert counts["checked"] >= min_checked
    return out, ref


SMALL = [
    # (workload index, V, B, lens, forced slice length)
    (0, None, None, None, None),
    (0, None, None, None, 96),      # fp32 rows of 1000 in 11 slices
    (1, 20000, None, None, None),
    (1, 20000, None, None, 1000),   # 20 slices per row
    (1, 20000, None, None, 640),    # 32 slices per row (the maximum)
    (2, 8191, 6, None, 512),        # odd V: rows not 16-byte aligned
    (2, 4099, 5, None, 1368),       # 3 slices, short last slice
    (3, 5003, 40, None, 800),       # ragged lengths
    (3, 777, None, [1, 16, 2, 1, 9], 200),
]


@pytest.mark.parametrize("mode", [W.SAMPLE, W.GREEDY])
@pytest.mark.parametrize("idx,V,B,lens,L", SMALL)
def test_small_workloads_every_request(cuda_lib, idx, V, B, lens, L, mode):
    w = W.make_workload(W.WORKLOADS[idx], mode, seed=7 + idx, device=DEV, B=B, V=V, lens=lens)
    with slice_len(L):
        run_and_compare(cuda_lib, w)


@pytest.mark.parametrize("idx,mode,sample", [
    (1, W.SAMPLE, None), (1, W.GREEDY, None),
    (2, W.SAMPLE, None), (2, W.GREEDY, None),
    (3, W.SAMPLE, None),
])
def test_full_size_workloads(cuda_lib, idx, mode, sample):
    """Full sizes in the launch configuration the bench times; the oracle
    checks every request (or a seeded sample of them)."""
    spec = W.WORKLOADS[idx]
    w = W.make_workload(spec, mode, seed=idx, device=DEV)
    reqs = None
    if sample is not None:
        reqs = sorted(np.random.default_rng(idx).choice(w.B, size=sample, replace=False).tolist())
    run_and_compare(cuda_lib, w, requests=reqs, want_stats=True)


def _pair_workload(t, d, x, lens, u, spec=W.WORKLOADS[2], mode=W.SAMPLE):
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    offs = torch.zeros(len(lens) + 1, dtype=torch.int32, device=DEV)
    offs[1:] = torch.cumsum(lens_t, 0)
    return W.Workload(spec, mode, t.contiguous(), d.contiguous(),
                      x.to(torch.int32).contiguous(), u.to(torch.float32).contiguous(), lens_t,
                      offs)


def test_no_drafted_positions(cuda_lib):
    w0 = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=3, device=DEV, V=3000, lens=[1] * 7)
    assert w0.draft.shape[0] == 0
    out, _ = run_and_compare(cuda_lib, w0)
    assert (out.accept_len.cpu() == 0).all()


def test_identical_rows_accept_all(cuda_lib):
    base = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=4, device=DEV, B=6, V=30011)
    offs = base.row_offsets.cpu().numpy()
    d = torch.cat([base.target[offs[r]:offs[r + 1] - 1] for r in range(base.B)])
    # drafted tokens drawn from the (shared) distribution
    g = torch.Generator(device=DEV).manual_seed(1)
    x = torch.multinomial(torch.softmax(d.float(), 1), 1, generator=g).flatten()
    w = _pair_workload(base.target, d, x, [16] * 6, base.uniforms)
    out, _ = run_and_compare(cuda_lib, w)
    assert (out.accept_len.cpu() == 15).all()
    assert np.allclose(out.conf.cpu().numpy(), 1.0, atol=1e-5)


def test_zero_residual_draws_from_target(cuda_lib):
    """Identical target and draft rows, with the drafted token of position 5
    masked (-inf) in both: p_d(x) = p_t(x) = 0 rejects it, the residual
    max(0, p_t - p_d) is zero everywhere and the final token is drawn from
    p_t of that row (the per-slice residual masses are rounding only, so the
    draw drops them slice by slice before it falls back)."""
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
    for L in (None, 1000):
        with slice_len(L):
            out, _ = run_and_compare(cuda_lib, w)
        assert (out.accept_len.cpu() == 5).all()


@pytest.mark.parametrize("mode", [W.SAMPLE, W.GREEDY])
def test_requests_longer_than_sixteen_rows(cuda_lib, mode):
    """l_r up to 64 (the stopping row's slice masses are read after a_r is
    known once a request has more rows than the draw kernel has warps)."""
    lens = [40, 17, 1, 64, 2, 33]
    w = W.make_workload(W.WORKLOADS[3], mode, seed=43, device=DEV, V=20011, lens=lens)
    for L in (None, 1368):
        with slice_len(L):
            run_and_compare(cuda_lib, w, max_len=64)


def test_long_requests_late_stop(cuda_lib):
    """Identical rows accept every drafted token until position 30 of request
    0, where the target masks the drafted token (a certain rejection and a
    residual draw from row 30), and to the bonus row of the others."""
    lens = [40, 33, 64]
    base = W.make_workload(W.WORKLOADS[3], W.SAMPLE, seed=44, device=DEV, V=20011, lens=lens)
    offs = base.row_offsets.cpu().numpy()
    t = base.target.clone()
    d = torch.cat([t[offs[r]:offs[r + 1] - 1] for r in range(base.B)]).clone()
    g = torch.Generator(device=DEV).manual_seed(4)
    x = torch.multinomial(torch.softmax(d.float(), 1), 1, generator=g).flatten()
    t[30, x[30]] = float("-inf")
    w = _pair_workload(t, d, x, lens, base.uniforms)
    out, _ = run_and_compare(cuda_lib, w, max_len=64)
    assert out.accept_len.cpu().tolist() == [30, 32, 63]


def test_disjoint_supports(cuda_lib):
    base = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=5, device=DEV, B=4, V=4096)
    t = base.target.clone()
    d = base.draft.clone()
    t[:, 1::2] = float("-inf")
    d[:, 0::2] = float("-inf")
    g = torch.Generator(device=DEV).manual_seed(2)
    x = torch.multinomial(torch.softmax(d.float(), 1), 1, generator=g).flatten()
    w = _pair_workload(t, d, x, [16] * 4, base.uniforms)
    out, _ = run_and_compare(cuda_lib, w)
    assert (out.accept_len.cpu() == 0).all()
    assert np.allclose(out.conf.cpu().numpy(), 0.0, atol=1e-6)
    offs = w.row_offsets.cpu().numpy()
    assert all(int(out.tokens[offs[r]]) % 2 == 0 for r in range(4))


def test_tied_maxima_lowest_id(cuda_lib):
    V = 9000
    t = torch.zeros((6, V), dtype=torch.bfloat16, device=DEV)
    for i, ids in enumerate([[5, 7000], [8999, 3], [100, 101, 102], [0, 8998], [4500], [1, 8000]]):
        t[i, ids] = 2.0
    d = t[:5].clone()
    x = torch.tensor([5, 3, 101, 0, 4500], device=DEV)
    w = _pair_workload(t, d, x, [6], torch.full((6,), 0.5, device=DEV), mode=W.GREEDY)
    out, _ = run_and_compare(cuda_lib, w)
    stats = out.row_stats.cpu().numpy()[:6, 2].view(np.int32)
    assert stats.tolist() == [5, 3, 100, 0, 4500, 1]
    assert int(out.accept_len[0]) == 2  # x0 = 5 ok, x1 = 3 ok, x2 = 101 != 100


@pytest.mark.parametrize("T", [0.05, 0.7, 10.0])
def test_temperatures(cuda_lib, T):
    w = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=9, device=DEV, B=6, V=12000)
    run_and_compare(cuda_lib, w, T=T)


def test_greedy_without_labels_or_stats(cuda_lib):
    w = W.make_workload(W.WORKLOADS[2], W.GREEDY, seed=10, device=DEV, B=8, V=50000)
    run_and_compare(cuda_lib, w, want_conf=False, want_stats=False)


def test_sampling_without_labels_or_stats(cuda_lib):
    """The final draw takes its slice masses from pass 2 even when no labels
    are asked for."""
    for idx, V, B in ((2, 50000, 8), (3, 20011, 24), (0, None, None)):
        w = W.make_workload(W.WORKLOADS[idx], W.SAMPLE, seed=11 + idx, device=DEV, B=B, V=V)
        run_and_compare(cuda_lib, w, want_conf=False, want_stats=False)


@pytest.mark.parametrize("mode", [W.SAMPLE, W.GREEDY])
def test_split_entry_points(cuda_lib, mode):
    """spec_verify_rows then spec_verify_finalize (the finalize kernels as
    their own launches) against the oracle."""
    cases = ((2, 30011, 6, None, None), (3, 20011, 24, None, 2000), (0, None, None, None, None),
             (3, 9001, None, [40, 1, 17, 3], None))
    for idx, V, B, lens, L in cases:
        w = W.make_workload(W.WORKLOADS[idx], mode, seed=51 + idx, device=DEV, B=B, V=V, lens=lens)
        max_len = max(16, int(w.verify_lens.max()))
        for want_conf in (True, False):
            out = cuda_lib.alloc_outputs(w.n_target_rows, w.B, DEV, want_conf=want_conf,
                                         want_stats=True)
            ws = cuda_lib.alloc_workspace(w.B, w.n_target_rows, DEV)
            args = (w.target, w.draft, w.draft_tokens, w.uniforms, w.verify_lens, w.row_offsets)
            kw = dict(max_len=max_len, temperature=w.spec.temperature, mode=mode, out=out,
                      workspace=ws)
            with slice_len(L):
                cuda_lib.prepare("spec_verify_rows", *args, **kw)()
                cuda_lib.prepare("spec_verify_finalize", *args, **kw)()
            torch.cuda.synchronize()
            assert int(out.dev_error.item()) == 0
            ref = oracle_requests(w, range(w.B), mode=mode, temperature=w.spec.temperature,
                                  top_k=0, top_p=1.0, want_conf=True)
            assert compare(w, out, ref, check_stats=True, check_conf=want_conf)["checked"] >= 1


def test_hand_derived_cases_on_gpu(cuda_lib):
    path = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")
    for case in json.load(open(path))["cases"]:
        rows = lambda rs: torch.tensor([[float(v) for v in r] for r in rs],  # noqa: E731
                                       dtype=torch.float32, device=DEV)
        t = rows(case["target"])
        d = rows(case["draft"]) if case["draft"] else torch.zeros((0, t.shape[1]), device=DEV)
        mode = W.SAMPLE if case["mode"] == "sample" else W.GREEDY
        w = _pair_workload(t, d, torch.tensor(case["draft_tokens"], device=DEV),
                           case["verify_lens"], torch.tensor(case["uniforms"], device=DEV),
                           mode=mode)
        out = cuda_lib.verify_workload(w, temperature=case["temperature"], top_k=case["top_k"],
                                       top_p=case["top_p"], max_len=16)
        torch.cuda.synchronize()
        np.testing.assert_allclose(out.conf.cpu().numpy(), case["conf"], atol=1e-6,
                                   err_msg=case["name"])
        if case.get("determined", [True])[0] is False:
            continue  # an accept test within 1e-6 of its ratio: no fixed chain to compare
        got = out.tokens.cpu().tolist()
        assert out.accept_len.cpu().tolist() == case["accept_len_expected"], case["name"]
        if "finals" in case:  # a near-tied draw: one of the admissible tokens
            a = case["accept_len_expected"][0]
            assert got[:a] == case["tokens"][:a] and got[a] in case["finals"][0], case["name"]
            assert got[a + 1:] == case["tokens"][a + 1:], case["name"]
        else:
            assert got == case["tokens"], case["name"]


def test_device_error_flags(cuda_lib):
    base = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=12, device=DEV, B=3, V=2048)
    t = base.target.clone()
    t[3, 17] = float("nan")
    w = _pair_workload(t, base.draft, base.draft_tokens, [16] * 3, base.uniforms)
    out = cuda_lib.verify_workload(w)
    torch.cuda.synchronize()
    assert int(out.dev_error.item()) & cuda_lib.SV_DEVERR_NAN
    x = base.draft_tokens.clone()
    x[4] = 2048
    w = _pair_workload(base.target, base.draft, x, [16] * 3, base.uniforms)
    out = cuda_lib.verify_workload(w)
    torch.cuda.synchronize()
    assert int(out.dev_error.item()) & cuda_lib.SV_DEVERR_TOKEN
    w = _pair_workload(base.target, base.draft, base.draft_tokens, [16] * 3, base.uniforms)
    w.verify_lens[1] = 15  # offsets no longer match the lengths
    out = cuda_lib.verify_workload(w)
    torch.cuda.synchronize()
    assert int(out.dev_error.item()) & cuda_lib.SV_DEVERR_LEN
    t = base.target.clone()
    t[0, :] = float("-inf")
    w = _pair_workload(t, base.draft, base.draft_tokens, [16] * 3, base.uniforms)
    out = cuda_lib.verify_workload(w)
    torch.cuda.synchronize()
    assert int(out.dev_error.item()) & cuda_lib.SV_DEVERR_NAN


def test_host_errors_through_binding(cuda_lib):
    w = W.make_workload(W.WORKLOADS[0], W.SAMPLE, seed=0, device=DEV)
    with pytest.raises(cuda_lib.SpecVerifyError):
        cuda_lib.verify_workload(w, temperature=0.0)
    with pytest.raises(cuda_lib.SpecVerifyError):
        cuda_lib.verify_workload(w, max_len=0)


def stages(n):
    return tuning(stages=n)


@pytest.mark.parametrize("warps,pass1", [(16, 4), (16, 11), (16, 12), (24, 12), (24, 15),
                                         (24, 16), (24, 20)])
@pytest.mark.parametrize("L", [None, 2504])
def test_consumer_warp_splits(cuda_lib, warps, pass1, L):
    """Any split of the consumer warps between pass 1 and pass 2 gives the
    oracle's results (labels on, so both groups run)."""
    w = W.make_workload(W.WORKLOADS[3], W.SAMPLE, seed=23, device=DEV, B=24, V=30011)
    with tuning(warps=warps, pass1_warps=pass1), slice_len(L):
        run_and_compare(cuda_lib, w)
        run_and_compare(cuda_lib, w, mode=W.GREEDY, want_conf=False, want_stats=True)


@pytest.mark.parametrize("L", [None, 2504])
def test_minimum_stage_count(cuda_lib, L):
    """Four shared-memory stages (the fewest the pipeline's barrier order
    allows) with many units per CTA."""
    w = W.make_workload(W.WORKLOADS[3], W.SAMPLE, seed=21, device=DEV, B=48, V=20000)
    with stages(4), slice_len(L):
        run_and_compare(cuda_lib, w)


def test_deterministic_across_runs_and_slice_lengths(cuda_lib):
    w = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=13, device=DEV, B=8, V=40000)
    first = None
    for L in (None, None, 10000, 6000, 2504, 1256):
        with slice_len(L):
            out = cuda_lib.verify_workload(w, want_stats=True)
        torch.cuda.synchronize()
        cur = (out.tokens.cpu().numpy(), out.accept_len.cpu().numpy(), out.conf.cpu().numpy(),
               out.row_stats.cpu().numpy())
        if first is None:
            first = cur
            continue
        if L is None:  # same configuration: bitwise identical
            for a, b in zip(first, cur):
                assert np.array_equal(a, b)
        else:
            np.testing.assert_allclose(cur[2], first[2], atol=2e-6)
            np.testing.assert_allclose(cur[3][:, :2], first[3][:, :2], rtol=2e-6)


FILTERED = [
    # (workload index, V, B, top_k, top_p)
    (0, None, None, 5, 1.0),      # fp32 rows of 1000, top-k only
    (0, None, None, 20, 0.9),
    (0, 50, 4, 0, 0.8),           # V <= 64: top-p over the whole vocabulary is served
    (1, 20000, None, 20, 0.95),
    (1, 20000, None, 64, 0.5),
    (1, 20000, None, 1, 1.0),     # top-1: the argmax only
    (2, 8191, 6, 64, 0.99),       # odd V: rows not 16-byte aligned
    (3, 5003, 40, 20, 0.95),      # ragged lengths
    (1, 20000, None, 40, 1.0),    # ranks 33..40 in the second register list
    (2, 8191, 6, 32, 0.9),        # one full register list
    (2, None, 3, 64, 1.0),        # V = 151,936: many merges into both lists
]


@pytest.mark.parametrize("mode", [W.SAMPLE, W.GREEDY])
@pytest.mark.parametrize("idx,V,B,top_k,top_p", FILTERED)
def test_filtered_every_request(cuda_lib, idx, V, B, top_k, top_p, mode):
    kw = {k: v for k, v in (("V", V), ("B", B)) if v is not None}
    w = W.make_workload(W.WORKLOADS[idx], mode, seed=41 + idx, device=DEV, **kw)
    run_and_compare(cuda_lib, w, top_k=top_k, top_p=top_p)


def test_filtered_full_size_workload(cuda_lib):
    """B=512 requests of block 16, V=262,144 bf16, top_k 20, top_p 0.95: the
    outputs of one call against the oracle on a seeded sample of 48 requests."""
    spec = W.WORKLOADS[4]
    w = W.make_workload(spec, W.SAMPLE, seed=43, device=DEV)
    reqs = sorted(np.random.default_rng(5).choice(w.B, 48, replace=False).tolist())
    run_and_compare(cuda_lib, w, requests=reqs, want_stats=True)


def test_filtered_ties_take_lowest_ids(cuda_lib):
    """Rows full of equal logits: the kept set is the lowest ids."""
    V, ell = 300, 3
    t = torch.zeros((ell, V), dtype=torch.float32, device=DEV)
    t[:, 7] = 2.0
    d = torch.zeros((ell - 1, V), dtype=torch.float32, device=DEV)
    w = _pair_workload(t, d, torch.tensor([7, 3], device=DEV), [ell],
                       torch.tensor([0.5, 0.5, 0.3], device=DEV), mode=W.SAMPLE)
    run_and_compare(cuda_lib, w, T=1.0, top_k=10, top_p=1.0)


# kept sets of any size: top_k above SV_MAX_FILTER_K, top-p over the whole
# vocabulary (the general path).  Cases whose top-p cuts sit clear of the
# near-tie margin (kept sets of about 60 to 1,100 tokens at T = 1; smaller
# at T < 1 with the +8 peak); a cut whose boundary token has probability
# near 1e-5 is fragile at fp32 precision and counted as a near tie.
GFILTERED = [
    # (workload index, V, B, top_k, top_p, T)
    (0, None, None, 0, 0.9, 1.0),       # fp32 rows of 1000, top-p alone
    (0, None, None, 200, 1.0, 1.0),     # fp32, top-k above the small-set limit
    (0, None, None, 500, 0.95, 1.0),
    (1, 20000, 8, 0, 0.95, 0.5),        # bf16, top-p over 20,000 tokens
    (1, 20000, 8, 65, 1.0, 1.0),
    (1, 20000, 8, 3000, 0.8, 0.7),
    (2, 4099, 12, 0, 0.8, 1.0),         # odd V: rows not 16-byte aligned
    (2, 8191, 12, 0, 0.7, 1.0),
    (2, 4099, 12, 2000, 0.9, 1.0),
    (2, 20011, 4, 0, 0.9, 1.0),         # about a thousand kept tokens per row
    (3, 5003, 40, 0, 0.9, 1.0),         # ragged lengths
]


@pytest.mark.parametrize("mode", [W.SAMPLE, W.GREEDY])
@pytest.mark.parametrize("idx,V,B,top_k,top_p,T", GFILTERED)
def test_large_kept_sets_every_request(cuda_lib, idx, V, B, top_k, top_p, T, mode):
    kw = {k: v for k, v in (("V", V), ("B", B)) if v is not None}
    w = W.make_workload(W.WORKLOADS[idx], mode, seed=71 + idx, device=DEV, **kw)
    run_and_compare(cuda_lib, w, T=T, top_k=top_k, top_p=top_p)


def test_large_kept_sets_ties_and_flat_rows(cuda_lib):
    """Equal logits across whole rows: top-k and top-p cuts inside one tie
    class keep the lowest ids (top_p values put the cuts well inside a
    token's mass, away from exact ties)."""
    V, ell = 3000, 4
    t = torch.zeros((ell, V), dtype=torch.float32, device=DEV)
    t[0, 11] = 1.5
    t[2, :] = -3.0  # flat row
    d = torch.zeros((ell - 1, V), dtype=torch.float32, device=DEV)
    d[1, 100:200] = 0.5
    # the last uniform sits between the cumulative steps of a uniform draw
    # over 100 equal weights (0.3 would land on one exactly)
    w = _pair_workload(t, d, torch.tensor([11, 150, 7], device=DEV), [ell],
                       torch.tensor([0.5, 0.5, 0.5, 0.305], device=DEV), mode=W.SAMPLE)
    for top_k, top_p in ((100, 1.0), (0, 0.3705), (2500, 0.6102)):
        run_and_compare(cuda_lib, w, T=1.0, top_k=top_k, top_p=top_p)


def test_large_kept_sets_full_vocabulary(cuda_lib):
    """conc32 rows (V = 151,936 bf16) under top-p 0.95 alone and top-k 1000:
    sampled requests against the oracle.  Kept sets of thousands of tokens
    leave many top-p cuts within 1e-6 of a boundary token; each such row is
    compared against every kept set the near tie allows."""
    w = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=72, device=DEV, B=6)
    run_and_compare(cuda_lib, w, top_k=0, top_p=0.95, requests=[0, 3, 5])
    run_and_compare(cuda_lib, w, top_k=1000, top_p=1.0, requests=[0, 3, 5])


@pytest.mark.parametrize("T", [0.02, 0.05, 0.1])
@pytest.mark.parametrize("seed,V,B", [(60, 12000, 6), (61, 40000, 4), (62, 151936, 2), (63, 7001, 8)])
@pytest.mark.parametrize("pass1", [8, 6, 10])
def test_low_temperature_statistics(cuda_lib, T, seed, V, B, pass1):
    """Low temperatures stretch the exponent range (sc = log2(e) / T), so the
    first-vector references of the fast path are far from the row maxima and
    overflow falls back to the exact path: statistics, labels and decisions
    must still match the oracle, for several consumer-warp splits."""
    w = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=seed, device=DEV, B=B, V=V)
    with tuning(pass1_warps=pass1):
        run_and_compare(cuda_lib, w, T=T)
        run_and_compare(cuda_lib, w, T=T, mode=W.GREEDY)


def test_cross_cta_wait_timeout_then_recovery(cuda_lib):
    """A zero limit on waits for other CTAs' published words (rows cut into
    32 slices, so every row's statistics come from 32 CTAs): the call
    returns, raises SV_DEVERR_TIMEOUT, and the next call with the default
    limit matches the oracle.  Waits on a CTA's own barriers and copies keep
    their limit, so every CTA still drains its own pipeline."""
    w = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=81, device=DEV, B=8, V=20000)
    with slice_len(640), tuning(xwait_ns=0):
        out = cuda_lib.verify_workload(w)
        torch.cuda.synchronize()
    assert int(out.dev_error.item()) & cuda_lib.SV_DEVERR_TIMEOUT
    with slice_len(640):
        run_and_compare(cuda_lib, w)
    run_and_compare(cuda_lib, w)


def _signed_zero_rows(V, n_rows, seed, dtype):
    """Rows of a few +1 logits, a large class of zeros with random signs, and
    -1 elsewhere: top-k and top-p cuts fall inside the zero class."""
    g = torch.Generator().manual_seed(seed)
    x = torch.full((n_rows, V), -1.0)
    for i in range(n_rows):
        perm = torch.randperm(V, generator=g)
        x[i, perm[:4]] = 1.0
        zeros = perm[4:4 + V // 2]
        sign = torch.randint(0, 2, (zeros.numel(),), generator=g).float() * 2 - 1
        x[i, zeros] = sign * 0.0  # -0.0 where sign is -1
    return x.to(dtype).to(DEV)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("top_k,top_p", [(20, 1.0), (64, 0.5), (100, 1.0), (0, 0.3), (0, 0.6)])
def test_signed_zeros_are_one_value(cuda_lib, dtype, top_k, top_p):
    """-0 and +0 logits form one tie class ordered by id, on the small
    kept-set path (top_k <= 64) and the general one (top_k 100, top-p over
    the whole row): the cuts inside the class keep its lowest ids."""
    V, lens = 1000, [4, 3]
    t = _signed_zero_rows(V, sum(lens), 91, dtype)
    d = _signed_zero_rows(V, sum(lens) - len(lens), 92, dtype)
    assert (torch.signbit(t.float()) & (t.float() == 0)).any()
    g = torch.Generator(device=DEV).manual_seed(5)
    x = torch.multinomial(torch.softmax(d.float(), 1), 1, generator=g).flatten()
    base = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=93, device=DEV, V=V, lens=lens)
    w = _pair_workload(t, d, x, lens, base.uniforms)
    for mode in (W.SAMPLE, W.GREEDY):
        run_and_compare(cuda_lib, w, T=1.0, top_k=top_k, top_p=top_p, mode=mode)


def test_small_residual_mass_is_drawn_from(cuda_lib):
    """A rejection whose residual mass R lies between 1e-6 and 7.6e-6: draft =
    target except that mass R moves from token y to the drafted token x (x's
    draft logit raised, y's lowered so that the normaliser stays put).  The
    residual max(0, p_t - p_d) then sits on y; the draw must take it (a
    cutoff above R would draw from p_t instead)."""
    base = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=94, device=DEV, B=6, V=12007)
    lens = [2] * 6
    offs = base.row_offsets.cpu().numpy()
    t = torch.stack([base.target[offs[r]].float() for r in range(6)]
                    + [base.target[offs[r] + 1].float() for r in range(6)])
    t = torch.cat([torch.stack([t[r], t[6 + r]]) for r in range(6)]).contiguous()
    d = t[0::2].clone()
    p = torch.softmax(t[0::2].double(), 1)
    top2 = torch.topk(p, 2, dim=1).indices
    xs, ys = top2[:, 0], top2[:, 1]
    Rs = [1.5e-6, 2e-6, 3e-6, 4e-6, 5.5e-6, 7e-6]
    for r, R in enumerate(Rs):
        px, py = float(p[r, xs[r]]), float(p[r, ys[r]])
        d[r, xs[r]] += math.log1p(R / px)
        d[r, ys[r]] -= -math.log1p(-R / py)
    # reject at position 0 with a clear margin (ratio ~ 1 - R / p_x), then
    # draw with u = 1/2
    u = torch.tensor([1 - 2.0 ** -24, 0.5] * 6, device=DEV)
    w = _pair_workload(t, d, xs.to(DEV), lens, u)
    out, ref = run_and_compare(cuda_lib, w, requests=range(6))
    toks = out.tokens.cpu().numpy()
    for r in range(6):
        assert int(out.accept_len[r]) == 0
        assert toks[2 * r] == int(ys[r]), (r, Rs[r], toks[2 * r], int(ys[r]))


@pytest.mark.parametrize("V", [1, 2, 3, 7, 17])
@pytest.mark.parametrize("idx", [0, 2])  # fp32, bf16
def test_tiny_vocabularies(cuda_lib, idx, V):
    """Degenerate vocabularies (a single token, rows shorter than one 16-byte
    vector, odd lengths): unfiltered in both modes, the small kept-set path
    and the general one."""
    for mode in (W.SAMPLE, W.GREEDY):
        w = W.make_workload(W.WORKLOADS[idx], mode, seed=90 + V, device=DEV, V=V, lens=[1, 3, 5, 2])
        run_and_compare(cuda_lib, w, T=1.0, top_k=0, top_p=1.0, mode=mode)
    w = W.make_workload(W.WORKLOADS[idx], W.SAMPLE, seed=95 + V, device=DEV, V=V, lens=[4, 1, 5])
    run_and_compare(cuda_lib, w, T=1.0, top_k=min(2, V), top_p=0.7)  # kept sets <= 64
    run_and_compare(cuda_lib, w, T=1.0, top_k=0, top_p=0.8)          # top-p over the vocabulary
    run_and_compare(cuda_lib, w, T=0.7, top_k=100, top_p=1.0)        # top_k >= V: off


@pytest.mark.parametrize("mode", [W.SAMPLE, W.GREEDY])
def test_maximum_request_length(cuda_lib, mode):
    """l_r = SV_MAX_LEN (256 target rows) next to short requests: random rows
    unfiltered and on both filtered paths, then identical target and draft
    rows, where every drafted token is accepted and the bonus row drawn."""
    lens = [256, 1, 200, 256]
    w = W.make_workload(W.WORKLOADS[3], mode, seed=47, device=DEV, V=3001, lens=lens)
    run_and_compare(cuda_lib, w, max_len=256)
    run_and_compare(cuda_lib, w, max_len=256, top_k=20, top_p=0.9)  # kept sets <= 64
    run_and_compare(cuda_lib, w, max_len=256, top_k=0, top_p=0.9)   # general path
    offs = w.row_offsets.cpu().numpy()
    t = w.target.clone()
    d = torch.cat([t[offs[r]:offs[r + 1] - 1] for r in range(w.B)]).clone()
    if mode == W.GREEDY:
        x = torch.argmax(d.float(), 1)
    else:
        g = torch.Generator(device=DEV).manual_seed(6)
        x = torch.multinomial(torch.softmax(d.float(), 1), 1, generator=g).flatten()
    same = _pair_workload(t, d, x, lens, w.uniforms, mode=mode)
    out, _ = run_and_compare(cuda_lib, same, max_len=256)
    assert out.accept_len.cpu().tolist() == [n - 1 for n in lens]
