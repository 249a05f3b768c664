"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests compares the oracle with itself: each one checks it
against a hand derivation (tests/golden), a closed form, a brute-force
re-derivation on tiny inputs, or a statistical property the pages state
(lossless output, acceptance probability = c*).
"""

import json
import math
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle
from oracle import SV_GREEDY, SV_SAMPLE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _f32_rows(rows):
    return np.array([[(-np.inf if v == "-inf" else float(v)) for v in r] for r in rows],
                    dtype=np.float32)


# --------------------------------------------------------------------------- golden
@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_derived_cases(case):
    mode = SV_SAMPLE if case["mode"] == "sample" else SV_GREEDY
    tgt = _f32_rows(case["target"])
    drf = _f32_rows(case["draft"]) if case["draft"] else np.zeros((0, tgt.shape[1]), np.float32)
    out = oracle.spec_verify_oracle(
        tgt, drf, np.array(case["draft_tokens"], np.int32),
        np.array(case["uniforms"], np.float64), np.array(case["verify_lens"]),
        np.array(case["row_offsets"]), "fp32", case["temperature"], case["top_k"],
        case["top_p"], mode)
    assert out["tokens"].tolist() == case["tokens"]
    assert out["accept_len"].tolist() == case["accept_len_expected"]
    np.testing.assert_allclose(out["conf"], case["conf"], rtol=0, atol=1e-7)
    for key in ("stats_t", "stats_d"):
        if key in case:
            np.testing.assert_allclose(out[key], np.array(case[key], float), rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", [c for c in json.load(open(GOLDEN))["cases"] if "margins" in c],
                         ids=lambda c: c["name"])
def test_hand_derived_margins(case):
    """The decision margins, near-tie flag, fixed-or-open accept chain and the
    admissible final tokens of hand-derived single-request cases (values in
    the golden file, derived on paper)."""
    mode = SV_SAMPLE if case["mode"] == "sample" else SV_GREEDY
    t = _f32_rows(case["target"]).astype(np.float64)
    d = (_f32_rows(case["draft"]).astype(np.float64) if case["draft"]
         else np.zeros((0, t.shape[1])))
    args = (t, d, case["draft_tokens"], np.array(case["uniforms"], np.float64),
            case["temperature"], case["top_k"], case["top_p"], mode)
    res = oracle.verify_request(*args)
    finite = [m for m in res["margins"] if np.isfinite(m)]
    assert finite == case["margins"]  # exact: every value is a sum of powers of two
    assert res["near_tie"] == case["near_tie"][0]
    adm = oracle.admissible_outcomes(*args)
    assert adm["determined"] == case["determined"][0]
    if adm["determined"]:
        assert adm["accept_len"] == case["accept_len_expected"][0]
        assert sorted(adm["finals"]) == case["finals"][0]
    if "topp_sizes_t" in case:
        got = [oracle.process_row(t[j], case["temperature"], case["top_k"], case["top_p"]).topp_sizes
               for j in range(t.shape[0])]
        assert got == case["topp_sizes_t"]
        assert [sorted(z) for z in adm["Z_t"]] == [sorted(z) for z in case["Z_t"]]


# --------------------------------------------------------------------------- helpers
def brute_processed(x, T, top_k, top_p):
    """Filtered distribution by pairwise rank counting (no sort) + scipy softmax."""
    V = len(x)
    z = [float(v) / T for v in x]
    rank = [sum(1 for w in range(V) if z[w] > z[v] or (z[w] == z[v] and w < v)) for v in range(V)]
    k = top_k if 0 < top_k < V else V
    kept = [v for v in range(V) if rank[v] < k]
    probs = special.softmax(np.array([z[v] for v in kept]))
    if top_p < 1.0:
        by_rank = sorted(range(len(kept)), key=lambda i: rank[kept[i]])
        total, n = 0.0, len(kept)
        for cnt, i in enumerate(by_rank, start=1):
            total += probs[i]
            if total >= top_p:
                n = cnt
                break
        keep_idx = by_rank[:n]
        kept = [kept[i] for i in keep_idx]
        probs = special.softmax(np.array([z[v] for v in kept]))
    p = np.zeros(V)
    p[kept] = probs
    return p


def inverse_cdf_loop(w, u):
    """Smallest id whose running sum exceeds u * sum(w), by a plain loop."""
    total = math.fsum(w)
    run = 0.0
    for v, wv in enumerate(w):
        run += wv
        if run > u * total:
            return v
    return max(v for v in range(len(w)) if w[v] > 0)


# --------------------------------------------------------------------------- greedy pin
def test_greedy_first_mismatch_bruteforce():
    rng = np.random.default_rng(1)
    for _ in range(300):
        V = int(rng.integers(2, 9))
        ell = int(rng.integers(1, 7))
        t = rng.integers(-2, 3, size=(ell, V)).astype(np.float32)  # many ties
        d = rng.integers(-2, 3, size=(max(ell - 1, 0), V)).astype(np.float32)
        x = rng.integers(0, V, size=ell - 1)
        out = oracle.verify_request(t.astype(float), d.astype(float), x, np.full(ell, 0.5),
                                    1.0, 0, 1.0, SV_GREEDY, want_conf=False)
        # brute force: first position whose draft differs from the first maximum
        a = 0
        for j in range(ell - 1):
            best = 0
            for v in range(V):
                if t[j, v] > t[j, best]:
                    best = v
            if x[j] != best:
                break
            a += 1
        best = 0
        for v in range(V):
            if t[a, v] > t[a, best]:
                best = v
        assert out["accept_len"] == a
        assert out["tokens"][:a].tolist() == x[:a].tolist()
        assert out["tokens"][a] == best
        assert (out["tokens"][a + 1:] == -1).all()


# --------------------------------------------------------------------------- identical rows
@pytest.mark.parametrize("filt", [(0, 1.0), (4, 0.9)])
def test_identical_rows_accept_everything(filt):
    rng = np.random.default_rng(2)
    for _ in range(20):
        V, ell = 12, 6
        t = rng.normal(0, 2, size=(ell, V))
        x = rng.integers(0, V, size=ell - 1)
        p = [brute_processed(t[j], 1.0, *filt) for j in range(ell)]
        # draw drafts from the shared distribution so that p_d(x) > 0
        x = np.array([rng.choice(V, p=p[j]) for j in range(ell - 1)])
        u = rng.uniform(0, 1, size=ell)
        out = oracle.verify_request(t, t[:-1], x, u, 1.0, filt[0], filt[1], SV_SAMPLE)
        assert out["accept_len"] == ell - 1
        np.testing.assert_allclose(out["conf"], 1.0, atol=1e-12)
        assert out["tokens"][-1] == inverse_cdf_loop(p[-1], u[-1])


# --------------------------------------------------------------------------- disjoint supports
def test_disjoint_supports_reject_first_and_resample_target():
    rng = np.random.default_rng(3)
    V = 10
    t = rng.normal(0, 1, size=(2, V))
    d = rng.normal(0, 1, size=(1, V))
    t[0, 1::2] = -np.inf
    d[0, 0::2] = -np.inf
    p_t = special.softmax(np.where(np.isinf(t[0]), -np.inf, t[0]))
    counts = np.zeros(V)
    n = 20000
    for i in range(n):
        x = [int(rng.choice(np.arange(1, V, 2)))]
        out = oracle.verify_request(t, d, x, rng.uniform(0, 1, size=2), 1.0, 0, 1.0, SV_SAMPLE)
        assert out["accept_len"] == 0
        assert out["conf"][0] == pytest.approx(0.0, abs=1e-12)
        counts[out["tokens"][0]] += 1
    assert counts[1::2].sum() == 0
    even = np.arange(0, V, 2)
    chi = stats.chisquare(counts[even], n * p_t[even])
    assert chi.pvalue > 1e-3


# --------------------------------------------------------------------------- closed forms (MC)
def _mc_rows(rng, V, ell, T, filt):
    t = rng.normal(0, 1.5, size=(ell, V))
    d = t[: ell - 1] + rng.normal(0, 1.0, size=(ell - 1, V))
    pt = [oracle.process_row(t[j], T, *filt) for j in range(ell)]
    pd = [oracle.process_row(d[j], T, *filt) for j in range(ell - 1)]
    bt = [brute_processed(t[j], T, *filt) for j in range(ell)]
    bd = [brute_processed(d[j], T, *filt) for j in range(ell - 1)]
    return pt, pd, bt, bd


@pytest.mark.parametrize("T,filt", [(1.0, (0, 1.0)), (0.7, (5, 0.85))])
def test_accept_probability_equals_conf_and_prefix_product(T, filt):
    """P(accept j | prefix accepted) = 1 - TV = c*_j (DSpark, 置信度预测头), and
    E[accepted] = sum_k prod_{i<=k} c_i (DSpark, STS section: prefix survival)."""
    rng = np.random.default_rng(4)
    V, ell, n = 10, 4, 100000
    pt, pd, bt, bd = _mc_rows(rng, V, ell, T, filt)
    c = np.array([1 - 0.5 * np.abs(bd[j] - bt[j]).sum() for j in range(ell - 1)])
    reached = np.zeros(ell - 1)
    passed = np.zeros(ell - 1)
    total_acc = 0
    xs = [rng.choice(V, size=n, p=bd[j]) for j in range(ell - 1)]
    us = rng.uniform(0, 1, size=(n, ell))
    for i in range(n):
        x = [xs[j][i] for j in range(ell - 1)]
        _, a, _ = oracle.decide_request(pt, pd, x, us[i], SV_SAMPLE)
        total_acc += a
        reached[: min(a + 1, ell - 1)] += 1
        passed[:a] += 1
    rate = passed / reached
    sigma = np.sqrt(c * (1 - c) / reached) + 1e-12
    assert np.all(np.abs(rate - c) < 5 * sigma), (rate, c)
    expect = sum(np.prod(c[: k + 1]) for k in range(ell - 1))
    assert abs(total_acc / n - expect) < 5 * math.sqrt(ell * ell / 4 / n)
    # the oracle's own label agrees with the closed form computed by scipy
    for j in range(ell - 1):
        assert oracle.conf_label(pt[j], pd[j]) == pytest.approx(c[j], abs=1e-12)


@pytest.mark.parametrize("T,filt", [(1.0, (0, 1.0)), (0.7, (5, 0.85)), (1.3, (0, 0.7))])
def test_lossless_chi_squared(T, filt):
    """Emitted token at each position, given the chain reached it, follows p_t
    exactly (DFlash page A3; DSpark FAQ: lossless)."""
    rng = np.random.default_rng(5)
    V, ell, n = 12, 3, 60000
    pt, pd, bt, bd = _mc_rows(rng, V, ell, T, filt)
    counts = np.zeros((ell, V))
    xs = [rng.choice(V, size=n, p=bd[j]) for j in range(ell - 1)]
    us = rng.uniform(0, 1, size=(n, ell))
    for i in range(n):
        x = [xs[j][i] for j in range(ell - 1)]
        toks, a, _ = oracle.decide_request(pt, pd, x, us[i], SV_SAMPLE)
        for j in range(a + 1):
            counts[j, toks[j]] += 1
    for j in range(ell):
        sup = bt[j] > 0
        assert counts[j][~sup].sum() == 0
        chi = stats.chisquare(counts[j][sup], counts[j].sum() * bt[j][sup])
        assert chi.pvalue > 1e-3, (j, chi)


# --------------------------------------------------------------------------- row statistics
def test_row_stats_closed_forms():
    for V in (1, 7, 1000):
        out = oracle.process_row(np.full(V, 3.0), 2.0, 0, 1.0)
        assert out.Z == pytest.approx(V, rel=1e-14)
        assert out.argmax == 0 and out.m == 1.5
    V, gap, hot = 500, 9.0, 123
    x = np.zeros(V)
    x[hot] = gap
    for T in (1.0, 0.5, 3.0):
        out = oracle.process_row(x, T, 0, 1.0)
        assert out.argmax == hot and out.m == gap / T
        assert out.Z == pytest.approx(1 + (V - 1) * math.exp(-gap / T), rel=1e-13)
    x = np.array([1.0, 4.0, -np.inf, 4.0])
    out = oracle.process_row(x, 1.0, 0, 1.0)
    assert out.argmax == 1 and out.p[2] == 0.0


def test_row_stats_against_sorted_sum():
    rng = np.random.default_rng(6)
    x = rng.normal(0, 3, size=4096)
    out = oracle.process_row(x, 1.0, 0, 1.0)
    terms = np.sort(np.exp(x - x.max()))
    assert out.Z == pytest.approx(math.fsum(terms), rel=1e-12)


# --------------------------------------------------------------------------- filters
def test_topk_topp_bruteforce():
    rng = np.random.default_rng(7)
    for _ in range(300):
        V = int(rng.integers(1, 40))
        x = rng.integers(-3, 4, size=V).astype(float) * 0.5  # engineered ties
        if rng.uniform() < 0.3:
            x[rng.integers(0, V)] = -np.inf
        if np.all(np.isinf(x)):
            x[0] = 0.0
        T = float(rng.choice([0.5, 1.0, 2.0]))
        k = int(rng.integers(-1, V + 2))
        p = float(rng.choice([1.0, 0.95, 0.6, 0.3]))
        got = oracle.process_row(x, T, k, p)
        want = brute_processed(x, T, k, p)
        np.testing.assert_allclose(got.p, want, rtol=0, atol=1e-12)
        assert got.p.sum() == pytest.approx(1.0, abs=1e-12)


def test_signed_zeros_tie_by_id():
    """Reading 7: -0 and +0 are one value, so a top-k cut inside a class of
    zero logits keeps the lowest ids whatever their signs."""
    x = np.array([-1.0, -0.0, 0.0, -0.0, 0.0, -2.0])
    got = oracle.process_row(x, 1.0, 3, 1.0)
    assert np.flatnonzero(got.p > 0).tolist() == [1, 2, 3]
    np.testing.assert_allclose(got.p[[1, 2, 3]], 1.0 / 3.0, rtol=0, atol=1e-15)
    assert got.argmax == 1  # lowest id holding the maximum


def test_final_pick_matches_loop():
    rng = np.random.default_rng(8)
    for _ in range(500):
        w = rng.uniform(0, 1, size=int(rng.integers(1, 20)))
        w[rng.uniform(size=w.size) < 0.3] = 0.0
        if w.sum() == 0:
            w[-1] = 1.0
        u = float(rng.uniform())
        v, margin = oracle.final_pick(w, u)
        assert v == inverse_cdf_loop(list(w), u)
        assert margin >= 0


# --------------------------------------------------------------------------- errors
def test_invalid_inputs_raise():
    with pytest.raises(ValueError):
        oracle.process_row(np.array([0.0, np.nan]), 1.0, 0, 1.0)
    with pytest.raises(ValueError):
        oracle.process_row(np.array([0.0, np.inf]), 1.0, 0, 1.0)
    with pytest.raises(ValueError):
        oracle.process_row(np.array([-np.inf, -np.inf]), 1.0, 0, 1.0)
    with pytest.raises(ValueError):
        oracle.verify_request(np.zeros((2, 3)), np.zeros((1, 3)), [3], [0.5, 0.5], 1.0, 0, 1.0,
                              SV_SAMPLE)


def test_bf16_decode():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x7F80, 0xFF80, 0x4049, 0x0001], np.uint16)
    got = oracle.decode_logits(bits, "bf16")
    assert got[:6].tolist() == [1.0, -1.0, 0.0, 0.0, np.inf, -np.inf]
    assert got[6] == 3.140625
    assert got[7] == 2.0 ** -133


# --------------------------------------------------------------------------- near-tie sets
def _draw_at(w, t):
    """Inverse-CDF draw at the point t of the running sum, by a plain loop:
    the first id whose running sum exceeds t, else the last positive id."""
    run = 0.0
    for v, wv in enumerate(w):
        run += wv
        if run > t:
            return v
    return max(v for v in range(len(w)) if w[v] > 0)


def _probe_points(edges, lo, hi):
    """Points of [lo, hi] that reach every piece of a step function with the
    given breakpoints: both ends, each breakpoint inside, the float just above
    it, and a dense grid."""
    pts = [lo, hi] + list(np.linspace(lo, hi, 2001))
    for e in edges:
        if lo <= e <= hi:
            pts += [e, np.nextafter(e, np.inf)]
    return [p for p in pts if lo <= p <= hi]


def test_pick_admissible_matches_pointwise_draws():
    rng = np.random.default_rng(11)
    for _ in range(300):
        n = int(rng.integers(1, 12))
        w = rng.uniform(0, 1, n) * 10.0 ** rng.integers(-7, 0, n)  # many tiny weights
        w[rng.uniform(size=n) < 0.3] = 0.0
        if w.sum() == 0:
            w[int(rng.integers(0, n))] = 1e-3
        cum = np.cumsum(w)
        u = float(rng.uniform())
        if rng.uniform() < 0.5:  # put u * total right next to an edge
            u = min(0.999999, max(0.0, (cum[int(rng.integers(0, n))] + rng.normal(0, 3e-7)) / cum[-1]))
        tol = float(rng.choice([1e-6, 1e-5, 1e-3]))
        target = u * cum[-1]
        lo, hi = max(0.0, target - tol), target + tol
        want = {_draw_at(w, t) for t in _probe_points(cum, lo, hi)}
        assert oracle.pick_admissible(w, u, tol) == want
        assert oracle.final_pick(w, u)[0] in want


def test_topp_sizes_match_pointwise_cuts():
    rng = np.random.default_rng(12)
    for _ in range(300):
        n = int(rng.integers(1, 15))
        p = rng.uniform(0, 1, n) * 10.0 ** rng.integers(-7, 0, n)
        p = np.sort(p)[::-1] / p.sum()
        cum = np.cumsum(p)
        top_p = float(rng.uniform(0.05, 0.999))
        if rng.uniform() < 0.5:  # a cut within a few 1e-7 of a cumulative value
            top_p = float(np.clip(cum[int(rng.integers(0, n))] + rng.normal(0, 4e-7), 1e-3, 0.9999))
        tol = float(rng.choice([1e-6, 1e-4]))

        def cut(tp):  # shortest prefix reaching tp
            for k in range(1, n + 1):
                if cum[k - 1] >= tp:
                    return k
            return n
        want = {cut(tp) for tp in _probe_points(cum, top_p - tol, top_p + tol)}
        assert set(oracle.topp_sizes(cum, top_p, tol)) == want


def test_admissible_outcomes_hold_every_perturbed_result():
    """Soundness of the near-tie sets: moving each uniform and top_p by less
    than the tolerance, the plain rules always land on an admissible outcome
    (and on the unique one when the chain is fixed)."""
    rng = np.random.default_rng(13)
    tol = 1e-6
    n_open = n_fixed = 0
    for trial in range(150):
        V, ell = int(rng.integers(3, 9)), int(rng.integers(1, 5))
        t = rng.integers(-3, 4, size=(ell, V)).astype(float) * 0.5
        d = t[: ell - 1] + rng.integers(-1, 2, size=(ell - 1, V)) * 0.5
        T = float(rng.choice([1.0, 0.7]))
        top_k, top_p = int(rng.choice([0, 4])), float(rng.choice([1.0, 0.9, 0.6]))
        pt = [oracle.process_row(t[j], T, top_k, top_p) for j in range(ell)]
        pd = [oracle.process_row(d[j], T, top_k, top_p) for j in range(ell - 1)]
        x = [int(rng.choice(V, p=pd[j].p)) for j in range(ell - 1)]
        u = rng.uniform(0, 1, ell)
        if ell > 1 and rng.uniform() < 0.5:  # an accept test right at its ratio
            r0 = pt[0].p[x[0]] / pd[0].p[x[0]]
            if r0 < 1:
                u[0] = r0 + rng.choice([-4e-7, 4e-7, 3e-6])
        if rng.uniform() < 0.3 and top_p < 1:  # a top-p cut right at a boundary
            top_p = float(np.cumsum(np.sort(pt[-1].p)[::-1])[0]) + float(rng.choice([-3e-7, 3e-7]))
        adm = oracle.admissible_outcomes(t, d, x, u, T, top_k, top_p, SV_SAMPLE, tol)
        n_fixed += adm["determined"]
        n_open += not adm["determined"]
        for _ in range(6):
            du = rng.uniform(-0.45 * tol, 0.45 * tol, ell)
            dp = float(rng.uniform(-0.45 * tol, 0.45 * tol)) if top_p < 1 else 0.0
            up = np.clip(u + du, 0.0, 1.0 - 1e-12)
            out = oracle.verify_request(t, d, x, up, T, top_k, min(1.0, top_p + dp), SV_SAMPLE)
            if adm["determined"]:
                assert out["accept_len"] == adm["accept_len"]
                assert int(out["tokens"][out["accept_len"]]) in adm["finals"]
    assert n_open > 0 and n_fixed > 50


def test_small_residual_mass_is_a_near_tie():
    """At a rejection, the choice between the residual and p_t switches at
    R = 0: R is that choice's margin.  Rows [0, 0] (target) and [delta, 0]
    (draft), x = 0: p_d(0) > p_t(0) = 1/2 and ratio = 1/2 (1 + e^-delta)
    ~ 1 - delta/2, so u = 1 - 2^-24 rejects with margin ~ delta/2 > 1e-6 for
    both deltas below; R = p_t(1) - p_d(1) = tanh(delta/2) / 2 ~ delta/4.
    The residual sits on id 1 alone; p_t with u = 1/4 would draw id 0."""
    for delta, finals in ((1e-5, {1}), (3e-6, {0, 1})):
        delta = float(np.float32(delta))
        t = np.array([[0.0, 0.0], [0.0, 0.0]])
        d = np.array([[delta, 0.0]])
        u = np.array([1 - 2.0 ** -24, 0.25])
        out = oracle.verify_request(t, d, [0], u, 1.0, 0, 1.0, SV_SAMPLE)
        assert out["accept_len"] == 0 and out["tokens"].tolist() == [1, -1]
        R = math.tanh(delta / 2) / 2
        # fp64 cancellation in p_t - p_d: about 1e-16 absolute
        assert any(abs(m - R) <= 1e-9 * R for m in out["margins"])
        assert out["margins"][0] > 1e-6  # the accept test itself is clear
        adm = oracle.admissible_outcomes(t, d, [0], u, 1.0, 0, 1.0, SV_SAMPLE)
        assert adm["determined"] and adm["accept_len"] == 0
        assert adm["finals"] == finals  # R < 1e-6 admits the p_t draw too
