"""Helpers shared by the GPU parity tests: run the oracle on chosen requests
of a device workload and compare element by element with the library's
outputs under the stated rules:
  - accept lengths and accepted tokens bit-exact whenever the oracle's
    accept chain is fixed (no accept test within 1e-6 of its ratio, under
    every kept set a near-tied top-p cut allows); requests whose chain is
    open are counted and left out;
  - the final token bit-exact when the oracle admits one token, and one of
    the oracle's admissible tokens when a draw lands within 1e-6 of an
    interval edge (or the residual mass is below 1e-6);
  - row normalisers (m, Z) within 1e-5 relative of the oracle's value under
    one of the admissible kept sets, argmax exact;
  - c* within 1e-5 absolute of the label under one of the admissible kept
    sets of its row pair.
Every comparison records its counts (requests, fully checked, open chains,
final tokens checked against a set, requests with any margin below 1e-6);
``tests/conftest.py`` prints them at the end of the run.
"""

import math
import os

import numpy as np

import oracle
from speculative_decoding_verification_16_gb300 import workloads

CONF_ATOL = 1e-5
NORM_RTOL = 1e-5
# Largest share of a test's requests whose accept chain may be open.  An
# accept test is open when u lands within 1e-6 of p_t/p_d: with u uniform on
# a 2^-23 grid that has probability about 2e-6 per test, so even 15 tests
# per request leave an open chain in about 3e-5 of the requests; a top-p
# cut can open a chain only when the drafted token is the cut's boundary
# token.  5 % is far above either.
MAX_OPEN_SHARE = 0.05

COUNTS = []  # (test id, requests, fully checked, open, final sets, near ties)


def oracle_requests(w, requests, *, mode, temperature, top_k, top_p, want_conf=True):
    """Oracle results for the listed requests of workload ``w`` (rows copied
    from the device one request at a time): per request the plain result
    (``verify_request``) and what near ties leave open
    (``admissible_outcomes``)."""
    lens = w.verify_lens.cpu().numpy()
    offs = w.row_offsets.cpu().numpy()
    dt = workloads.dtype_name(w.target)
    res = {}
    for r in requests:
        off, ell = int(offs[r]), int(lens[r])
        doff = off - r
        t = oracle.decode_logits(workloads.bits_of(w.target[off:off + ell]), dt)
        d = oracle.decode_logits(workloads.bits_of(w.draft[doff:doff + ell - 1]), dt)
        d = d.reshape(ell - 1, t.shape[1])
        x = w.draft_tokens[doff:doff + ell - 1].cpu().numpy()
        u = w.uniforms[off:off + ell].double().cpu().numpy()
        exact = oracle.verify_request(t, d, x, u, temperature, top_k, top_p, mode,
                                      want_conf=want_conf)
        T = temperature if (mode == oracle.SV_SAMPLE or want_conf) else 0.0
        adm = oracle.admissible_outcomes(t, d, x, u, T, top_k, top_p, mode)
        res[r] = {"exact": exact, "adm": adm}
    return res


def _near(v, choices, *, atol=0.0, rtol=0.0):
    return any(abs(v - c) <= atol + rtol * abs(c) for c in choices)


def compare(w, out, ref, *, check_stats=False, check_conf=True, max_open=None):
    """Compare library outputs with oracle results; returns a dict of counts
    (n, checked, open, final_sets, near_tie).  Raises AssertionError with the
    first mismatch, or when more than ``max_open`` requests (default: 5 % of
    them, rounded down) have an open accept chain."""
    lens = w.verify_lens.cpu().numpy()
    offs = w.row_offsets.cpu().numpy()
    toks = out.tokens.cpu().numpy()
    acc = out.accept_len.cpu().numpy()
    conf = out.conf.cpu().numpy() if (check_conf and out.conf is not None) else None
    stats = out.row_stats.cpu().numpy() if (check_stats and out.row_stats is not None) else None
    Nt = w.n_target_rows
    c = {"n": len(ref), "checked": 0, "open": 0, "final_sets": 0, "near_tie": 0}
    for r, o in ref.items():
        ex, adm = o["exact"], o["adm"]
        off, ell = int(offs[r]), int(lens[r])
        doff = off - r
        c["near_tie"] += bool(ex["near_tie"])
        if conf is not None:
            for j in range(ell - 1):
                assert _near(conf[doff + j], adm["conf"][j], atol=CONF_ATOL), \
                    f"conf of request {r} position {j}: {conf[doff + j]} vs {adm['conf'][j]}"
        if stats is not None:
            for j in range(ell):
                _check_stat(stats[off + j], ex["stats_t"][j], adm["Z_t"][j], f"target row {off + j}")
            for j in range(ell - 1):
                _check_stat(stats[Nt + doff + j], ex["stats_d"][j], adm["Z_d"][j],
                            f"draft row {doff + j}")
        if not adm["determined"]:
            c["open"] += 1
            continue
        a = adm["accept_len"]
        assert acc[r] == a, f"accept_len of request {r}: {acc[r]} vs {a}"
        got = toks[off:off + ell].tolist()
        assert got[:a] == ex["tokens"][:a].tolist(), f"accepted tokens of request {r}: {got}"
        assert got[a] in adm["finals"], \
            f"final token of request {r}: {got[a]} not in {sorted(adm['finals'])}"
        assert all(v == -1 for v in got[a + 1:]), f"tokens after the final one, request {r}: {got}"
        if len(adm["finals"]) > 1:
            c["final_sets"] += 1
        c["checked"] += 1
    limit = math.floor(MAX_OPEN_SHARE * c["n"]) if max_open is None else max_open
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    COUNTS.append((test, c["n"], c["checked"], c["open"], c["final_sets"], c["near_tie"]))
    assert c["open"] <= limit, f"{c['open']} of {c['n']} requests have an open accept chain"
    return c


def _check_stat(got, want, z_choices, what):
    m, Z, am = want
    assert int(np.float32(got[2]).view(np.int32)) == am, f"argmax of {what}"
    assert abs(got[0] - m) <= NORM_RTOL * max(1.0, abs(m)), f"m of {what}: {got[0]} vs {m}"
    assert _near(got[1], z_choices, rtol=NORM_RTOL), f"Z of {what}: {got[1]} vs {z_choices}"
