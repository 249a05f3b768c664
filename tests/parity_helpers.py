"""Helpers shared by the GPU parity tests: run the oracle on chosen requests
of a device workload and compare element by element with the library's
outputs under the stated rules:
  - accept lengths and token ids bit-exact, except requests the oracle marks
    near-tied (a decision margin below 1e-6), which are counted;
  - row normalisers (m, Z) within 1e-5 relative, argmax exact;
  - c* within 1e-5 absolute.
"""

import numpy as np

import oracle
from speculative_decoding_verification_16_gb300 import workloads

CONF_ATOL = 1e-5
NORM_RTOL = 1e-5


def oracle_requests(w, requests, *, mode, temperature, top_k, top_p, want_conf=True):
    """Oracle results for the listed requests of workload ``w`` (rows copied
    from the device one request at a time)."""
    lens = w.verify_lens.cpu().numpy()
    offs = w.row_offsets.cpu().numpy()
    dt = workloads.dtype_name(w.target)
    res = {}
    for r in requests:
        off, ell = int(offs[r]), int(lens[r])
        doff = off - r
        t = oracle.decode_logits(workloads.bits_of(w.target[off:off + ell]), dt)
        d = oracle.decode_logits(workloads.bits_of(w.draft[doff:doff + ell - 1]), dt)
        x = w.draft_tokens[doff:doff + ell - 1].cpu().numpy()
        u = w.uniforms[off:off + ell].double().cpu().numpy()
        res[r] = oracle.verify_request(t, d.reshape(ell - 1, t.shape[1]), x, u, temperature, top_k,
                                       top_p, mode, want_conf=want_conf)
    return res


def compare(w, out, ref, *, check_stats=False, check_conf=True):
    """Compare library outputs with oracle results; returns (n_checked,
    n_near_tie).  Raises AssertionError with the first mismatch."""
    lens = w.verify_lens.cpu().numpy()
    offs = w.row_offsets.cpu().numpy()
    toks = out.tokens.cpu().numpy()
    acc = out.accept_len.cpu().numpy()
    conf = out.conf.cpu().numpy() if (check_conf and out.conf is not None) else None
    stats = out.row_stats.cpu().numpy() if (check_stats and out.row_stats is not None) else None
    Nt = w.n_target_rows
    n_tie = 0
    for r, o in ref.items():
        off, ell = int(offs[r]), int(lens[r])
        doff = off - r
        # a top-p cut within 1e-6 of top_p may keep one token more or less on
        # either side: such rows' Z and labels are not compared
        tie_t, tie_d = o["topp_near_tie_t"], o["topp_near_tie_d"]
        if conf is not None and ell > 1:
            keep = [j for j in range(ell - 1) if not (tie_t[j] or tie_d[j])]
            np.testing.assert_allclose(conf[doff:doff + ell - 1][keep], o["conf"][keep], rtol=0,
                                       atol=CONF_ATOL, err_msg=f"conf of request {r}")
        if stats is not None:
            for j in range(ell):
                _check_stat(stats[off + j], o["stats_t"][j], f"target row {off + j}",
                            check_z=not tie_t[j])
            for j in range(ell - 1):
                _check_stat(stats[Nt + doff + j], o["stats_d"][j], f"draft row {doff + j}",
                            check_z=not tie_d[j])
        if o["near_tie"]:
            n_tie += 1
            continue
        assert acc[r] == o["accept_len"], f"accept_len of request {r}: {acc[r]} vs {o['accept_len']}"
        assert toks[off:off + ell].tolist() == o["tokens"].tolist(), \
            f"tokens of request {r}: {toks[off:off + ell]} vs {o['tokens']}"
    return len(ref), n_tie


def _check_stat(got, want, what, check_z=True):
    m, Z, am = want
    assert int(np.float32(got[2]).view(np.int32)) == am, f"argmax of {what}"
    assert abs(got[0] - m) <= NORM_RTOL * max(1.0, abs(m)), f"m of {what}: {got[0]} vs {m}"
    if check_z:
        assert abs(got[1] - Z) <= NORM_RTOL * abs(Z), f"Z of {what}: {got[1]} vs {Z}"
