"""fp64 CPU oracle of the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY (see the package docstring): it is imported by the
tests, by ``__graft_entry__.smoke()`` and by the CPU legs of ``bench.py``,
never by the product path.  It is deliberately plain and slow: one request
at a time, one row at a time, numpy in float64, no blocking, no fusion.

What it computes, and where each step comes from (page title, section):

* Draft -> verify -> accept/reject.  "DeepSeek DSpark speculative decoding"
  tutorial, section "推测解码的两步流程": walk the drafted tokens from the
  first one, keep each one that passes the check, at the first failure
  sample one replacement token and drop every later candidate; when all
  pass, add one extra token from the target.  The same flow is drawn on the
  Didi EAGLE-3 page (Draft / Verify / Accept-Reject) and the DSpine page
  ("原理": only the leading run of accepted tokens counts).
* The check itself is lossless rejection sampling (DFlash/Spec V2 page,
  A3, and the DSpark FAQ: the output distribution equals the target's;
  the DFlash page cites Leviathan et al. for the method): token x drafted
  from p_d is kept when u < min(1, p_t(x)/p_d(x)); at the first rejection
  the replacement is drawn from max(0, p_t - p_d) renormalised; after a
  fully accepted block the bonus token is drawn from p_t.
* Confidence label c* = 1 - 1/2 * ||p_d - p_t||_1 for every drafted
  position (DSpark tutorial, section "置信度预测头").
* Ragged per-request verify length l_r (DSpark tutorial, section
  "硬件感知前缀调度器"); block 16 = 1 known start token + 15 guesses
  (DSpine page, "这份权重是什么").
* Sampling parameters temperature, top_p, top_k (DSpine page, "加速效果":
  temperature 1.0, top_p 0.95, top_k 20).

Readings where the pages are silent:

* Filter order: z = logit / T; keep the top_k tokens by (z desc, id asc);
  renormalise; keep the shortest prefix of that same order whose
  cumulative probability reaches top_p; renormalise.  top_k <= 0 or
  top_k >= V disables top-k, top_p >= 1 disables top-p.  The same
  processing is applied to target and draft rows.
* Accept test written as u * p_d(x) < p_t(x) (strict).  p_d(x) = 0 < p_t(x)
  accepts; p_d(x) = p_t(x) = 0 rejects.
* Inverse CDF walks token ids in ascending order and returns the smallest
  v with cumsum(w)[v] > u * sum(w) (strict).  If the residual mass is
  exactly zero (rounding only), the replacement is drawn from p_t.
* One uniform per target row: u_j tests draft j (j < l_r - 1), the last
  one (j = l_r - 1) drives the replacement or bonus draw.
* Greedy mode accepts x_j iff x_j == argmax of target row j (lowest id on
  ties) and emits the argmax of the row where it stops.
* Row statistics reported for parity: m = max_v z_v, Z = sum over the
  final kept set of exp(z_v - m), argmax = lowest id with the largest
  logit.
* Near ties (DSpine page, "调参与显存": batched floating point can flip a
  near-tied choice): every decision records its margin in absolute
  probability units -- |u - p_t/p_d| for the accept test,
  |cumsum_b - u*R| at the two edges of the chosen interval for an inverse
  CDF, |cumsum_b - top_p| at the two edges of a top-p cut, and the residual
  mass R itself for the choice between the residual and p_t at a rejection
  (the rule switches to p_t at R = 0; an exact zero is no near tie, since
  then p_t = p_d and both branches draw from the same distribution).  A
  request with any margin below NEAR_TIE is reported as near-tied.
* What a near tie leaves open: ``admissible_outcomes`` lists every result
  the rules give when each cumulative sum, ratio and residual mass may move
  by up to NEAR_TIE: the top-p kept-set sizes of every row, whether the
  accept chain is fixed, and the set of final tokens.  A computation in
  lower precision is correct when its result is one of these.
"""

from __future__ import annotations

import numpy as np

SV_GREEDY = 0
SV_SAMPLE = 1
NEAR_TIE = 1e-6


def decode_logits(raw, dtype: str) -> np.ndarray:
    """Decode stored logits to float64.

    ``dtype == "bf16"``: ``raw`` holds the 16-bit patterns (uint16, or any
    2-byte array viewed as such); a bf16 value is the float32 whose upper
    16 bits are those bits and whose lower 16 bits are zero.
    ``dtype == "fp32"``: ``raw`` holds float32 values.
    """
    a = np.asarray(raw)
    if dtype == "bf16":
        if a.dtype != np.uint16:
            a = a.view(np.uint16)
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "fp32":
        return a.astype(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


class Processed:
    """One processed row: probabilities and the statistics reported for parity."""

    __slots__ = ("p", "m", "Z", "argmax", "topp_margin", "n_kept", "topp_sizes")

    def __init__(self, p, m, Z, argmax, topp_margin, n_kept, topp_sizes=None):
        self.p = p
        self.m = m
        self.Z = Z
        self.argmax = argmax
        self.topp_margin = topp_margin
        self.n_kept = n_kept
        # kept-set sizes a top-p cut could take within the near-tie band
        # (just n_kept when no cut is near a boundary or top-p is off)
        self.topp_sizes = [n_kept] if topp_sizes is None else topp_sizes


def topp_sizes(cum, top_p: float, tol: float):
    """Kept-set sizes n' that the top-p rule "shortest prefix whose cumulative
    probability reaches top_p" gives when the cumulative sums may move by up
    to ``tol``: cum[n'-1] >= top_p - tol, and the prefix one shorter does
    not reach top_p + tol (cum[n'-2] < top_p + tol; nothing to check for
    n' = 1).  ``cum`` is the cumulative probability along the (value desc,
    id asc) order."""
    sizes = []
    for n in range(1, len(cum) + 1):
        if cum[n - 1] >= top_p - tol and (n == 1 or cum[n - 2] < top_p + tol):
            sizes.append(n)
    return sizes or [len(cum)]


def process_row(x: np.ndarray, temperature: float, top_k: int, top_p: float,
                keep_n: int | None = None) -> Processed:
    """Temperature, then top-k, renormalise, then top-p, renormalise.

    ``x`` is one row of logits in float64.  NaN or +inf anywhere, or a row
    that is entirely -inf, has no distribution and raises ValueError.
    With ``temperature <= 0`` only the argmax is defined (greedy decisions
    need nothing else); p, m and Z are then None.  ``keep_n`` replaces the
    top-p prefix length by a given one (one of ``topp_sizes``; used to list
    what a near-tied cut leaves open).
    """
    x = np.asarray(x, dtype=np.float64)
    V = x.size
    if np.isnan(x).any() or np.isposinf(x).any():
        raise ValueError("row holds NaN or +inf")
    xmax = x.max()
    if xmax == -np.inf:
        raise ValueError("row is entirely -inf")
    argmax = int(np.flatnonzero(x == xmax)[0])
    if not temperature > 0:
        return Processed(None, None, None, argmax, np.inf, V)

    z = x / temperature
    m = z.max()
    use_k = 0 < top_k < V
    use_p = top_p < 1.0
    if not (use_k or use_p):
        w = np.exp(z - m)
        Z = w.sum()
        return Processed(w / Z, m, Z, argmax, np.inf, V)

    # rank every token by (z desc, id asc)
    order = np.lexsort((np.arange(V), -z))
    kept = order[:top_k] if use_k else order
    w = np.exp(z[kept] - m)
    margin = np.inf
    sizes = None
    if use_p:
        cum = np.cumsum(w / w.sum())
        reach = np.flatnonzero(cum >= top_p)
        n = int(reach[0]) + 1 if reach.size else kept.size
        margin = abs(cum[n - 1] - top_p)
        if n >= 2:
            margin = min(margin, abs(cum[n - 2] - top_p))
        sizes = topp_sizes(cum, top_p, NEAR_TIE)
        if keep_n is not None:
            n = int(keep_n)
        kept = kept[:n]
        w = w[:n]
    Z = w.sum()
    p = np.zeros(V)
    p[kept] = w / Z
    return Processed(p, m, Z, argmax, margin, kept.size, sizes)


def row_alternatives(x: np.ndarray, temperature: float, top_k: int, top_p: float):
    """Every processed form of one row that a top-p cut within the near-tie
    band allows (one entry when the cut is clear of it): the oracle's own
    choice first."""
    first = process_row(x, temperature, top_k, top_p)
    alts = [first]
    for n in first.topp_sizes:
        if n != first.n_kept:
            alts.append(process_row(x, temperature, top_k, top_p, keep_n=n))
    return alts


def final_pick(weights: np.ndarray, u: float):
    """Inverse CDF over ascending token ids.

    Returns (v, margin): v is the smallest id with cumsum(weights)[v] >
    u * sum(weights); margin is the distance of u * sum(weights) to the two
    ends of v's interval, in the units of ``weights``.
    """
    cum = np.cumsum(weights)
    target = u * cum[-1]
    above = np.flatnonzero(cum > target)
    v = int(above[0]) if above.size else int(np.flatnonzero(weights > 0)[-1])
    lo = cum[v - 1] if v > 0 else 0.0
    return v, min(abs(cum[v] - target), abs(target - lo))


def pick_admissible(weights: np.ndarray, u: float, tol: float):
    """Every token an inverse-CDF draw over ascending ids can return when
    the point u * sum(weights) moves by up to ``tol`` (units of weights) and
    stays at or above 0: the tokens v of positive weight whose interval
    [cum[v-1], cum[v]) meets that band, and the last token of positive
    weight when the band reaches the total (the draw's own fallback)."""
    cum = np.cumsum(weights)
    target = u * cum[-1]
    lo_band, hi_band = max(0.0, target - tol), target + tol
    out = set()
    for v in range(len(weights)):
        start = cum[v - 1] if v > 0 else 0.0
        if weights[v] > 0 and start <= hi_band and cum[v] > lo_band:
            out.add(v)
    if hi_band >= cum[-1]:
        out.add(int(np.flatnonzero(weights > 0)[-1]))
    return out


def pair_step(pt: Processed, pd: Processed, x: int, u: float, mode: int):
    """Accept test for one drafted position.

    Returns (accepted, margin).  Greedy: x == argmax of the target row.
    Sampling: u * p_d(x) < p_t(x), margin |u - p_t(x)/p_d(x)|.
    """
    if mode == SV_GREEDY:
        return x == pt.argmax, np.inf
    ptx = pt.p[x]
    pdx = pd.p[x]
    if pdx > 0:
        ratio = ptx / pdx
        return bool(u < ratio), abs(u - ratio)
    return bool(ptx > 0), np.inf


def decide_request(pt, pd, x, u, mode):
    """Accept chain and final token of one request, from its processed rows.

    pt: l processed target rows (row l-1 is the bonus row); pd: l-1
    processed draft rows; x: l-1 drafted tokens; u: l uniforms.
    Returns (tokens, accept_len, margins).
    """
    ell = len(pt)
    margins = []
    a = 0
    for j in range(ell - 1):
        ok, mg = pair_step(pt[j], pd[j], int(x[j]), float(u[j]), mode)
        margins.append(mg)
        if not ok:
            break
        a += 1

    if mode == SV_GREEDY:
        final = pt[a].argmax
    else:
        if a < ell - 1:
            w = np.maximum(0.0, pt[a].p - pd[a].p)
            R = w.sum()
            if R == 0.0:
                w = pt[a].p
            else:
                margins.append(R)  # distance to the switch to p_t at R = 0
        else:
            w = pt[ell - 1].p
        final, mg = final_pick(w, float(u[ell - 1]))
        margins.append(mg)

    tokens = np.full(ell, -1, dtype=np.int64)
    tokens[:a] = [int(v) for v in x[:a]]
    tokens[a] = final
    return tokens, a, margins


def conf_label(pt: Processed, pd: Processed) -> float:
    """c* = 1 - 1/2 * sum_v |p_d(v) - p_t(v)|  (DSpark tutorial, "置信度预测头")."""
    return 1.0 - 0.5 * np.abs(pd.p - pt.p).sum()


def verify_request(t_rows, d_rows, x, u, temperature, top_k, top_p, mode,
                   want_conf: bool = True):
    """Verify one request.

    t_rows: (l, V) float64 target logits, l >= 1; row l-1 is the bonus row.
    d_rows: (l-1, V) float64 draft logits; draft row j proposed x[j].
    u:      (l,) uniforms; u[j] tests draft j, u[l-1] drives the final draw.
    Returns a dict with tokens (l,), accept_len, conf (l-1,) or None,
    stats_t / stats_d (m, Z, argmax per row), near_tie, margins.
    """
    t_rows = np.atleast_2d(np.asarray(t_rows, dtype=np.float64))
    ell = t_rows.shape[0]
    d_rows = np.asarray(d_rows, dtype=np.float64).reshape(ell - 1, t_rows.shape[1])
    V = t_rows.shape[1]
    x = [int(v) for v in np.asarray(x).reshape(-1)]
    if any(v < 0 or v >= V for v in x):
        raise ValueError("draft token out of range")
    T = temperature if (mode == SV_SAMPLE or want_conf) else 0.0
    if mode == SV_SAMPLE and not T > 0:
        raise ValueError("sampling needs temperature > 0")

    pt = [process_row(t_rows[j], T, top_k, top_p) for j in range(ell)]
    pd = [process_row(d_rows[j], T, top_k, top_p) for j in range(ell - 1)]

    conf = None
    if want_conf and T > 0:
        conf = np.array([conf_label(pt[j], pd[j]) for j in range(ell - 1)])

    tokens, a, margins = decide_request(pt, pd, x, u, mode)
    margins = margins + [r.topp_margin for r in pt] + [r.topp_margin for r in pd]
    stats = lambda r: (r.m, r.Z, r.argmax)  # noqa: E731
    return {
        "tokens": tokens,
        "accept_len": a,
        "conf": conf,
        "stats_t": [stats(r) for r in pt],
        "stats_d": [stats(r) for r in pd],
        "near_tie": bool(min(margins) < NEAR_TIE) if margins else False,
        "margins": margins,
        "topp_near_tie_t": [r.topp_margin < NEAR_TIE for r in pt],
        "topp_near_tie_d": [r.topp_margin < NEAR_TIE for r in pd],
    }


def admissible_outcomes(t_rows, d_rows, x, u, temperature, top_k, top_p, mode,
                        tol: float = NEAR_TIE):
    """What the verify rules leave open for one request when every decision
    may be flipped by a perturbation below ``tol`` (same arguments as
    verify_request).

    Each row may take any kept set of ``row_alternatives``.  Drafted
    position j is decided when every pair of alternatives of its rows gives
    the same accept outcome with margin |u_j - p_t/p_d| >= tol.  When every
    test up to the first rejection (or the bonus row) is decided, the accept
    length a is fixed and the final token lies in the union, over the
    alternatives of row a's pair, of ``pick_admissible``; a residual mass
    R with 0 < R < tol admits the draws from p_t as well.

    Returns a dict: ``determined`` (the accept chain is fixed), ``accept_len``,
    ``finals`` (set of admissible final tokens), ``conf`` (per drafted
    position, the list of labels over the alternatives of its pair),
    ``Z_t`` / ``Z_d`` (per row, the normalisers over its alternatives).
    """
    t_rows = np.atleast_2d(np.asarray(t_rows, dtype=np.float64))
    ell = t_rows.shape[0]
    V = t_rows.shape[1]
    d_rows = np.asarray(d_rows, dtype=np.float64).reshape(ell - 1, V)
    x = [int(v) for v in np.asarray(x).reshape(-1)]
    T = temperature if temperature > 0 else 0.0
    at = [row_alternatives(t_rows[j], T, top_k, top_p) for j in range(ell)]
    ad = [row_alternatives(d_rows[j], T, top_k, top_p) for j in range(ell - 1)]
    res = {"determined": True, "accept_len": None, "finals": set(),
           "conf": [[conf_label(a, b) for a in at[j] for b in ad[j]] if T > 0 else []
                    for j in range(ell - 1)],
           "Z_t": [[r.Z for r in alts] for alts in at],
           "Z_d": [[r.Z for r in alts] for alts in ad]}
    a = ell - 1
    for j in range(ell - 1):
        outcomes = set()
        for pt in at[j]:
            for pd in ad[j]:
                ok, mg = pair_step(pt, pd, x[j], float(u[j]), mode)
                outcomes.add(bool(ok))
                if mg < tol:
                    outcomes.add(not ok)
        if len(outcomes) > 1:
            res["determined"] = False
            return res
        if not outcomes.pop():
            a = j
            break
    res["accept_len"] = a
    uf = float(u[ell - 1])
    if mode == SV_GREEDY:
        res["finals"] = {at[a][0].argmax}
        return res
    for pt in at[a]:
        if a == ell - 1:
            res["finals"] |= pick_admissible(pt.p, uf, tol)
            continue
        for pd in ad[a]:
            w = np.maximum(0.0, pt.p - pd.p)
            R = w.sum()
            if R > 0.0:
                res["finals"] |= pick_admissible(w, uf, tol)
            if R < tol:
                res["finals"] |= pick_admissible(pt.p, uf, tol)
    return res


def spec_verify_oracle(target, draft, draft_tokens, uniforms, verify_lens, row_offsets,
                       dtype, temperature, top_k, top_p, mode, want_conf=True,
                       requests=None):
    """Whole-batch oracle with the C entry point's argument layout (host arrays).

    target: (N_t, V) raw logits (bf16 bit patterns or float32); draft:
    (N_d, V), N_d = N_t - B.  Request r owns target rows
    row_offsets[r] .. row_offsets[r] + l_r - 1 and draft rows starting at
    row_offsets[r] - r.  ``requests`` restricts the work to a subset of
    request ids (the other entries of the outputs stay at their fill values).
    Returns tokens (N_t,), accept_len (B,), conf (N_d,), stats_t (N_t, 3),
    stats_d (N_d, 3) and per-request near-tie flags.
    """
    verify_lens = np.asarray(verify_lens).astype(np.int64)
    row_offsets = np.asarray(row_offsets).astype(np.int64)
    B = verify_lens.size
    if row_offsets.size != B + 1 or row_offsets[0] != 0:
        raise ValueError("row_offsets must have B+1 entries starting at 0")
    if np.any(row_offsets[1:] - row_offsets[:-1] != verify_lens) or np.any(verify_lens < 1):
        raise ValueError("row_offsets are not the prefix sums of verify_lens")
    N_t = int(row_offsets[-1])
    N_d = N_t - B
    V = target.shape[1]
    tokens = np.full(N_t, -1, dtype=np.int64)
    accept_len = np.full(B, -1, dtype=np.int64)
    conf = np.full(N_d, np.nan)
    stats_t = np.full((N_t, 3), np.nan)
    stats_d = np.full((N_d, 3), np.nan)
    near_tie = np.zeros(B, dtype=bool)
    for r in (range(B) if requests is None else requests):
        off, ell = int(row_offsets[r]), int(verify_lens[r])
        doff = off - r
        t_rows = decode_logits(target[off:off + ell], dtype).reshape(ell, V)
        d_rows = decode_logits(draft[doff:doff + ell - 1], dtype).reshape(ell - 1, V)
        res = verify_request(t_rows, d_rows, draft_tokens[doff:doff + ell - 1],
                             uniforms[off:off + ell], temperature, top_k, top_p, mode,
                             want_conf=want_conf)
        tokens[off:off + ell] = res["tokens"]
        accept_len[r] = res["accept_len"]
        if res["conf"] is not None:
            conf[doff:doff + ell - 1] = res["conf"]
        for j, s in enumerate(res["stats_t"]):
            stats_t[off + j] = [np.nan if v is None else v for v in s]
        for j, s in enumerate(res["stats_d"]):
            stats_d[doff + j] = [np.nan if v is None else v for v in s]
        near_tie[r] = res["near_tie"]
    return {"tokens": tokens, "accept_len": accept_len, "conf": conf,
            "stats_t": stats_t, "stats_d": stats_d, "near_tie": near_tie}
