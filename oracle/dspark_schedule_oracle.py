"""fp64 CPU oracle of the DSpark hardware-aware prefix scheduler.

TEST INFRASTRUCTURE ONLY (see the package docstring): imported by the tests
and the CPU legs of ``bench.py``, never by the product path.  Plain numpy in
float64, one candidate at a time, in the order the pages give the steps.

What it computes ("DeepSeek DSpark speculative decoding" tutorial):

* Section "置信度预测头": each drafted position k of request r carries a
  conditional survival probability c_{r,k}, the chance that the token
  passes verification given that every earlier one of the request did.
* Section "时序温度缩放校准（STS）": the scheduler works on the prefix
  survival probability S_{r,k} = prod_{i <= k} c_{r,i}.
* Section "硬件感知前缀调度器": pick each request's verify length l_r to
  maximise the global throughput Theta = tau * SPS(B), with B the total
  number of verified tokens in the batch and SPS(B) a measured steps-per-
  second curve of the target model.  Greedy execution: sort every request's
  candidate tokens by cumulative survival probability, descending; add them
  one at a time, recomputing Theta; stop as soon as Theta no longer rises.

Readings where the pages are silent:

* tau is the expected number of tokens one verify step produces: one per
  request (the replacement or bonus token) plus each verified draft k,
  which is kept when drafts 1..k all pass, probability S_{r,k}.  So, with
  positions counted from k = 0, tau = sum_r (1 + sum_{k < l_r - 1} S_{r,k}).
* l_r counts verified target rows (1 + drafted tokens verified), as in the
  verify step; every request starts at l_r = 1, so B starts at the number
  of requests and tau at the same number.  B = sum_r l_r.
* c is a probability: values are clamped to [0, 1] (NaN counts as 0), which
  keeps S non-increasing along a request, so the sorted order adds every
  request's candidates as a prefix.
* Equal S: the lower request index first, then the lower position.
* "No longer rises": the candidate whose addition would give
  Theta_next <= Theta is not added and the scan stops; it also stops when
  the candidates run out or when the SPS table has no entry for the next B.
* SPS is a table sps[b] for batch sizes b = 0 .. len(sps) - 1.
"""

from __future__ import annotations

import numpy as np


def prefix_survival(conf: np.ndarray) -> np.ndarray:
    """S_{r,k} = prod_{i <= k} c_{r,i} in float64, after clamping each c to
    [0, 1] (NaN -> 0)."""
    c = np.nan_to_num(np.asarray(conf, dtype=np.float64), nan=0.0)
    c = np.clip(c, 0.0, 1.0)
    return np.cumprod(c, axis=1)


def schedule_prefix(conf, sps):
    """Greedy prefix schedule.

    conf: [B, K] conditional survival probabilities (any float dtype).
    sps:  [n] steps per second at batch size b = index.
    Returns a dict: ``lens`` int64 [B] in 1 .. K+1, ``theta`` (the final
    Theta), ``added`` (candidates added), ``margin`` (the smallest relative
    gap |Theta_next - Theta| / Theta over every comparison made, for
    near-tie reporting; comparisons whose outcome cannot depend on rounding
    are left out).
    """
    S = prefix_survival(conf)
    B, K = S.shape
    sps = np.asarray(sps, dtype=np.float64)
    if B < 1 or len(sps) <= B:
        raise ValueError("the SPS table must cover the starting batch B")
    # every candidate (S, request, position), best first
    order = sorted(((S[r, k], r, k) for r in range(B) for k in range(K)),
                   key=lambda t: (-t[0], t[1], t[2]))
    lens = np.ones(B, dtype=np.int64)
    b = B
    tau = float(B)
    theta = tau * sps[b]
    margin = np.inf
    added = 0
    for s, r, k in order:
        if b + 1 >= len(sps):
            break
        tau_next = tau + s
        theta_next = tau_next * sps[b + 1]
        # a zero-S candidate against a curve that does not rise leaves
        # Theta_next <= Theta exactly in any arithmetic: not a near tie
        if not (s == 0.0 and sps[b + 1] <= sps[b]):
            margin = min(margin, abs(theta_next - theta) / max(abs(theta), 1e-300))
        if not theta_next > theta:
            break
        assert lens[r] == k + 1, "candidates of a request come as a prefix"
        lens[r] += 1
        b += 1
        tau = tau_next
        theta = theta_next
        added += 1
    return {"lens": lens, "theta": theta, "added": added, "margin": margin}


def expected_tokens(conf, lens) -> float:
    """tau for given verify lengths: sum_r (1 + sum_{k < l_r - 1} S_{r,k})."""
    S = prefix_survival(conf)
    return float(sum(1.0 + S[r, :int(lens[r]) - 1].sum() for r in range(S.shape[0])))
