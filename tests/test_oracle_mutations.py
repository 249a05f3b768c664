"""The pins catch plausible mistakes in the oracle's near-tie bookkeeping.

Each case plants one mistake in a copy of the oracle's source (on the CPU,
never in the product) -- the wrong neighbour for an interval edge, a margin
in relative instead of absolute units, a one-sided top-p margin, a dropped
residual-mass margin, an off-by-one in the tie band, a tolerance that is
ignored, an absolute instead of relative scheduler gap -- and runs the
existing pins against the copy: at least one of them must fail.
"""

import pathlib
import types

import pytest

import test_oracle_pins as pins
import test_schedule_oracle as spins

ORACLE = pathlib.Path(__file__).resolve().parent.parent / "oracle"
VERIFY_SRC = (ORACLE / "spec_verify_oracle.py").read_text()
SCHEDULE_SRC = (ORACLE / "dspark_schedule_oracle.py").read_text()

MUTATIONS = [
    # (name, file, original text, planted text)
    ("pick_lo_two_back", "verify",
     "lo = cum[v - 1] if v > 0 else 0.0", "lo = cum[v - 2] if v > 1 else 0.0"),
    ("pick_margin_relative", "verify",
     "return v, min(abs(cum[v] - target), abs(target - lo))",
     "return v, min(abs(cum[v] - target), abs(target - lo)) / cum[-1]"),
    ("accept_margin_relative", "verify",
     "return bool(u < ratio), abs(u - ratio)", "return bool(u < ratio), abs(u - ratio) / ratio"),
    ("topp_margin_one_side", "verify",
     "margin = min(margin, abs(cum[n - 2] - top_p))", "margin = margin"),
    ("residual_margin_dropped", "verify",
     "margins.append(R)  # distance", "pass  # distance"),
    ("topp_band_one_sided", "verify",
     "(n == 1 or cum[n - 2] < top_p + tol)", "(n == 1 or cum[n - 2] < top_p)"),
    ("pick_band_not_widened", "verify",
     "lo_band, hi_band = max(0.0, target - tol), target + tol",
     "lo_band, hi_band = target, target"),
    ("accept_tolerance_ignored", "verify",
     "                if mg < tol:\n", "                if mg < 0.0:\n"),
    ("residual_tie_ignored", "verify",
     "            if R < tol:\n", "            if R == 0.0:\n"),
    ("schedule_margin_absolute", "schedule",
     "abs(theta_next - theta) / max(abs(theta), 1e-300)", "abs(theta_next - theta)"),
]


def _module(src, old, new, name):
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mod = types.ModuleType(name)
    exec(compile(src.replace(old, new), name, "exec"), mod.__dict__)
    return mod


def _facade(verify_mod, schedule_mod):
    ns = types.SimpleNamespace()
    for mod in (verify_mod, schedule_mod):
        for k, v in vars(mod).items():
            if not k.startswith("_"):
                setattr(ns, k, v)
    return ns


def _pin_calls():
    """The pins to run against a mutated copy, cheap ones first."""
    import json
    cases = json.load(open(pins.GOLDEN))["cases"]
    calls = [(f"margins[{c['name']}]", pins.test_hand_derived_margins, (c,))
             for c in cases if "margins" in c]
    calls += [(f"golden[{c['name']}]", pins.test_hand_derived_cases, (c,)) for c in cases]
    calls += [("small_residual", pins.test_small_residual_mass_is_a_near_tie, ()),
              ("pick_pointwise", pins.test_pick_admissible_matches_pointwise_draws, ()),
              ("topp_pointwise", pins.test_topp_sizes_match_pointwise_cuts, ()),
              ("final_pick_loop", pins.test_final_pick_matches_loop, ())]
    calls += [(f"theta_margin[{s}]", spins.test_near_tied_theta_margin, (s, l, a))
              for s, l, a in ((+1, [2], 1), (-1, [1], 0))]
    return calls


def test_unmutated_copy_passes_every_pin(monkeypatch):
    fac = _facade(_exec_plain(VERIFY_SRC, "v"), _exec_plain(SCHEDULE_SRC, "s"))
    monkeypatch.setattr(pins, "oracle", fac)
    monkeypatch.setattr(spins, "oracle", fac)
    for name, fn, args in _pin_calls():
        fn(*args)


def _exec_plain(src, name):
    mod = types.ModuleType(name)
    exec(compile(src, name, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,which,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(monkeypatch, name, which, old, new):
    vmod = _module(VERIFY_SRC, old, new, "v") if which == "verify" else _exec_plain(VERIFY_SRC, "v")
    smod = (_module(SCHEDULE_SRC, old, new, "s") if which == "schedule"
            else _exec_plain(SCHEDULE_SRC, "s"))
    fac = _facade(vmod, smod)
    monkeypatch.setattr(pins, "oracle", fac)
    monkeypatch.setattr(spins, "oracle", fac)
    for pin, fn, args in _pin_calls():
        try:
            fn(*args)
        except AssertionError:
            return  # caught
    pytest.fail(f"no pin caught the planted mistake {name}")
