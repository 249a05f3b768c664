"""GPU parity of the DSpark prefix scheduler (spec_verify_schedule) against
the fp64 oracle: lengths exact, Theta to 1e-12 relative, pools whose greedy
decision sits within 1e-10 of a tie counted apart."""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_16_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def curves(n):
    b = np.arange(n, dtype=np.float64)
    return {
        "flat": np.full(n, 50.0),
        "inverse": np.concatenate([[0.0], 1000.0 / b[1:]]),
        "knee": 1e4 / np.maximum(64.0, b) / (1.0 + 0.001 * b),  # flat, then falling
        "quadratic": 1000.0 / (1.0 + 0.05 * b + 0.002 * b * b),
    }


def check(cuda_lib, conf_np, sps_np, min_margin=1e-10):
    conf = torch.tensor(conf_np, dtype=torch.float32, device=DEV).contiguous()
    sps = torch.tensor(sps_np, dtype=torch.float64, device=DEV)
    lens, theta = cuda_lib.spec_verify_schedule(conf, sps)
    torch.cuda.synchronize()
    ref = oracle.schedule_prefix(conf.cpu().numpy(), sps_np)
    if ref["margin"] < min_margin:
        return False
    assert lens.cpu().numpy().tolist() == ref["lens"].tolist()
    th = theta.cpu().numpy()
    assert th[1] == ref["added"]
    assert th[0] == pytest.approx(ref["theta"], rel=1e-12)
    return True


@pytest.mark.parametrize("curve", ["flat", "inverse", "knee", "quadratic"])
def test_random_pools(cuda_lib, curve):
    rng = np.random.default_rng(5)
    checked = 0
    for B, K in ((1, 1), (1, 15), (3, 4), (32, 15), (100, 7), (256, 15), (512, 15), (546, 15),
                 (8192, 1), (17, 0)):
        conf = rng.beta(4.0, 1.5, (B, K))  # mostly high survival, like accepted drafts
        sps = curves(B * (K + 1) + 2)[curve]
        checked += check(cuda_lib, conf, sps)
    assert checked >= 8


def test_ties_clamps_and_short_tables(cuda_lib):
    B, K = 40, 6
    # every c = 1: equal S everywhere, order by request then position
    assert check(cuda_lib, np.ones((B, K)), curves(B * (K + 1) + 2)["knee"], min_margin=0)
    # out-of-range and non-finite confidences
    rng = np.random.default_rng(6)
    conf = rng.uniform(-0.5, 1.5, (B, K))
    conf[3, 2] = np.nan
    conf[5, 0] = -0.0
    assert check(cuda_lib, conf, curves(B * (K + 1) + 2)["flat"])
    # an SPS table that stops the batch before the candidates run out
    assert check(cuda_lib, rng.uniform(0.5, 1.0, (B, K)), np.full(B + 9, 3.0))
    assert check(cuda_lib, rng.uniform(0.5, 1.0, (B, K)), np.full(B + 1, 3.0))


def test_schedule_from_verify_labels(cuda_lib):
    """The verify step's labels c* as the survival probabilities of the next
    step's drafted positions (no trained confidence head here)."""
    w = W.make_workload(W.WORKLOADS[2], W.SAMPLE, seed=21, device=DEV, B=64, V=20011)
    out = cuda_lib.verify_workload(w)
    torch.cuda.synchronize()
    conf = out.conf.view(w.B, w.spec.max_len - 1).contiguous()
    assert check(cuda_lib, conf.cpu().numpy(), curves(w.B * w.spec.max_len + 2)["knee"])
