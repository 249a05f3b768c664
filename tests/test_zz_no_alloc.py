"""The entry point that allocates nothing (spec_verify_static, scratch in the
library's static device array) gives what spec_verify with a caller
workspace gives, on two calls in a row.  Collected last on purpose: it must
pass alone in a fresh process and after every other test."""

import numpy as np
import pytest
import torch

from speculative_decoding_verification_16_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _outputs(cuda_lib, w, want_stats):
    return cuda_lib.alloc_outputs(w.target.shape[0], w.B, DEV, want_conf=True,
                                  want_stats=want_stats)


def _host(o):
    return (o.tokens.cpu().numpy(), o.accept_len.cpu().numpy(), o.conf.cpu().numpy(),
            None if o.row_stats is None else o.row_stats.cpu().numpy(),
            int(o.dev_error.item()))


@pytest.mark.parametrize("idx,mode,B,top_k,top_p", [
    (0, W.SAMPLE, None, None, None),
    (2, W.SAMPLE, None, None, None),   # conc32: B=32, block 16, V=151,936 bf16
    (2, W.GREEDY, None, None, None),
    (3, W.SAMPLE, 200, None, None),    # ragged lengths, V=129,280
    (4, W.SAMPLE, 8, None, None),      # top_k 20, top_p 0.95: the small kept-set path
    (2, W.SAMPLE, 8, 0, 0.95),         # top-p over the whole row: the general path
])
def test_static_entry_matches_workspace_entry(cuda_lib, idx, mode, B, top_k, top_p):
    spec = W.WORKLOADS[idx]
    w = W.make_workload(spec, mode, seed=31, device=DEV, **({} if B is None else {"B": B}))
    assert w.target.shape[0] <= cuda_lib.SV_STATIC_MAX_ROWS
    kw = dict(max_len=spec.max_len, temperature=spec.temperature,
              top_k=spec.top_k if top_k is None else top_k,
              top_p=spec.top_p if top_p is None else top_p, mode=mode)
    ref = cuda_lib.spec_verify(w.target, w.draft, w.draft_tokens, w.uniforms, w.verify_lens,
                               w.row_offsets, want_conf=True, want_stats=True, **kw)
    torch.cuda.synchronize()
    r = _host(ref)
    assert r[4] == 0
    for _ in range(2):  # the second call reuses the scratch the first one left
        out = _outputs(cuda_lib, w, want_stats=True)
        cuda_lib.spec_verify_static(w.target, w.draft, w.draft_tokens, w.uniforms,
                                    w.verify_lens, w.row_offsets, out=out, **kw)
        torch.cuda.synchronize()
        o = _host(out)
        assert o[4] == 0
        # same kernels on the same inputs: tokens and accept lengths bit-exact,
        # labels and statistics within the parity tolerances
        assert np.array_equal(o[0], r[0])
        assert np.array_equal(o[1], r[1])
        np.testing.assert_allclose(o[2], r[2], atol=1e-5, rtol=0)
        np.testing.assert_allclose(o[3][:, :2], r[3][:, :2], rtol=1e-5, atol=0)
        assert np.array_equal(o[3][:, 2], r[3][:, 2])


def test_static_entry_rejects_more_rows_than_its_scratch(cuda_lib):
    spec = W.WORKLOADS[2]
    B, ell = 300, 16  # 4800 target rows > 4096
    w = W.make_workload(spec, W.SAMPLE, seed=32, device=DEV, B=B, V=256)
    assert w.target.shape[0] == B * ell
    out = _outputs(cuda_lib, w, want_stats=False)
    with pytest.raises(cuda_lib.SpecVerifyError) as e:
        cuda_lib.spec_verify_static(w.target, w.draft, w.draft_tokens, w.uniforms,
                                    w.verify_lens, w.row_offsets, max_len=16, out=out)
    assert e.value.status == cuda_lib.SV_ERR_TOO_LARGE
