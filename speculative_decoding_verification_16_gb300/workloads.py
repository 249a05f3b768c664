"""Seeded synthetic verify workloads.

This module only draws inputs: target and draft logits, drafted tokens,
uniforms, per-request verify lengths and row offsets.  It holds none of the
verify step's arithmetic and imports neither the CUDA binding nor the
oracle; both sides are fed from here.

Shapes and distributions follow the settings printed on the source pages:
block 16 = 1 known start token + 15 drafted positions (DSpine page,
"这份权重是什么"; DFlash page, A4: block size 16), concurrency 1 / 32
(DFlash page, A4; Didi page, inference section), ragged per-request verify
length l_r (DSpark tutorial, "硬件感知前缀调度器"), sampling temperature 1.0,
top_p 0.95, top_k 20 (DSpine page, "加速效果").  No benchmark data set is
used or reproduced.

Recipe (per row, before rounding to the stored dtype):
  target  t = N(0, sigma_t^2), plus +peak on one token per row whose id is
          Zipf(s)-distributed over ranks 1..V (id = rank - 1), when a peak
          is configured;
  draft   d = t + N(0, sigma_r^2) with sigma_r fixed or U[lo, hi] per request;
  stored  bf16 by round-to-nearest-even, or fp32.
Drafted tokens: greedy mode takes the argmax of the stored draft row;
sampling mode draws x from softmax(d / T) by the Gumbel-max trick, over the
draft row's top_k candidates when top_k is set (top_p is not applied by
the generator, so a drafted token may fall outside the draft's top-p set).
Uniforms: u = (k + 1/2) * 2^-23 with k uniform in [0, 2^23): 2k + 1 needs
at most 24 significant bits, so u is exact in float32 and float64, and
never 0 or 1.

Sub-streams (torch.Generator seeds = 1000 * seed + stream): 0 target noise,
1 draft noise, 2 peak ids, 3 per-request sigma, 4 verify lengths,
5 draft sampling, 6 verify uniforms.
"""

from __future__ import annotations

import dataclasses
import math

import torch

GREEDY = 0
SAMPLE = 1


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    B: int
    max_len: int            # verify length l_r (target rows) or its maximum when ragged
    ragged: bool            # l_r ~ U{1..max_len} per request
    V: int
    dtype: str              # "bf16" or "fp32"
    sigma_t: float
    peak: float             # 0 disables the Zipf peak
    zipf_s: float
    noise: tuple            # ("fixed", s) or ("uniform", lo, hi)
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    modes: tuple = ("sample", "greedy")


# The five synthetic workloads, in order.
WORKLOADS = [
    WorkloadSpec("tiny_v1000_fp32", B=1, max_len=5, ragged=False, V=1000, dtype="fp32",
                 sigma_t=2.0, peak=0.0, zipf_s=1.1, noise=("fixed", 0.5),
                 modes=("greedy", "sample")),
    WorkloadSpec("dflash_b1_l16_v151936", B=1, max_len=16, ragged=False, V=151936, dtype="bf16",
                 sigma_t=3.0, peak=8.0, zipf_s=1.1, noise=("fixed", 1.0)),
    WorkloadSpec("conc32_l16_v151936", B=32, max_len=16, ragged=False, V=151936, dtype="bf16",
                 sigma_t=3.0, peak=8.0, zipf_s=1.1, noise=("uniform", 0.3, 2.0),
                 modes=("greedy", "sample")),
    WorkloadSpec("dspark_ragged_b256_v129280", B=256, max_len=16, ragged=True, V=129280,
                 dtype="bf16", sigma_t=3.0, peak=8.0, zipf_s=1.1, noise=("uniform", 0.3, 2.0),
                 modes=("sample",)),
    WorkloadSpec("filtered_b512_l16_v262144", B=512, max_len=16, ragged=False, V=262144,
                 dtype="bf16", sigma_t=3.0, peak=8.0, zipf_s=1.1, noise=("uniform", 0.3, 2.0),
                 top_k=20, top_p=0.95, modes=("sample",)),
]


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(1000 * int(seed) + int(stream))
    return g


def _zipf_cdf(V: int, s: float, device) -> torch.Tensor:
    w = torch.arange(1, V + 1, dtype=torch.float64, device=device).pow(-s)
    c = torch.cumsum(w, 0)
    return c / c[-1]


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    mode: int
    target: torch.Tensor        # (N_t, V) bf16 or fp32
    draft: torch.Tensor         # (N_d, V)
    draft_tokens: torch.Tensor  # (N_d,) int32
    uniforms: torch.Tensor      # (N_t,) float32
    verify_lens: torch.Tensor   # (B,) int32
    row_offsets: torch.Tensor   # (B+1,) int32

    @property
    def B(self):
        return self.verify_lens.numel()

    @property
    def V(self):
        return self.target.shape[1]

    @property
    def n_target_rows(self):
        return self.target.shape[0]

    @property
    def n_draft_rows(self):
        return self.draft.shape[0]

    def logit_bytes(self) -> int:
        return (self.target.numel() + self.draft.numel()) * self.target.element_size()


def make_workload(spec: WorkloadSpec, mode: int = SAMPLE, seed: int = 0, device="cpu",
                  *, B: int | None = None, V: int | None = None, lens=None,
                  chunk_rows: int = 512) -> Workload:
    """Draw one workload.  ``B``, ``V`` and ``lens`` override the spec (tests
    use them for small cases); ``lens`` is an explicit list of l_r."""
    device = torch.device(device)
    B = spec.B if B is None else B
    V = spec.V if V is None else V
    if lens is not None:
        lens_t = torch.as_tensor(list(lens), dtype=torch.int64, device=device)
        B = lens_t.numel()
    elif spec.ragged:
        lens_t = torch.randint(1, spec.max_len + 1, (B,), generator=_gen(seed, 4, device),
                               device=device)
    else:
        lens_t = torch.full((B,), spec.max_len, dtype=torch.int64, device=device)
    offsets = torch.zeros(B + 1, dtype=torch.int64, device=device)
    offsets[1:] = torch.cumsum(lens_t, 0)
    N_t = int(offsets[-1])
    N_d = N_t - B

    if spec.noise[0] == "fixed":
        sig_r = torch.full((B,), float(spec.noise[1]), dtype=torch.float32, device=device)
    else:
        lo, hi = spec.noise[1], spec.noise[2]
        sig_r = lo + (hi - lo) * torch.rand(B, generator=_gen(seed, 3, device), device=device)

    # request id of every target row, and whether the row has a draft partner
    req_of_row = torch.repeat_interleave(torch.arange(B, device=device), lens_t)
    j_in_req = torch.arange(N_t, device=device) - offsets[req_of_row]
    has_draft = j_in_req < (lens_t[req_of_row] - 1)
    drafted_rows = torch.nonzero(has_draft).flatten()  # target row of each draft row, in order

    store = torch.bfloat16 if spec.dtype == "bf16" else torch.float32
    target = torch.empty((N_t, V), dtype=store, device=device)
    draft = torch.empty((N_d, V), dtype=store, device=device)
    g_t, g_d, g_p = _gen(seed, 0, device), _gen(seed, 1, device), _gen(seed, 2, device)
    cdf = _zipf_cdf(V, spec.zipf_s, device) if spec.peak else None
    d_next = 0
    for r0 in range(0, N_t, chunk_rows):
        r1 = min(N_t, r0 + chunk_rows)
        t = torch.randn((r1 - r0, V), generator=g_t, device=device) * spec.sigma_t
        if spec.peak:
            u = torch.rand(r1 - r0, generator=g_p, device=device, dtype=torch.float64)
            ids = torch.searchsorted(cdf, u).clamp_(max=V - 1)
            t[torch.arange(r1 - r0, device=device), ids] += spec.peak
        target[r0:r1] = t.to(store)
        sel = torch.nonzero(has_draft[r0:r1]).flatten()
        if sel.numel():
            n = torch.randn((sel.numel(), V), generator=g_d, device=device)
            sig = sig_r[req_of_row[r0 + sel]].unsqueeze(1)
            draft[d_next:d_next + sel.numel()] = (t[sel] + sig * n).to(store)
            d_next += sel.numel()
        del t
    assert d_next == N_d

    draft_tokens = _draw_draft_tokens(draft, spec, mode, seed, device, chunk_rows)
    g_u = _gen(seed, 6, device)
    k = torch.randint(0, 1 << 23, (N_t,), generator=g_u, device=device)
    uniforms = ((k.to(torch.float64) + 0.5) * 2.0 ** -23).to(torch.float32)
    del drafted_rows
    return Workload(spec, mode, target, draft, draft_tokens, uniforms,
                    lens_t.to(torch.int32), offsets.to(torch.int32))


def _draw_draft_tokens(draft, spec, mode, seed, device, chunk_rows):
    N_d, V = draft.shape
    out = torch.empty(N_d, dtype=torch.int32, device=device)
    g = _gen(seed, 5, device)
    T = spec.temperature
    for r0 in range(0, N_d, chunk_rows):
        r1 = min(N_d, r0 + chunk_rows)
        d = draft[r0:r1].float()
        if mode == GREEDY:
            out[r0:r1] = torch.argmax(d, dim=1).to(torch.int32)
            continue
        if 0 < spec.top_k < V:
            vals, idx = torch.topk(d, spec.top_k, dim=1)
        else:
            vals, idx = d, None
        e = torch.rand(vals.shape, generator=g, device=device, dtype=torch.float32)
        e = e.clamp_(min=2.0 ** -30)
        gumbel = -torch.log(-torch.log(e))
        pick = torch.argmax(vals / T + gumbel, dim=1)
        out[r0:r1] = (pick if idx is None else idx.gather(1, pick[:, None])[:, 0]).to(torch.int32)
    return out


def round_to_bf16_bits(x: torch.Tensor) -> torch.Tensor:
    """float tensor -> int16 view of its bf16 (round-to-nearest-even) bits."""
    return x.to(torch.bfloat16).view(torch.int16)


def bits_of(t: torch.Tensor):
    """Host numpy view of stored logits as the oracle reads them (uint16 bits
    for bf16, float32 otherwise)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def dtype_name(t: torch.Tensor) -> str:
    return "bf16" if t.dtype == torch.bfloat16 else "fp32"


def expected_bytes(spec: WorkloadSpec) -> int:
    esize = 2 if spec.dtype == "bf16" else 4
    mean_len = (spec.max_len + 1) / 2 if spec.ragged else spec.max_len
    return int(math.ceil((2 * mean_len - 1) * spec.B * spec.V * esize))
