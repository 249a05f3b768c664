"""ctypes binding of libspecverify.so (the C ABI in include/spec_verify.h).

Argument marshalling only: every step of the verify path runs in the
library's kernels.  torch is used for device memory (outputs, workspace)
and for the current CUDA stream.  Importing this module fails loudly when
the library has not been built -- there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspecverify.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -m "
        "speculative_decoding_verification_16_gb300.build, or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

SV_BF16, SV_FP32 = 0, 1
SV_GREEDY, SV_SAMPLE = 0, 1
SV_OK = 0
SV_ERR_TOO_LARGE = -6
SV_STATIC_MAX_ROWS = 4096
SV_DEVERR_NAN, SV_DEVERR_TOKEN, SV_DEVERR_LEN, SV_DEVERR_TIMEOUT = 1, 2, 4, 8

_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
_ARGTYPES = [_vp, _vp, _vp, _vp, _vp, _vp,            # logits, tokens, uniforms, lens, offsets
             _i32, _i32, _i32, _i32,                  # B, V, n_target_rows, max_len
             _i32, _f32, _i32, _f32, _i32,            # dtype, T, top_k, top_p, mode
             _vp, _vp, _vp, _vp, _vp,                 # outputs, dev_error
             _vp, _sz, _vp]                           # workspace, bytes, stream
for _name in ("spec_verify", "spec_verify_rows", "spec_verify_finalize"):
    _fn = getattr(_lib, _name)
    _fn.argtypes = _ARGTYPES
    _fn.restype = ctypes.c_int
_lib.spec_verify_static.argtypes = _ARGTYPES[:20] + [_vp]   # no workspace arguments
_lib.spec_verify_static.restype = ctypes.c_int
_lib.spec_verify_workspace_size.argtypes = [_i32, _i32]
_lib.spec_verify_workspace_size.restype = ctypes.c_size_t
_lib.spec_verify_status_string.argtypes = [ctypes.c_int]
_lib.spec_verify_status_string.restype = ctypes.c_char_p
_lib.spec_verify_slices_per_row.argtypes = [_i32, _i32, _i32, _f32]
_lib.spec_verify_slices_per_row.restype = ctypes.c_int
_lib.spec_verify_schedule.argtypes = [_vp, _i32, _i32, _vp, _i32, _vp, _vp, _vp]
_lib.spec_verify_schedule.restype = ctypes.c_int
SV_SCHEDULE_MAX_CANDIDATES = 8192


SV_TUNE_SLICE, SV_TUNE_STAGES, SV_TUNE_WARPS, SV_TUNE_PASS1_WARPS = 0, 1, 2, 3
SV_TUNE_POLL_NS, SV_TUNE_XWAIT_NS = 4, 5
_lib.spec_verify_set_tuning.argtypes = [_i32, ctypes.c_int64]
_lib.spec_verify_set_tuning.restype = ctypes.c_int


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"spec_verify failed ({status}): {spec_verify_status_string(status)}")
        self.status = status


def spec_verify_set_tuning(knob: int, value: int) -> None:
    """Process-wide tuning knob of the rows kernel (tests and sweeps);
    ``value`` < 0 restores the default."""
    rc = _lib.spec_verify_set_tuning(int(knob), int(value))
    if rc != SV_OK:
        raise SpecVerifyError(rc)


def spec_verify_status_string(status: int) -> str:
    return _lib.spec_verify_status_string(int(status)).decode()


def spec_verify_workspace_size(B: int, n_target_rows: int) -> int:
    return int(_lib.spec_verify_workspace_size(int(B), int(n_target_rows)))


def spec_verify_slices_per_row(V: int, dtype: int, top_k: int = 0, top_p: float = 1.0) -> int:
    return int(_lib.spec_verify_slices_per_row(int(V), int(dtype), int(top_k), float(top_p)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_FP32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


class Outputs:
    """Device output buffers of one call."""

    def __init__(self, tokens, accept_len, conf, row_stats, dev_error):
        self.tokens = tokens
        self.accept_len = accept_len
        self.conf = conf
        self.row_stats = row_stats
        self.dev_error = dev_error


def alloc_outputs(n_target_rows: int, B: int, device, want_conf=True, want_stats=False):
    Nd = n_target_rows - B
    return Outputs(
        torch.empty(n_target_rows, dtype=torch.int32, device=device),
        torch.empty(B, dtype=torch.int32, device=device),
        torch.empty(Nd, dtype=torch.float32, device=device) if want_conf else None,
        torch.empty((n_target_rows + Nd, 3), dtype=torch.float32, device=device)
        if want_stats else None,
        torch.zeros(1, dtype=torch.int32, device=device))


def alloc_workspace(B: int, n_target_rows: int, device) -> torch.Tensor:
    """Device workspace for calls with these sizes, zeroed as the C ABI
    requires before its first use."""
    return torch.zeros(spec_verify_workspace_size(B, n_target_rows), dtype=torch.uint8,
                       device=device)


class PreparedCall:
    """A call with its arguments marshalled once; ``__call__`` re-issues it
    (used by timing loops, where per-call marshalling would dominate).  The
    call runs with the tensors' device current, as the C ABI requires."""

    def __init__(self, fn, args, device):
        self._fn = fn
        self._args = args
        self._device = device

    def __call__(self):
        if torch.cuda.current_device() != self._device:
            with torch.cuda.device(self._device):
                rc = self._fn(*self._args)
        else:
            rc = self._fn(*self._args)
        if rc != SV_OK:
            raise SpecVerifyError(rc)


def prepare(entry: str, target_logits, draft_logits, draft_tokens, uniforms, verify_lens,
            row_offsets, *, max_len, temperature=1.0, top_k=0, top_p=1.0, mode=SV_SAMPLE,
            out: Outputs, workspace: torch.Tensor, stream=None) -> PreparedCall:
    """Marshal the arguments of one C entry point (``spec_verify``,
    ``spec_verify_rows`` or ``spec_verify_finalize``)."""
    B = verify_lens.numel()
    n_target_rows, V = target_logits.shape
    if stream is None:
        stream = torch.cuda.current_stream(target_logits.device)
    args = (_ptr(target_logits), _ptr(draft_logits) if draft_logits.numel() else None,
            _ptr(draft_tokens) if draft_tokens.numel() else None, _ptr(uniforms),
            _ptr(verify_lens), _ptr(row_offsets),
            _i32(B), _i32(V), _i32(n_target_rows), _i32(max_len),
            _i32(_dtype_code(target_logits)), _f32(temperature), _i32(top_k), _f32(top_p),
            _i32(mode),
            _ptr(out.tokens), _ptr(out.accept_len), _ptr(out.conf), _ptr(out.row_stats),
            _ptr(out.dev_error), _ptr(workspace), _sz(workspace.numel()),
            ctypes.c_void_p(stream.cuda_stream))
    return PreparedCall(getattr(_lib, entry), args, target_logits.device.index)


def spec_verify(target_logits, draft_logits, draft_tokens, uniforms, verify_lens, row_offsets,
                *, max_len=16, temperature=1.0, top_k=0, top_p=1.0, mode=SV_SAMPLE,
                want_conf=True, want_stats=False, out: Outputs | None = None,
                workspace: torch.Tensor | None = None, stream=None) -> Outputs:
    """One verify call on the current (or given) stream; returns device
    outputs without synchronising.  Tensors must be contiguous CUDA tensors:
    logits bf16/fp32 [N_t, V] and [N_d, V], int32 tokens/lengths/offsets,
    float32 uniforms."""
    for t in (target_logits, draft_logits, draft_tokens, uniforms, verify_lens, row_offsets):
        if not t.is_contiguous():
            raise ValueError("inputs must be contiguous")
    B = verify_lens.numel()
    n_target_rows = target_logits.shape[0]
    dev = target_logits.device
    if out is None:
        out = alloc_outputs(n_target_rows, B, dev, want_conf, want_stats)
    else:
        out.dev_error.zero_()
    if workspace is None:
        workspace = alloc_workspace(B, n_target_rows, dev)
    prepare("spec_verify", target_logits, draft_logits, draft_tokens, uniforms, verify_lens,
            row_offsets, max_len=max_len, temperature=temperature, top_k=top_k, top_p=top_p,
            mode=mode, out=out, workspace=workspace, stream=stream)()
    return out


def spec_verify_static(target_logits, draft_logits, draft_tokens, uniforms, verify_lens,
                       row_offsets, *, max_len=16, temperature=1.0, top_k=0, top_p=1.0,
                       mode=SV_SAMPLE, out: Outputs, stream=None) -> Outputs:
    """The C entry point that allocates nothing (scratch in the library's
    static device array).  ``out`` must be given: this path allocates no
    device memory, not even through torch."""
    for t in (target_logits, draft_logits, draft_tokens, uniforms, verify_lens, row_offsets):
        if not t.is_contiguous():
            raise ValueError("inputs must be contiguous")
    B = verify_lens.numel()
    n_target_rows, V = target_logits.shape
    if stream is None:
        stream = torch.cuda.current_stream(target_logits.device)
    out.dev_error.zero_()  # this call's flags only (a kernel on the stream, no allocation)
    # the library picks the static array of the current device
    with torch.cuda.device(target_logits.device):
        rc = _call_static(target_logits, draft_logits, draft_tokens, uniforms, verify_lens,
                          row_offsets, B, V, n_target_rows, max_len, temperature, top_k, top_p,
                          mode, out, stream)
    if rc != SV_OK:
        raise SpecVerifyError(rc)
    return out


def _call_static(target_logits, draft_logits, draft_tokens, uniforms, verify_lens, row_offsets,
                 B, V, n_target_rows, max_len, temperature, top_k, top_p, mode, out, stream):
    return _lib.spec_verify_static(
        _ptr(target_logits), _ptr(draft_logits) if draft_logits.numel() else None,
        _ptr(draft_tokens) if draft_tokens.numel() else None, _ptr(uniforms),
        _ptr(verify_lens), _ptr(row_offsets),
        _i32(B), _i32(V), _i32(n_target_rows), _i32(max_len),
        _i32(_dtype_code(target_logits)), _f32(temperature), _i32(top_k), _f32(top_p),
        _i32(mode),
        _ptr(out.tokens), _ptr(out.accept_len), _ptr(out.conf), _ptr(out.row_stats),
        _ptr(out.dev_error), ctypes.c_void_p(stream.cuda_stream))


def verify_workload(w, *, want_conf=True, want_stats=False, **kw) -> Outputs:
    """Run the library on a ``workloads.Workload`` held on a CUDA device."""
    spec = w.spec
    return spec_verify(w.target, w.draft, w.draft_tokens, w.uniforms, w.verify_lens,
                       w.row_offsets, max_len=kw.pop("max_len", spec.max_len),
                       temperature=kw.pop("temperature", spec.temperature),
                       top_k=kw.pop("top_k", spec.top_k), top_p=kw.pop("top_p", spec.top_p),
                       mode=kw.pop("mode", w.mode), want_conf=want_conf, want_stats=want_stats,
                       **kw)


def spec_verify_schedule(conf: torch.Tensor, sps: torch.Tensor, *, out_lens=None,
                         out_theta=None, stream=None):
    """DSpark prefix schedule of a pool: ``conf`` [B, K] float32 (survival
    probability of each drafted position), ``sps`` [n] float64 (steps per
    second at each batch size).  Returns (lens int32 [B], theta float64 [2]:
    Theta and the number of candidates added), all on the device."""
    assert conf.dim() == 2 and conf.dtype == torch.float32 and conf.is_contiguous()
    assert sps.dim() == 1 and sps.dtype == torch.float64 and sps.is_contiguous()
    B, K = conf.shape
    dev = conf.device
    if out_lens is None:
        out_lens = torch.empty(B, dtype=torch.int32, device=dev)
    if out_theta is None:
        out_theta = torch.empty(2, dtype=torch.float64, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    rc = _lib.spec_verify_schedule(_ptr(conf) if conf.numel() else None, _i32(B), _i32(K),
                                   _ptr(sps), _i32(sps.numel()), _ptr(out_lens),
                                   _ptr(out_theta), ctypes.c_void_p(stream.cuda_stream))
    if rc != SV_OK:
        raise SpecVerifyError(rc)
    return out_lens, out_theta



# ---- the verify step over a vocabulary split across ranks
#      (include/spec_verify_shard.h)

SV_SHARD_MAX_WORLD = 32
SV_SHARD_REC_WORDS, SV_SHARD_ROW_WORDS, SV_SHARD_MASS_WORDS = 12, 8, 4
_lib.spec_verify_shard_stats.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp,
                                         _i32, _i32, _i32, _i32, _f32, _vp, _vp]
_lib.spec_verify_shard_merge.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                         _f32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.spec_verify_shard_masses.argtypes = [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                          _i32, _f32, _i32, _vp, _vp]
_lib.spec_verify_shard_draw.argtypes = [_vp, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp,
                                        _vp, _vp, _i32, _i32, _i32, _i32, _f32, _i32, _vp, _vp,
                                        _vp, _vp]
_lib.spec_verify_shard_finish.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp,
                                          _vp]
for _name in ("spec_verify_shard_stats", "spec_verify_shard_merge", "spec_verify_shard_masses",
              "spec_verify_shard_draw", "spec_verify_shard_finish"):
    getattr(_lib, _name).restype = ctypes.c_int


def _check(rc):
    if rc != SV_OK:
        raise SpecVerifyError(rc)


def _stream_of(t, stream):
    s = torch.cuda.current_stream(t.device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def spec_verify_shard_stats(target_shard, draft_shard, v_begin, V, draft_tokens, verify_lens,
                            row_offsets, *, max_len, temperature, out_rec, stream=None):
    """Step 1 on this rank: partial statistics of its columns (target_shard
    [N_t, V_q], draft_shard [N_d, V_q], ids v_begin .. v_begin + V_q - 1 of
    a vocabulary of V) into out_rec [N_t, 12] int32."""
    n_t, vq = target_shard.shape
    with torch.cuda.device(target_shard.device):
        _check(_lib.spec_verify_shard_stats(
            _ptr(target_shard), _ptr(draft_shard) if draft_shard.numel() else None, _i32(vq),
            _i32(v_begin), _i32(V), _ptr(draft_tokens) if draft_tokens.numel() else None,
            _ptr(verify_lens), _ptr(row_offsets), _i32(verify_lens.numel()), _i32(n_t),
            _i32(max_len), _i32(_dtype_code(target_shard)), _f32(temperature), _ptr(out_rec),
            _stream_of(target_shard, stream)))


def spec_verify_shard_merge(recs, draft_tokens, uniforms, verify_lens, row_offsets, V, *,
                            max_len, temperature, mode, out_merged, out: Outputs, stream=None):
    """Step 1 on every rank: merge the gathered records recs [world, N_t, 12]."""
    world, n_t, _ = recs.shape
    with torch.cuda.device(recs.device):
        _check(_lib.spec_verify_shard_merge(
            _ptr(recs), _i32(world), _ptr(draft_tokens) if draft_tokens.numel() else None,
            _ptr(uniforms), _ptr(verify_lens), _ptr(row_offsets), _i32(verify_lens.numel()),
            _i32(V), _i32(n_t), _i32(max_len), _f32(temperature), _i32(mode), _ptr(out_merged),
            _ptr(out.tokens), _ptr(out.accept_len), _ptr(out.row_stats), _ptr(out.dev_error),
            _stream_of(recs, stream)))


def spec_verify_shard_masses(target_shard, draft_shard, merged, verify_lens, row_offsets,
                             accept_len, *, max_len, temperature, all_rows, out_mass,
                             stream=None):
    """Step 2 on this rank: its shares of the masses into out_mass [N_t, 4]."""
    n_t, vq = target_shard.shape
    with torch.cuda.device(target_shard.device):
        _check(_lib.spec_verify_shard_masses(
            _ptr(target_shard), _ptr(draft_shard) if draft_shard.numel() else None, _i32(vq),
            _ptr(merged), _ptr(verify_lens), _ptr(row_offsets), _ptr(accept_len),
            _i32(verify_lens.numel()), _i32(n_t), _i32(max_len), _i32(_dtype_code(target_shard)),
            _f32(temperature), _i32(1 if all_rows else 0), _ptr(out_mass),
            _stream_of(target_shard, stream)))


def spec_verify_shard_draw(masses, rank, target_shard, draft_shard, v_begin, merged, uniforms,
                           verify_lens, row_offsets, *, max_len, temperature, mode,
                           out: Outputs, out_cand, stream=None):
    """Step 3 on every rank: labels into out.conf and, sampling, this rank's
    candidate token per request into out_cand [B] (-1 where another rank
    owns the draw)."""
    world = masses.shape[0]
    n_t, vq = target_shard.shape
    with torch.cuda.device(target_shard.device):
        _check(_lib.spec_verify_shard_draw(
            _ptr(masses), _i32(world), _i32(rank), _ptr(target_shard),
            _ptr(draft_shard) if draft_shard.numel() else None, _i32(vq), _i32(v_begin),
            _ptr(merged), _ptr(uniforms), _ptr(verify_lens), _ptr(row_offsets),
            _ptr(out.accept_len), _i32(verify_lens.numel()), _i32(n_t), _i32(max_len),
            _i32(_dtype_code(target_shard)), _f32(temperature), _i32(mode), _ptr(out.conf),
            _ptr(out_cand), _ptr(out.dev_error), _stream_of(target_shard, stream)))


def spec_verify_shard_finish(cands, merged, verify_lens, row_offsets, *, out: Outputs,
                             stream=None):
    """Step 3 on every rank: the final tokens from the gathered candidates
    cands [world, B]."""
    world, B = cands.shape
    with torch.cuda.device(cands.device):
        _check(_lib.spec_verify_shard_finish(
            _ptr(cands), _i32(world), _ptr(merged), _ptr(verify_lens), _ptr(row_offsets),
            _ptr(out.accept_len), _i32(B), _i32(out.tokens.numel()), _ptr(out.tokens),
            _ptr(out.dev_error), _stream_of(cands, stream)))
