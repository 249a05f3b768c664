"""The C-ABI library loads, exports every declared symbol, and rejects
invalid host arguments before touching a device (no compute calls here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_16_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for f in sorted(os.listdir(HEADER_DIR)):
        if f.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(spec_verify\w*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("spec_verify", "spec_verify_rows", "spec_verify_finalize",
              "spec_verify_workspace_size", "spec_verify_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    lib.spec_verify_status_string.restype = ctypes.c_char_p
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.spec_verify_status_string(code)
    assert lib.spec_verify_status_string(123) == b"unknown status"


def test_workspace_size(lib):
    lib.spec_verify_workspace_size.restype = ctypes.c_size_t
    lib.spec_verify_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int32]
    a = lib.spec_verify_workspace_size(32, 512)
    b = lib.spec_verify_workspace_size(32, 1024)
    assert a % 256 == 0 and b % 256 == 0 and b > a >= 512 * 32


def _call(lib, **over):
    """Call spec_verify with fake (never dereferenced) pointers; the host
    checks must reject the arguments before anything is enqueued."""
    fake = 1 << 20  # 16- and 256-byte aligned, never dereferenced
    a = dict(target=fake, draft=fake, tokens=fake, uniforms=fake, lens=fake, offs=fake,
             B=2, V=1000, Nt=8, max_len=4, dtype=0, T=1.0, top_k=0, top_p=1.0, mode=1,
             out_tokens=fake, out_acc=fake, out_conf=fake, out_stats=None, dev_error=None,
             ws=fake, ws_bytes=1 << 20, stream=None)
    a.update(over)
    f = lib.spec_verify
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    f.argtypes = [vp] * 6 + [i32] * 4 + [i32, f32, i32, f32, i32] + [vp] * 5 + \
        [vp, ctypes.c_size_t, vp]
    f.restype = ctypes.c_int
    return f(a["target"], a["draft"], a["tokens"], a["uniforms"], a["lens"], a["offs"],
             a["B"], a["V"], a["Nt"], a["max_len"], a["dtype"], a["T"], a["top_k"], a["top_p"],
             a["mode"], a["out_tokens"], a["out_acc"], a["out_conf"], a["out_stats"],
             a["dev_error"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(dtype=7), -2),
    (dict(B=0), -1),
    (dict(V=0), -1),
    (dict(Nt=1), -1),                 # fewer target rows than requests
    (dict(max_len=0), -1),
    (dict(max_len=257), -1),
    (dict(Nt=9, max_len=4), -1),      # more rows than B * max_len
    (dict(mode=3), -1),
    (dict(T=0.0), -1),                # sampling needs T > 0
    (dict(T=float("nan")), -1),
    (dict(top_p=0.0), -1),
    (dict(top_p=1.5), -1),
    (dict(target=None), -1),
    (dict(draft=None), -1),           # N_d = 6 > 0 needs draft logits
    (dict(uniforms=None), -1),
    (dict(out_tokens=None), -1),
    (dict(target=(1 << 20) + 8), -1),  # logits must be 16-byte aligned
    (dict(tokens=(1 << 20) + 2), -1),
    (dict(ws=None), -5),
    (dict(ws=(1 << 20) + 128), -5),   # workspace must be 256-byte aligned
    (dict(ws_bytes=64), -5),
    (dict(V=(1 << 21) + 8, top_p=0.9), -4),  # general filter path beyond its V limit
])
def test_host_argument_checks(lib, over, code):
    assert _call(lib, **over) == code


def test_greedy_without_labels_accepts_any_temperature(lib):
    # T is not used in greedy mode without labels or statistics: the host
    # checks pass, so the call reaches the device stage; stop it there by an
    # undersized workspace to keep this a host-only test.
    assert _call(lib, mode=0, T=0.0, out_conf=None, ws_bytes=64) == -5


def test_static_entry_rejects_oversized_problem_before_any_device_call(lib):
    """The no-allocation entry point refuses more target rows than its static
    scratch holds, before it looks up a device."""
    fake = 1 << 20
    f = lib.spec_verify_static
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    f.argtypes = [vp] * 6 + [i32] * 4 + [i32, f32, i32, f32, i32] + [vp] * 5 + [vp]
    f.restype = ctypes.c_int
    B, max_len = 512, 16
    for nt, code in ((4097, -6), (8192, -6)):
        assert f(fake, fake, fake, fake, fake, fake, B, 151936, nt, max_len, 0, 1.0, 0, 1.0, 1,
                 fake, fake, fake, None, None, None) == code


def test_schedule_rejects_bad_host_arguments(lib):
    """spec_verify_schedule checks its arguments on the host (fake pointers,
    never dereferenced: every call below must be refused first)."""
    f = lib.spec_verify_schedule
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    p, q = 0x10000, 0x20000
    assert f(p, 0, 4, q, 10, p, None, None) == -1            # B < 1
    assert f(p, 4, -1, q, 10, p, None, None) == -1           # K < 0
    assert f(p, 4, 3, q, 4, p, None, None) == -1             # no SPS entry beyond B
    assert f(None, 4, 3, q, 10, p, None, None) == -1         # conf missing
    assert f(p, 4, 3, None, 10, p, None, None) == -1         # sps missing
    assert f(p, 4, 3, q, 10, None, None, None) == -1         # out_lens missing
    assert f(p, 4, 3, q + 4, 10, p, None, None) == -1        # sps not 8-byte aligned
    assert f(p, 1000, 9, q, 10000, p, None, None) == -4      # above SV_SCHEDULE_MAX_CANDIDATES


def test_static_entry_checks_arguments_before_anything_else(lib):
    """A first call of the no-allocation entry point with a bad argument
    returns SV_ERR_ARG from its host checks, before it looks up its array or
    enqueues its clear (no device call happens: this runs without a GPU)."""
    fake = 1 << 20
    f = lib.spec_verify_static
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    f.argtypes = [vp] * 6 + [i32] * 4 + [i32, f32, i32, f32, i32] + [vp] * 5 + [vp]
    f.restype = ctypes.c_int
    assert f(fake, fake, fake, fake, fake, fake, 2, 1000, 8, 4, 0, 0.0, 0, 1.0, 1,
             fake, fake, fake, None, None, None) == -1  # sampling with T = 0
    assert f(None, fake, fake, fake, fake, fake, 2, 1000, 8, 4, 0, 1.0, 0, 1.0, 1,
             fake, fake, fake, None, None, None) == -1  # no target logits


def test_set_tuning_checks_knobs(lib):
    f = lib.spec_verify_set_tuning
    f.argtypes = [ctypes.c_int32, ctypes.c_int64]
    f.restype = ctypes.c_int
    assert f(99, 1) == -1              # unknown knob
    assert f(1, 3) == -1               # fewer stages than the pipeline allows
    assert f(2, 20) == -1              # consumer warps are 16 or 24
    assert f(5, 10 ** 12) == -1        # cross-CTA wait limit above 200 ms
    for knob in range(6):              # defaults restore
        assert f(knob, -1) == 0
    assert f(4, 256) == 0 and f(4, -1) == 0
