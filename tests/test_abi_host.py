"""The C ABI library loads, exports what include/epd.h declares, and rejects bad
arguments on the host before any launch (no GPU needed: none of these calls
reaches the CUDA runtime)."""
import ctypes
import os
import re

import pytest

from unpermute_ep_dispatch_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "epd.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _binding.load_library()


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"^EPD_API\s+[\w\s\*]+?\**\s*(\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("ep_dispatch_layout", "ep_scan_offsets", "ep_permute", "ep_unpermute",
              "epd_workspace_bytes", "epd_workspace_init"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
        assert n in _binding.SIGNATURES, f"binding lacks {n}"
    assert set(_binding.SIGNATURES) == set(names)


def test_status_strings_and_version(lib):
    assert _binding.status_string(0) == "ok"
    assert "look-back" in _binding.status_string(_binding.EPD_ERR_TIMEOUT)
    assert _binding.status_string(99) == "unknown status"
    assert _binding.version() >= 10000


def test_workspace_bytes(lib):
    n = lib.epd_workspace_bytes(8192, 8, 256, 32, 4)
    assert n >= 8192 * 8 * 4 and n % 256 == 0
    assert lib.epd_workspace_bytes(0, 8, 256, 32, 4) > 0
    assert lib.epd_workspace_bytes(64, 2, 16, 8, 2) > 0
    # invalid topologies give 0
    assert lib.epd_workspace_bytes(64, 2, 16, 3, 1) == 0      # E % R
    assert lib.epd_workspace_bytes(64, 2, 16, 8, 3) == 0      # R % N
    assert lib.epd_workspace_bytes(-1, 2, 16, 8, 2) == 0
    assert lib.epd_workspace_bytes(64, 65, 16, 8, 2) == 0     # k > EPD_MAX_TOPK
    assert lib.epd_workspace_bytes(64, 2, 8192, 8, 2) == 0    # E > EPD_MAX_EXPERTS
    # grows with T*k
    assert lib.epd_workspace_bytes(1 << 20, 8, 256, 32, 4) > (1 << 20) * 8 * 4


NULL = None
FAKE = ctypes.c_void_p(0x10000)        # aligned, never dereferenced: rejected before launch
FAKE_ODD = ctypes.c_void_p(0x10004)    # 4-aligned, not 16-aligned


def test_layout_rejects_bad_args(lib):
    E = _binding.EPD_ERR_INVALID_ARG
    f = lib.ep_dispatch_layout
    # E % R != 0
    assert f(FAKE, 4, 2, 16, 3, 1, FAKE, FAKE, NULL, NULL, FAKE, FAKE, NULL) == E
    # null counts / workspace / status
    assert f(FAKE, 4, 2, 16, 8, 2, NULL, FAKE, NULL, NULL, FAKE, FAKE, NULL) == E
    assert f(FAKE, 4, 2, 16, 8, 2, FAKE, FAKE, NULL, NULL, NULL, FAKE, NULL) == E
    assert f(FAKE, 4, 2, 16, 8, 2, FAKE, FAKE, NULL, NULL, FAKE, NULL, NULL) == E
    # null topk with work to do
    assert f(NULL, 4, 2, 16, 8, 2, FAKE, FAKE, NULL, NULL, FAKE, FAKE, NULL) == E
    # k beyond the limit, negative T
    assert f(FAKE, 4, 65, 16, 8, 2, FAKE, FAKE, NULL, NULL, FAKE, FAKE, NULL) == E
    assert f(FAKE, -1, 2, 16, 8, 2, FAKE, FAKE, NULL, NULL, FAKE, FAKE, NULL) == E


def test_scan_rejects_bad_args(lib):
    E = _binding.EPD_ERR_INVALID_ARG
    assert lib.ep_scan_offsets(FAKE, 0, FAKE, FAKE, FAKE, NULL) == E
    assert lib.ep_scan_offsets(FAKE, 5000, FAKE, FAKE, FAKE, NULL) == E
    assert lib.ep_scan_offsets(NULL, 16, FAKE, FAKE, FAKE, NULL) == E
    assert lib.ep_scan_offsets(FAKE, 16, FAKE, NULL, FAKE, NULL) == E


def test_permute_rejects_bad_args(lib):
    E = _binding.EPD_ERR_INVALID_ARG
    f = lib.ep_permute
    ok = dict(x=FAKE, dt=0, xs=NULL, topk=FAKE, T=4, k=2, H=64, E=8, start=FAKE, ws=FAKE,
              cap=8, out=FAKE, outs=NULL, mi=FAKE, oi=FAKE, st=FAKE, s=NULL)

    def call(**kw):
        a = dict(ok, **kw)
        return f(*a.values())
    assert call(cap=7) == E                      # capacity below T*k
    assert call(H=60) == E                       # bf16 rows need H % 8
    assert call(xs=FAKE) == E                    # bf16 takes no scales
    assert call(dt=1, H=64, xs=FAKE, outs=FAKE) == E   # fp8 needs H % 128
    assert call(dt=1, H=128) == E                # fp8 without scales
    assert call(dt=7) == E                       # unknown dtype
    assert call(x=FAKE_ODD) == E                 # rows must be 16-byte aligned
    assert call(out=FAKE_ODD) == E
    assert call(ws=NULL) == E
    assert call(st=NULL) == E
    assert call(cap=1 << 40) == E                # beyond int32 rows


def test_unpermute_rejects_bad_args(lib):
    E = _binding.EPD_ERR_INVALID_ARG
    f = lib.ep_unpermute
    assert f(FAKE, 8, FAKE, FAKE, 4, 2, 60, FAKE, FAKE, NULL) == E     # H % 8
    assert f(FAKE, 8, FAKE, FAKE, 4, 2, 64, FAKE_ODD, FAKE, NULL) == E  # y alignment
    assert f(FAKE_ODD, 8, FAKE, FAKE, 4, 2, 64, FAKE, FAKE, NULL) == E  # eo alignment
    assert f(FAKE, 8, FAKE, FAKE, 4, 2, 64, FAKE, NULL, NULL) == E     # status
    assert f(FAKE, -1, FAKE, FAKE, 4, 2, 64, FAKE, FAKE, NULL) == E    # capacity
    # nothing to do: accepted without touching the GPU
    assert f(NULL, 0, NULL, NULL, 0, 2, 64, NULL, FAKE, NULL) == _binding.EPD_OK


def test_stalled_tile_hook_validates(lib):
    E = _binding.EPD_ERR_INVALID_ARG
    f = lib.epd_test_layout_stalled_tile
    assert f(FAKE, 4, 2, 16, 8, 2, FAKE, FAKE, NULL, NULL, FAKE, FAKE, -1, 100, NULL) == E
    assert f(FAKE, 4, 2, 16, 8, 2, FAKE, FAKE, NULL, NULL, FAKE, FAKE, 0, 1 << 30, NULL) == E
    assert f(FAKE, 4, 2, 16, 8, 2, FAKE, FAKE, NULL, NULL, FAKE, FAKE, 0, 0, NULL) == E


def test_binding_fails_loudly_without_library(tmp_path):
    missing = str(tmp_path / "libepd.so")
    saved = _binding._lib
    _binding._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            _binding.load_library(missing)
    finally:
        _binding._lib = saved


def test_permute_ex_rejects_bad_views(lib):
    E = _binding.EPD_ERR_INVALID_ARG
    f = lib.ep_permute_ex

    def call(view, row_bytes=64, cap=8, xs=NULL, outs=NULL):
        return f(FAKE, row_bytes, xs, FAKE, 4, 2, 8, FAKE, FAKE, cap, ctypes.byref(view), FAKE,
                 outs, FAKE, FAKE, FAKE, NULL)
    V = _binding.PermuteView
    assert f(FAKE, 64, NULL, FAKE, 4, 2, 8, FAKE, FAKE, 8, None, FAKE, NULL, FAKE, FAKE, FAKE,
             NULL) == E                                           # no view
    assert call(V(0, 9, 0, 0, 0)) == E                           # past num_experts
    assert call(V(4, 4, 0, 0, 0)) == E                           # empty range
    assert call(V(-1, 4, 0, 0, 0)) == E
    assert call(V(0, 8, 0, 2, 0)) == E                           # unknown scale layout
    assert call(V(0, 8, 3, 1, 4), xs=FAKE, outs=FAKE) == E       # ld below capacity
    assert call(V(0, 8, 3, 0, 0)) == E                           # scales without pointers
    assert call(V(0, 8, 0, 0, 0), row_bytes=60) == E             # rows not 16-byte multiples
    assert call(V(0, 8, 0, 0, 0), cap=-1) == E


def test_dispatch_rejects_bad_args(lib):
    E = _binding.EPD_ERR_INVALID_ARG
    f = lib.ep_dispatch
    ok = dict(x=FAKE, dt=0, xs=NULL, topk=FAKE, T=4, k=2, H=64, E=8, R=4, N=2, align=1,
              per_e=FAKE, per_r=FAKE, per_n=NULL, itr=NULL, start=FAKE, total=FAKE, ws=FAKE,
              cap=8, out=FAKE, outs=NULL, mi=FAKE, oi=FAKE, st=FAKE, s=NULL)

    def call(**kw):
        a = dict(ok, **kw)
        return f(*a.values())
    assert call(cap=7) == E                      # capacity below T*k
    assert call(cap=1 << 40) == E                # beyond int32 rows
    assert call(H=60) == E                       # bf16 rows need H % 8
    assert call(xs=FAKE) == E                    # bf16 takes no scales
    assert call(dt=1, H=64, xs=FAKE, outs=FAKE) == E   # fp8 needs H % 128
    assert call(dt=1, H=128) == E                # fp8 without scales
    assert call(dt=7) == E                       # unknown dtype
    assert call(R=3) == E                        # E % R
    assert call(N=3) == E                        # R % N
    assert call(align=0) == E
    assert call(align=8192) == E                 # above EPD_MAX_ALIGNMENT
    assert call(x=FAKE_ODD) == E                 # rows must be 16-byte aligned
    assert call(out=FAKE_ODD) == E
    assert call(ws=NULL) == E
    assert call(st=NULL) == E
    assert call(start=NULL) == E
    assert call(total=NULL) == E
    assert call(mi=NULL) == E


def test_dispatch_lowlatency_rejects_bad_args(lib):
    E = _binding.EPD_ERR_INVALID_ARG
    f = lib.ep_dispatch_lowlatency
    ok = dict(x=FAKE, topk=FAKE, T=4, k=2, H=128, E=8, R=4, N=2, b=0, e=8, rows=4, ws=FAKE,
              q=FAKE, qs=FAKE, rc=FAKE, oi=FAKE, src=NULL, st=FAKE, s=NULL)

    def call(**kw):
        a = dict(ok, **kw)
        return f(*a.values())
    assert call(H=64) == E                       # H % 128
    assert call(R=3) == E                        # E % R
    assert call(b=4, e=4) == E                   # empty view
    assert call(e=9) == E                        # view past E
    assert call(rows=-1) == E
    assert call(ws=NULL) == E
    assert call(rc=NULL) == E
    assert call(st=NULL) == E
    assert call(x=FAKE_ODD) == E                 # rows must be 16-byte aligned
    assert call(q=NULL) == E                     # rectangles with rows but no buffer
