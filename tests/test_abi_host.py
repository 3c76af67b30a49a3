"""C-ABI checks that need no GPU: the library builds and loads, exports exactly the
entry points include/gdn.h declares, and rejects bad arguments on the host
before any CUDA call (so a rejected call touches no memory)."""
import ctypes
import os
import re
import subprocess

import pytest

import gated_deltanet_linear_16_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

OK, ARG, UNSUP, ALIGN, ALIAS, CUDA = 0, 1, 2, 3, 4, 5
A = 1 << 20          # fake, 16-byte aligned "device" addresses: never dereferenced by a rejected call


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def built():
    gdn.build()
    return gdn.load()


@pytest.fixture(scope="module")
def lib(built):
    """The library, for calls with fake addresses: only where no CUDA device exists, so a
    call that wrongly passed validation could never reach a real GPU."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("fake-pointer validation tests run only on hosts without a GPU")
    return built


def test_exports_match_header(built):
    want = declared_symbols()
    assert want == sorted(["gdn_decode", "gdn_decode_norm", "gdn_decode_chunk2", "gdn_decode_conv_norm",
                           "gdn_decode_conv_norm_noalloc", "gdn_decode_norm_q8", "gdn_gate_norm",
                           "gdn_gate_norm_q8", "gdn_prefill_seq", "gdn_prefill_chunked", "gdn_device_wait_timeouts", "gdn_set_wait_polls",
                           "gdn_set_mma_wait_polls",
                           "gdn_h_f32_to_f16",
                           "gdn_h_f16_to_f32", "gdn_status_str", "gdn_last_cuda_error"])
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = sorted({line.split()[-1] for line in out.splitlines() if line.split()[-1].startswith("gdn_")})
    assert exported == want
    for name in want:
        assert hasattr(built, name)


def test_status_strings(built):
    for code in range(6):
        assert gdn.gdn_status_str(code).startswith(gdn.STATUS[code])
    assert gdn.gdn_status_str(99) == "GDN_ERR_UNKNOWN"


def decode(lib, **kw):
    a = dict(state=A, dt=0, pitch=48 * 128 * 128, q=A + (1 << 30), k=A + (2 << 30), v=A + (3 << 30),
             alpha=A + (4 << 30), beta=A + (5 << 30), o=A + (6 << 30), batch=2, nk=16, nv=48, d=128,
             qk=16 * 128, vs=48 * 128, gb=48, os=48 * 128)
    a.update(kw)
    return lib.gdn_decode(a["state"], a["dt"], a["pitch"], a["q"], a["k"], a["v"], a["alpha"], a["beta"],
                          a["o"], a["batch"], a["nk"], a["nv"], a["d"], a["qk"], a["vs"], a["gb"], a["os"], None)


def decode_norm(lib, **kw):
    a = dict(state=A, dt=1, pitch=4 * 4 * 4, q=A + (1 << 30), k=A + (2 << 30), v=A + (3 << 30),
             alpha=A + (4 << 30), beta=A + (5 << 30), z=A + (7 << 30), gn=A + (8 << 30), eps=1e-6,
             out=A + (6 << 30), batch=2, nk=1, nv=4, d=4, qk=4, vs=16, gb=4, zs=16, outs=16)
    a.update(kw)
    return lib.gdn_decode_norm(a["state"], a["dt"], a["pitch"], a["q"], a["k"], a["v"], a["alpha"], a["beta"],
                               a["z"], a["gn"], a["eps"], a["out"], a["batch"], a["nk"], a["nv"], a["d"],
                               a["qk"], a["vs"], a["gb"], a["zs"], a["outs"], None)


def chunk2(lib, **kw):
    a = dict(state=A, dt=0, pitch=3 * 128 * 128, mid=A + (9 << 30), mpitch=3 * 128 * 128, q=A + (1 << 30),
             k=A + (2 << 30), v=A + (3 << 30), alpha=A + (4 << 30), beta=A + (5 << 30), o=A + (6 << 30),
             batch=2, nk=1, nv=3, d=128, qk=128, vs=3 * 128, gb=3, os=3 * 128)
    a.update(kw)
    return lib.gdn_decode_chunk2(a["state"], a["dt"], a["pitch"], a["mid"], a["mpitch"], a["q"], a["k"], a["v"],
                                 a["alpha"], a["beta"], a["o"], a["batch"], a["nk"], a["nv"], a["d"], a["qk"],
                                 a["vs"], a["gb"], a["os"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(mid=None), ARG), (dict(mpitch=3 * 128 * 128 - 1), ARG), (dict(dt=3), UNSUP),
    (dict(mid=A + 1024), ALIAS),                         # intermediate state inside the state
    (dict(o=A + (9 << 30) + 64), ALIAS),                 # output inside the intermediate state
    (dict(mid=A + (9 << 30) + 2), ALIGN),                # fp32 intermediate not 4-byte aligned
    (dict(os=100), ARG),
])
def test_chunk2_rejects(lib, kw, want):
    assert chunk2(lib, **kw) == want


def test_chunk2_empty_is_ok(lib):
    assert chunk2(lib, batch=0) == OK


def conv_norm(lib, **kw):
    nk, nv, d, taps = 2, 6, 128, 4
    C = (2 * nk + nv) * d
    a = dict(state=A, dt=0, pitch=nv * d * d, ring=A + (9 << 30), rpitch=taps * C, taps=taps, x=A + (1 << 30),
             w=A + (2 << 30), br=A + (3 << 30), ar=A + (4 << 30), dtb=A + (5 << 30), rate=A + (5 << 30) + 4096,
             z=A + (7 << 30), gn=A + (8 << 30), l2=1e-6, eps=1e-6, out=A + (6 << 30), ws=A + (10 << 30),
             batch=2, nk=nk, nv=nv, d=d, xs=C, gs=nv, zs=nv * d, outs=nv * d)
    a.update(kw)
    return lib.gdn_decode_conv_norm(a["state"], a["dt"], a["pitch"], a["ring"], a["rpitch"], a["taps"], a["x"], a["w"],
                                    a["br"], a["ar"], a["dtb"], a["rate"], a["z"], a["gn"], a["l2"], a["eps"],
                                    a["out"], a["ws"], a["batch"], a["nk"], a["nv"], a["d"], a["xs"], a["gs"], a["zs"],
                                    a["outs"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(nv=5, pitch=5 * 128 * 128), UNSUP),             # NV not a multiple of NK
    (dict(taps=0), ARG), (dict(taps=9), ARG), (dict(rpitch=4 * 1280 - 1), ARG),
    (dict(l2=-1.0), ARG), (dict(eps=float("nan")), ARG), (dict(ring=None), ARG), (dict(rate=None), ARG),
    (dict(xs=1279), ARG), (dict(gs=5), ARG),
    (dict(ring=A + 8192), ALIAS),                         # conv state inside the h-state
    (dict(out=A + (9 << 30) + 64), ALIAS),                # output inside the conv state
    (dict(ring=A + (9 << 30) + 2), ALIGN),
    (dict(ws=None), ARG), (dict(ws=A + (10 << 30) + 2), ALIGN), (dict(ws=A + (6 << 30)), ALIAS),
])
def test_conv_norm_rejects(lib, kw, want):
    assert conv_norm(lib, **kw) == want


def test_conv_norm_empty_is_ok(lib):
    assert conv_norm(lib, batch=0) == OK


def conv_norm_noalloc(lib, **kw):
    nk, nv, d, taps = 2, 6, 128, 4
    C = (2 * nk + nv) * d
    a = dict(state=A, dt=0, pitch=nv * d * d, ring=A + (9 << 30), rpitch=taps * C, taps=taps, x=A + (1 << 30),
             w=A + (2 << 30), br=A + (3 << 30), ar=A + (4 << 30), dtb=A + (5 << 30), rate=A + (5 << 30) + 4096,
             z=A + (7 << 30), gn=A + (8 << 30), l2=1e-6, eps=1e-6, out=A + (6 << 30),
             batch=2, nk=nk, nv=nv, d=d, xs=C, gs=nv, zs=nv * d, outs=nv * d)
    a.update(kw)
    return lib.gdn_decode_conv_norm_noalloc(a["state"], a["dt"], a["pitch"], a["ring"], a["rpitch"], a["taps"],
                                            a["x"], a["w"], a["br"], a["ar"], a["dtb"], a["rate"], a["z"], a["gn"],
                                            a["l2"], a["eps"], a["out"], a["batch"], a["nk"], a["nv"], a["d"],
                                            a["xs"], a["gs"], a["zs"], a["outs"], None)


def test_conv_norm_noalloc_rejects_beyond_static_counters(lib):
    """batch * NK above the static counter array is refused first, before any CUDA call."""
    assert conv_norm_noalloc(lib, batch=gdn.GDN_NOALLOC_MAX_KEY_HEADS // 2 + 1) == UNSUP


def test_conv_norm_noalloc_without_device_reports_cuda_error(lib):
    """On a host without a GPU a valid call passes every check, then the per-device set-up fails and
    says so (GDN_ERR_CUDA)."""
    assert conv_norm_noalloc(lib) == CUDA
    assert lib.gdn_last_cuda_error() != 0


@pytest.mark.parametrize("kw,want", [
    (dict(batch=0), OK),                                 # empty call: no CUDA call at all
    (dict(state=None), ARG), (dict(ring=None), ARG), (dict(out=None), ARG), (dict(gn=None), ARG),
    (dict(nk=0), ARG), (dict(d=0), ARG), (dict(taps=0), ARG), (dict(taps=9), ARG), (dict(eps=-1.0), ARG),
    (dict(nv=5), UNSUP),                                 # NV not a multiple of NK
    (dict(dt=2), UNSUP),
    (dict(out=A + 4096), ALIAS),                         # output inside the state
])
def test_conv_norm_noalloc_checks_arguments_before_any_cuda_call(lib, kw, want):
    """The argument checks of gdn_decode_conv_norm come before the address lookup: without a GPU
    these calls still get their own status, not GDN_ERR_CUDA."""
    assert conv_norm_noalloc(lib, **kw) == want


def prefill(lib, **kw):
    a = dict(state=A, dt=0, pitch=3 * 128 * 128, q=A + (1 << 30), k=A + (2 << 30), v=A + (3 << 30),
             alpha=A + (4 << 30), beta=A + (5 << 30), o=A + (6 << 30), batch=2, T=5, nk=1, nv=3, d=128,
             qk=128, vs=3 * 128, gb=3, os=3 * 128)
    chunked = kw.pop("chunked", False)
    a.update(kw)
    fn = lib.gdn_prefill_chunked if chunked else lib.gdn_prefill_seq
    return fn(a["state"], a["dt"], a["pitch"], a["q"], a["k"], a["v"], a["alpha"], a["beta"],
              a["o"], a["batch"], a["T"], a["nk"], a["nv"], a["d"], a["qk"], a["vs"], a["gb"], a["os"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(state=None), ARG), (dict(q=None), ARG), (dict(o=None), ARG), (dict(beta=None), ARG),
    (dict(batch=-1), ARG), (dict(nk=0), ARG), (dict(nv=0), ARG), (dict(d=0), ARG),
    (dict(d=257, pitch=48 * 257 * 257, qk=16 * 257, vs=48 * 257, os=48 * 257), UNSUP),
    (dict(dt=2), UNSUP),
    (dict(pitch=48 * 128 * 128 - 1), ARG),               # slot pitch shorter than NV*D*D
    (dict(qk=16 * 128 - 1), ARG), (dict(vs=48 * 128 - 4), ARG), (dict(gb=47), ARG), (dict(os=100), ARG),
    (dict(q=A + (1 << 30) + 2), ALIGN),                  # fp32 pointer not 4-byte aligned
    (dict(state=A + 1, dt=1), ALIGN),                    # fp16 state not 2-byte aligned
    (dict(o=A + 4096), ALIAS),                           # output inside the state
    (dict(o=A + (1 << 30) + 64), ALIAS),                 # output overlapping q
    (dict(q=A + 8), ALIAS),                              # input inside the state (state is written)
])
def test_decode_rejects(lib, kw, want):
    assert decode(lib, **kw) == want


def test_decode_empty_batch_is_ok(lib):
    assert decode(lib, batch=0) == OK
    assert decode(lib, batch=0, q=None) == ARG


@pytest.mark.parametrize("kw,want", [
    (dict(eps=-1.0), ARG), (dict(eps=float("inf")), ARG), (dict(eps=float("nan")), ARG),
    (dict(z=None), ARG), (dict(gn=None), ARG), (dict(out=None), ARG),
    (dict(out=A + (6 << 30) + 1), ALIGN),                # bf16 output not 2-byte aligned
    (dict(zs=15), ARG), (dict(outs=15), ARG),
    (dict(out=A + (8 << 30) + 8), ALIAS),                # output on top of gn
])
def test_decode_norm_rejects(lib, kw, want):
    assert decode_norm(lib, **kw) == want


def decode_norm_q8(lib, **kw):
    a = dict(state=A, dt=0, pitch=2 * 64 * 64, q=A + (1 << 30), k=A + (2 << 30), v=A + (3 << 30),
             alpha=A + (4 << 30), beta=A + (5 << 30), z=A + (7 << 30), gn=A + (8 << 30), eps=1e-6,
             xq=A + (6 << 30), xs=A + (9 << 30), y=A + (10 << 30), batch=2, nk=1, nv=2, d=64, qk=64, vs=128,
             gb=2, zs=128, xqs=128, xss=4, ys=128)
    a.update(kw)
    return lib.gdn_decode_norm_q8(a["state"], a["dt"], a["pitch"], a["q"], a["k"], a["v"], a["alpha"],
                                  a["beta"], a["z"], a["gn"], a["eps"], a["xq"], a["xs"], a["y"], a["batch"],
                                  a["nk"], a["nv"], a["d"], a["qk"], a["vs"], a["gb"], a["zs"], a["xqs"],
                                  a["xss"], a["ys"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(d=48, pitch=2 * 48 * 48, qk=48, vs=96, zs=96, xqs=96, xss=3, ys=96), UNSUP),   # D % 32 != 0
    (dict(xq=None), ARG), (dict(xs=None), ARG), (dict(xss=3), ARG), (dict(xqs=127), ARG),
    (dict(eps=-1.0), ARG), (dict(xs=A + (9 << 30) + 2), ALIGN),
    (dict(xq=A + (9 << 30) + 8), ALIAS),                # codes over the scales
    (dict(y=A + 64), ALIAS),                            # normed values inside the state
    (dict(xs=A + (3 << 30)), ALIAS),                    # scales over v
])
def test_decode_norm_q8_rejects(lib, kw, want):
    assert decode_norm_q8(lib, **kw) == want


def test_decode_norm_q8_empty_and_optional_y(lib):
    assert decode_norm_q8(lib, batch=0) == OK
    assert decode_norm_q8(lib, batch=0, y=None) == OK
    assert decode_norm_q8(lib, batch=0, xq=None) == ARG


def gate_norm(lib, q8=False, **kw):
    a = dict(o=A, z=A + (1 << 30), gn=A + (2 << 30), eps=1e-6, out=A + (3 << 30), xq=A + (3 << 30),
             xs=A + (4 << 30), y=A + (5 << 30), rows=7, nv=3, d=64, os=192, zs=192, outs=192, xqs=192, xss=6,
             ys=192)
    a.update(kw)
    if q8:
        return lib.gdn_gate_norm_q8(a["o"], a["z"], a["gn"], a["eps"], a["xq"], a["xs"], a["y"], a["rows"], a["nv"],
                                    a["d"], a["os"], a["zs"], a["xqs"], a["xss"], a["ys"], None)
    return lib.gdn_gate_norm(a["o"], a["z"], a["gn"], a["eps"], a["out"], a["rows"], a["nv"], a["d"], a["os"],
                             a["zs"], a["outs"], None)


@pytest.mark.parametrize("q8,kw,want", [
    (False, dict(d=257, os=771, zs=771, outs=771), UNSUP), (False, dict(nv=0), ARG), (False, dict(rows=-1), ARG),
    (False, dict(o=None), ARG), (False, dict(eps=float("inf")), ARG), (False, dict(os=100), ARG),
    (False, dict(out=A + 2), ALIAS), (False, dict(out=A + (3 << 30) + 1), ALIGN),
    (True, dict(d=48, os=144, zs=144, xqs=144, xss=4, ys=144), UNSUP), (True, dict(xs=None), ARG),
    (True, dict(xq=A + (4 << 30) + 4), ALIAS), (True, dict(y=A + (1 << 30) + 64), ALIAS),
])
def test_gate_norm_rejects(lib, q8, kw, want):
    assert gate_norm(lib, q8=q8, **kw) == want


def test_gate_norm_empty_is_ok(lib):
    assert gate_norm(lib, rows=0) == OK
    assert gate_norm(lib, q8=True, rows=0, y=None) == OK


@pytest.mark.parametrize("kw,want", [
    (dict(dt=2), UNSUP), (dict(T=-1), ARG), (dict(o=None), ARG), (dict(state=A + 1, dt=1), ALIGN),
    (dict(os=10), ARG), (dict(o=A + 100), ALIAS),
])
@pytest.mark.parametrize("chunked", [False, True])
def test_prefill_rejects(lib, kw, want, chunked):
    """gdn_prefill_chunked shares gdn_prefill_seq's checks."""
    assert prefill(lib, chunked=chunked, **kw) == want


@pytest.mark.parametrize("chunked", [False, True])
def test_prefill_empty_is_ok(lib, chunked):
    assert prefill(lib, T=0, chunked=chunked) == OK
    assert prefill(lib, batch=0, chunked=chunked) == OK


def test_device_wait_timeouts_without_device(lib):
    import ctypes
    assert lib.gdn_device_wait_timeouts(None) == ARG
    c = ctypes.c_uint(7)
    assert lib.gdn_device_wait_timeouts(ctypes.byref(c)) == CUDA


def test_converters_reject(lib):
    f = lib.gdn_h_f32_to_f16
    g = lib.gdn_h_f16_to_f32
    assert f(None, A, 10, None) == ARG and g(A, None, 10, None) == ARG
    assert f(A, A + (1 << 30), 0, None) == OK and g(A, A + (1 << 30), 0, None) == OK
    assert f(A + 1, A + (1 << 30), 10, None) == ALIGN
    assert g(A + 1, A + (1 << 30), 10, None) == ALIGN
    assert f(A, A + 8, 10, None) == ALIAS            # in-place narrowing would race
    assert g(A + 16, A, 10, None) == ALIAS


def test_converter_adjacent_ranges_are_not_alias(lib):
    # [A, A+40) and [A+40, A+60): touching, not overlapping -> passes the alias check.  With no GPU
    # the launch itself fails, which must come back as GDN_ERR_CUDA, not a crash.
    st = lib.gdn_h_f32_to_f16(A, A + 40, 10, None)
    assert st == CUDA
    assert lib.gdn_last_cuda_error() != 0
