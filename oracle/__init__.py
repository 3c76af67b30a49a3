"""fp64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may import this package.  The product
library never calls it, links it or falls back to it; the two share no code.

The arithmetic lives in ``gdn_oracle.c`` (plain loops, fp64, compiled with
``-O2 -ffp-contract=off`` so x86 and Arm hosts give the same bits).  This
module builds it with gcc on first use and wraps it with ctypes, taking numpy
arrays in the contiguous layouts documented in the C file.  ctypes releases
the GIL during a call, so :func:`parallel_map` runs independent units on
several host threads.

Passages followed (page title, section):
  * logicaffeine_compile/codegen_cuda/gdn.rs, kernel ``gdn_step`` -- the
    recurrence, g = h mod NK, o scaled by 1/sqrt(D);
  * same page, kernel ``gdn_gate_norm`` -- RMS norm then silu(z) gate;
  * metrale_model_layers/layers/ops/ssm_gdn_a.rs, ``gdn_prefill_regresident``
    -- token-sequential prefill; ``ssm_h_state_f32_to_f16`` /
    ``ssm_h_state_f16_to_f32`` -- round-to-nearest-even converters;
  * gdn.rs, kernel ``gdn_gate_norm_q`` -- int8 activation groups of 32.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, invariants, a textbook special case (D = 1 scalar recurrence), the
pages' alternative row form and numpy's own binary16 conversion.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "_gdn_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (idempotent); returns the .so path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def bind(path):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, u64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
    lib.orc_decode.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P]
    lib.orc_decode.restype = None
    lib.orc_prefill.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
    lib.orc_prefill.restype = None
    lib.orc_gated_rmsnorm.argtypes = [i64, i32, P, P, P, f64, P]
    lib.orc_gated_rmsnorm.restype = None
    lib.orc_f32_to_f16_array.argtypes = [P, P, u64]
    lib.orc_f32_to_f16_array.restype = None
    lib.orc_f16_to_f32_array.argtypes = [P, P, u64]
    lib.orc_f16_to_f32_array.restype = None
    lib.orc_conv_silu.argtypes = [i32, i32, P, P, P, P]
    lib.orc_conv_silu.restype = None
    lib.orc_l2norm_heads.argtypes = [i32, i32, P, f64]
    lib.orc_l2norm_heads.restype = None
    lib.orc_gates.argtypes = [i32, P, P, P, P, P, P]
    lib.orc_gates.restype = None
    lib.orc_decode_f64.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P]
    lib.orc_decode_f64.restype = None
    lib.orc_quant_q8_groups.argtypes = [i64, P, P, P]
    lib.orc_quant_q8_groups.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def decode(S, q, k, v, alpha, beta, nk):
    """One decode step, in place on the fp64 state.

    S: [B][NV][D][D] float64 (updated in place); q,k: [B][NK*D]; v: [B][NV*D];
    alpha, beta: [B][NV] (float32, as the kernels receive them).
    Returns o: [B][NV*D] float64 = S_new q / sqrt(D) per head.
    """
    lib = _load()
    assert S.dtype == np.float64 and S.flags.c_contiguous and S.ndim == 4
    B, nv, d, _ = S.shape
    q, k, v = _c(q, np.float32), _c(k, np.float32), _c(v, np.float32)
    alpha, beta = _c(alpha, np.float32), _c(beta, np.float32)
    assert q.size == B * nk * d and k.size == B * nk * d and v.size == B * nv * d
    assert alpha.size == B * nv and beta.size == B * nv
    o = np.empty((B, nv * d), dtype=np.float64)
    lib.orc_decode(B, nk, nv, d, _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(o))
    return o


def gated_rmsnorm(o, z, gn, eps):
    """out = gn * o / sqrt(mean(o^2) + eps) * silu(z), per head of D.

    o: [..., D] float64 (heads on the leading axes); z: same shape (float32);
    gn: [D] float32.  Returns float64 of o's shape.
    """
    lib = _load()
    d = gn.shape[-1]
    o = _c(o, np.float64)
    z = _c(z, np.float32)
    gn = _c(gn, np.float32)
    assert o.size % d == 0 and z.size == o.size
    out = np.empty_like(o)
    lib.orc_gated_rmsnorm(o.size // d, d, _ptr(o), _ptr(z), _ptr(gn), float(eps), _ptr(out))
    return out


def prefill(S, q, k, v, alpha, beta, nk):
    """Token-sequential prefill, in place on the fp64 state.

    S: [B][NV][D][D] float64; q,k: [B][T][NK*D]; v: [B][T][NV*D];
    alpha, beta: [B][T][NV].  Returns o: [B][T][NV*D] float64 (raw, no norm).
    """
    lib = _load()
    assert S.dtype == np.float64 and S.flags.c_contiguous and S.ndim == 4
    B, nv, d, _ = S.shape
    q, k, v = _c(q, np.float32), _c(k, np.float32), _c(v, np.float32)
    alpha, beta = _c(alpha, np.float32), _c(beta, np.float32)
    T = q.shape[1]
    assert q.size == B * T * nk * d and v.size == B * T * nv * d and alpha.size == B * T * nv
    o = np.empty((B, T, nv * d), dtype=np.float64)
    lib.orc_prefill(B, T, nk, nv, d, _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(o))
    return o


def f32_to_f16_bits(x):
    """binary32 -> binary16 bit patterns, round to nearest, ties to even."""
    lib = _load()
    x = np.ascontiguousarray(x)
    if x.dtype not in (np.float32, np.uint32):
        raise TypeError("f32_to_f16_bits takes float32 values or uint32 bit patterns")
    src = x.view(np.uint32)
    dst = np.empty(src.shape, dtype=np.uint16)
    lib.orc_f32_to_f16_array(_ptr(src), _ptr(dst), src.size)
    return dst


def f16_to_f32_bits(h):
    """binary16 -> binary32 bit patterns (exact widening)."""
    lib = _load()
    h = np.ascontiguousarray(h)
    if h.dtype not in (np.float16, np.uint16):
        raise TypeError("f16_to_f32_bits takes float16 values or uint16 bit patterns")
    src = h.view(np.uint16)
    dst = np.empty(src.shape, dtype=np.uint32)
    lib.orc_f16_to_f32_array(_ptr(src), _ptr(dst), src.size)
    return dst


def conv_silu(ring, x, w):
    """One token through the depthwise causal conv with silu, per channel.

    ring: [taps][C] float32, shift register (updated in place, newest entry last);
    x: [C] float32; w: [taps][C] float32.  Returns y: [C] float64."""
    lib = _load()
    assert ring.dtype == np.float32 and ring.flags.c_contiguous and ring.ndim == 2
    taps, C = ring.shape
    x, w = _c(x, np.float32), _c(w, np.float32)
    assert x.size == C and w.size == taps * C
    y = np.empty(C, dtype=np.float64)
    lib.orc_conv_silu(taps, C, _ptr(ring), _ptr(x), _ptr(w), _ptr(y))
    return y


def l2norm_heads(y, d, eps):
    """Per-head y / sqrt(sum y^2 + eps) over consecutive heads of d (fp64, returns a copy)."""
    lib = _load()
    y = np.array(y, dtype=np.float64, order="C")
    assert y.size % d == 0
    lib.orc_l2norm_heads(y.size // d, d, _ptr(y), float(eps))
    return y


def gates(br, ar, dt, rate):
    """beta = sigmoid(br), alpha = (1 + e^(ar + dt))^rate, elementwise (fp64)."""
    lib = _load()
    br, ar, dt, rate = (_c(a, np.float32) for a in (br, ar, dt, rate))
    n = br.size
    assert ar.size == n and dt.size == n and rate.size == n
    beta = np.empty(br.shape, dtype=np.float64)
    alpha = np.empty(br.shape, dtype=np.float64)
    lib.orc_gates(n, _ptr(br), _ptr(ar), _ptr(dt), _ptr(rate), _ptr(beta), _ptr(alpha))
    return beta, alpha


def decode_f64(S, q, k, v, alpha, beta, nk):
    """decode() with fp64 token inputs (same layouts)."""
    lib = _load()
    assert S.dtype == np.float64 and S.flags.c_contiguous and S.ndim == 4
    B, nv, d, _ = S.shape
    q, k, v, alpha, beta = (_c(a, np.float64) for a in (q, k, v, alpha, beta))
    assert q.size == B * nk * d and k.size == B * nk * d and v.size == B * nv * d
    assert alpha.size == B * nv and beta.size == B * nv
    o = np.empty((B, nv * d), dtype=np.float64)
    lib.orc_decode_f64(B, nk, nv, d, _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(o))
    return o


def quant_q8(y):
    """Int8 groups of 32 (gdn.rs `gdn_gate_norm_q`): fp32 values -> (int8 codes, fp32 scales);
    scale = max|y| / 127 over the group (1 if all zero), code = y / scale rounded half to even,
    all decisions in fp32 as the page takes them.  len(y) must be a multiple of 32."""
    yy = _c(np.asarray(y).reshape(-1), np.float32)
    n = yy.size
    if n % 32:
        raise ValueError("quant_q8: length must be a multiple of 32")
    code = np.empty(n, dtype=np.int8)
    scale = np.empty(n // 32, dtype=np.float32)
    _load().orc_quant_q8_groups(n, _ptr(yy), _ptr(code), _ptr(scale))
    return code, scale


def parallel_map(fn, items, threads=None):
    """Run fn over items on host threads (the C calls release the GIL)."""
    threads = threads or os.cpu_count() or 1
    if threads <= 1 or len(items) <= 1:
        return [fn(x) for x in items]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))
