"""gated_deltanet_linear_16_gb300 -- GB300 (sm_103a) gated delta rule library.

A thin Python binding over the C-ABI library ``libgdn.so`` (declared in
``include/gdn.h``).  Every function here has the name of its C entry point and
only marshals arguments: torch tensors (or raw integer device addresses) become
pointers, sizes and strides are passed through, the current torch CUDA stream
is the default stream.  Every step of the computation runs in libgdn's CUDA
kernels; there is no CPU path.  A nonzero status raises :class:`GdnError`.

The step (logicaffeine_compile/codegen_cuda/gdn.rs, kernel ``gdn_step``), per
sequence, value head h (key head g = h mod NK) and state row a:
``S[a] <- alpha S[a] + beta (v[a] - alpha S[a].k) k`` and
``o[a] = S_new[a].q / sqrt(D)``; the fused norm (same page, ``gdn_gate_norm``)
gives ``out = gn o / sqrt(mean(o^2) + eps) * silu(z)`` in bf16.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "GdnError", "load", "build", "library_path",
    "GDN_STATE_F32", "GDN_STATE_F16", "STATUS",
    "gdn_decode", "gdn_decode_norm", "gdn_decode_chunk2", "gdn_decode_conv_norm", "gdn_prefill_seq",
    "gdn_prefill_chunked", "gdn_device_wait_timeouts", "gdn_set_wait_polls", "gdn_set_mma_wait_polls",
    "GDN_DEFAULT_WAIT_POLLS",
    "gdn_decode_conv_norm_noalloc", "GDN_NOALLOC_MAX_KEY_HEADS", "gdn_decode_norm_q8",
    "gdn_gate_norm", "gdn_gate_norm_q8",
    "gdn_h_f32_to_f16", "gdn_h_f16_to_f32", "gdn_status_str", "gdn_last_cuda_error",
]

GDN_STATE_F32 = 0
GDN_STATE_F16 = 1
GDN_NOALLOC_MAX_KEY_HEADS = 16384     # batch * NK limit of gdn_decode_conv_norm_noalloc
GDN_DEFAULT_WAIT_POLLS = 4194304      # default bound of the tensor-core kernels' MMA-completion waits
STATUS = {0: "GDN_OK", 1: "GDN_ERR_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_ALIGN",
          4: "GDN_ERR_ALIAS", 5: "GDN_ERR_CUDA"}

_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    """A libgdn call returned a nonzero status."""

    def __init__(self, fn, status, detail=""):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} {detail}".strip())


def library_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgdn.so")


def build(force: bool = False) -> str:
    """Compile libgdn.so in-tree with nvcc (sm_103a)."""
    from . import builder
    return builder.build(force=force)


def _declare(lib):
    P, i32, i64, u64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
    lib.gdn_decode.argtypes = [P, i32, i64, P, P, P, P, P, P, i32, i32, i32, i32, i64, i64, i64, i64, P]
    lib.gdn_decode_norm.argtypes = [P, i32, i64, P, P, P, P, P, P, P, f32, P, i32, i32, i32, i32,
                                    i64, i64, i64, i64, i64, P]
    lib.gdn_decode_norm_q8.argtypes = [P, i32, i64, P, P, P, P, P, P, P, f32, P, P, P, i32, i32, i32, i32,
                                       i64, i64, i64, i64, i64, i64, i64, P]
    lib.gdn_gate_norm.argtypes = [P, P, P, f32, P, i64, i32, i32, i64, i64, i64, P]
    lib.gdn_gate_norm_q8.argtypes = [P, P, P, f32, P, P, P, i64, i32, i32, i64, i64, i64, i64, i64, P]
    lib.gdn_decode_conv_norm.argtypes = [P, i32, i64, P, i64, i32, P, P, P, P, P, P, P, P, f32, f32, P, P,
                                         i32, i32, i32, i32, i64, i64, i64, i64, P]
    lib.gdn_decode_conv_norm_noalloc.argtypes = [P, i32, i64, P, i64, i32, P, P, P, P, P, P, P, P, f32, f32, P,
                                                 i32, i32, i32, i32, i64, i64, i64, i64, P]
    lib.gdn_decode_chunk2.argtypes = [P, i32, i64, P, i64, P, P, P, P, P, P, i32, i32, i32, i32,
                                      i64, i64, i64, i64, P]
    lib.gdn_prefill_seq.argtypes = [P, i32, i64, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                    i64, i64, i64, i64, P]
    lib.gdn_prefill_chunked.argtypes = lib.gdn_prefill_seq.argtypes
    lib.gdn_device_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.gdn_set_wait_polls.argtypes = [ctypes.c_uint]
    lib.gdn_set_wait_polls.restype = None
    lib.gdn_set_mma_wait_polls.argtypes = [ctypes.c_uint]
    lib.gdn_set_mma_wait_polls.restype = None
    lib.gdn_h_f32_to_f16.argtypes = [P, P, u64, P]
    lib.gdn_h_f16_to_f32.argtypes = [P, P, u64, P]
    for fn in ("gdn_decode", "gdn_decode_norm", "gdn_decode_chunk2", "gdn_decode_conv_norm", "gdn_prefill_seq",
               "gdn_prefill_chunked", "gdn_device_wait_timeouts",
               "gdn_decode_conv_norm_noalloc", "gdn_decode_norm_q8", "gdn_gate_norm", "gdn_gate_norm_q8",
               "gdn_h_f32_to_f16",
               "gdn_h_f16_to_f32"):
        getattr(lib, fn).restype = i32
    lib.gdn_status_str.argtypes = [i32]
    lib.gdn_status_str.restype = ctypes.c_char_p
    lib.gdn_last_cuda_error.argtypes = []
    lib.gdn_last_cuda_error.restype = i32
    return lib


def load(path: str | None = None):
    """Load libgdn.so (building it first if it is missing); raises if that fails."""
    global _lib
    with _lock:
        if _lib is None:
            path = path or library_path()
            if not os.path.exists(path):
                build()
            _lib = _declare(ctypes.CDLL(path))
    return _lib


# ------------------------------------------------------------------ marshalling

def _ptr(x):
    """Device address of a tensor (its first element) or an int address; None -> NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, st):
    if st != 0:
        detail = ""
        if st == 5:
            detail = f"(cudaError {load().gdn_last_cuda_error()})"
        raise GdnError(fn, st, detail)


def _state_dtype(state, state_dtype):
    if state_dtype is not None:
        return state_dtype
    import torch
    if isinstance(state, int):
        raise ValueError("state_dtype is required when state is a raw address")
    if state.dtype == torch.float32:
        return GDN_STATE_F32
    if state.dtype == torch.float16:
        return GDN_STATE_F16
    raise ValueError(f"unsupported state dtype {state.dtype}")


def gdn_decode(state, q, k, v, alpha, beta, o, *, batch, nk, nv, d,
               state_pitch=None, state_dtype=None,
               qk_stride=None, v_stride=None, gb_stride=None, o_stride=None, stream=None):
    """One token through the recurrence; raw fp32 o.  See include/gdn.h."""
    lib = load()
    sd = _state_dtype(state, state_dtype)
    st = lib.gdn_decode(
        _ptr(state), sd, state_pitch if state_pitch is not None else nv * d * d,
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(o),
        batch, nk, nv, d,
        qk_stride if qk_stride is not None else nk * d,
        v_stride if v_stride is not None else nv * d,
        gb_stride if gb_stride is not None else nv,
        o_stride if o_stride is not None else nv * d,
        _stream(stream))
    _check("gdn_decode", st)


def gdn_decode_norm(state, q, k, v, alpha, beta, z, gn, out, *, batch, nk, nv, d, eps=1e-6,
                    state_pitch=None, state_dtype=None,
                    qk_stride=None, v_stride=None, gb_stride=None, z_stride=None, out_stride=None,
                    stream=None):
    """One token through the recurrence with the fused gated RMS norm; bf16 out."""
    lib = load()
    sd = _state_dtype(state, state_dtype)
    st = lib.gdn_decode_norm(
        _ptr(state), sd, state_pitch if state_pitch is not None else nv * d * d,
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(z), _ptr(gn), float(eps), _ptr(out),
        batch, nk, nv, d,
        qk_stride if qk_stride is not None else nk * d,
        v_stride if v_stride is not None else nv * d,
        gb_stride if gb_stride is not None else nv,
        z_stride if z_stride is not None else nv * d,
        out_stride if out_stride is not None else nv * d,
        _stream(stream))
    _check("gdn_decode_norm", st)


def gdn_decode_norm_q8(state, q, k, v, alpha, beta, z, gn, xq, xs, y=None, *, batch, nk, nv, d, eps=1e-6,
                       state_pitch=None, state_dtype=None, qk_stride=None, v_stride=None, gb_stride=None,
                       z_stride=None, xq_stride=None, xs_stride=None, y_stride=None, stream=None):
    """gdn_decode_norm with int8 output groups of 32 (codes xq, fp32 scales xs; y, if given,
    receives the fp32 normed values).  D must be a multiple of 32."""
    lib = load()
    sd = _state_dtype(state, state_dtype)
    st = lib.gdn_decode_norm_q8(
        _ptr(state), sd, state_pitch if state_pitch is not None else nv * d * d,
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(z), _ptr(gn), float(eps),
        _ptr(xq), _ptr(xs), _ptr(y) if y is not None else None,
        batch, nk, nv, d,
        qk_stride if qk_stride is not None else nk * d,
        v_stride if v_stride is not None else nv * d,
        gb_stride if gb_stride is not None else nv,
        z_stride if z_stride is not None else nv * d,
        xq_stride if xq_stride is not None else nv * d,
        xs_stride if xs_stride is not None else nv * d // 32,
        y_stride if y_stride is not None else nv * d,
        _stream(stream))
    _check("gdn_decode_norm_q8", st)


def gdn_gate_norm(o, z, gn, out, *, rows, nv, d, eps=1e-6, o_stride=None, z_stride=None, out_stride=None,
                  stream=None):
    """The gated RMS norm over `rows` rows of NV heads x D raw outputs (e.g. a prefill's o); bf16 out."""
    lib = load()
    hv = nv * d
    st = lib.gdn_gate_norm(_ptr(o), _ptr(z), _ptr(gn), float(eps), _ptr(out), rows, nv, d,
                           o_stride if o_stride is not None else hv, z_stride if z_stride is not None else hv,
                           out_stride if out_stride is not None else hv, _stream(stream))
    _check("gdn_gate_norm", st)


def gdn_gate_norm_q8(o, z, gn, xq, xs, y=None, *, rows, nv, d, eps=1e-6, o_stride=None, z_stride=None,
                     xq_stride=None, xs_stride=None, y_stride=None, stream=None):
    """gdn_gate_norm with int8 output groups of 32 (codes xq, fp32 scales xs, optional fp32 y)."""
    lib = load()
    hv = nv * d
    st = lib.gdn_gate_norm_q8(_ptr(o), _ptr(z), _ptr(gn), float(eps), _ptr(xq), _ptr(xs), _ptr(y), rows, nv, d,
                              o_stride if o_stride is not None else hv, z_stride if z_stride is not None else hv,
                              xq_stride if xq_stride is not None else hv,
                              xs_stride if xs_stride is not None else hv // 32,
                              y_stride if y_stride is not None else hv, _stream(stream))
    _check("gdn_gate_norm_q8", st)


def gdn_decode_conv_norm(state, conv_state, x, conv_w, br, ar, dt, rate, z, gn, out, workspace, *, batch, nk,
                         nv, d, taps, eps=1e-6, l2_eps=1e-6, state_pitch=None, conv_pitch=None,
                         state_dtype=None, x_stride=None, gate_stride=None, z_stride=None, out_stride=None,
                         stream=None):
    """One token from the projections (conv ring + silu, q/k L2 norm, gates from logits, the step,
    the gated norm) in one launch; bf16 out.  workspace: batch*nk int32, zero before the first call
    and left zero.  See include/gdn.h for the layouts."""
    lib = load()
    sd = _state_dtype(state, state_dtype)
    C = (2 * nk + nv) * d
    st = lib.gdn_decode_conv_norm(
        _ptr(state), sd, state_pitch if state_pitch is not None else nv * d * d,
        _ptr(conv_state), conv_pitch if conv_pitch is not None else taps * C, taps,
        _ptr(x), _ptr(conv_w), _ptr(br), _ptr(ar), _ptr(dt), _ptr(rate), _ptr(z), _ptr(gn),
        float(l2_eps), float(eps), _ptr(out), _ptr(workspace), batch, nk, nv, d,
        x_stride if x_stride is not None else C,
        gate_stride if gate_stride is not None else nv,
        z_stride if z_stride is not None else nv * d,
        out_stride if out_stride is not None else nv * d,
        _stream(stream))
    _check("gdn_decode_conv_norm", st)


def gdn_decode_conv_norm_noalloc(state, conv_state, x, conv_w, br, ar, dt, rate, z, gn, out, *, batch, nk,
                                 nv, d, taps, eps=1e-6, l2_eps=1e-6, state_pitch=None, conv_pitch=None,
                                 state_dtype=None, x_stride=None, gate_stride=None, z_stride=None,
                                 out_stride=None, stream=None):
    """gdn_decode_conv_norm without a workspace: the counters live in the library's static device
    memory (batch*nk <= GDN_NOALLOC_MAX_KEY_HEADS; calls that may overlap on one device race).
    See include/gdn.h."""
    lib = load()
    sd = _state_dtype(state, state_dtype)
    C = (2 * nk + nv) * d
    st = lib.gdn_decode_conv_norm_noalloc(
        _ptr(state), sd, state_pitch if state_pitch is not None else nv * d * d,
        _ptr(conv_state), conv_pitch if conv_pitch is not None else taps * C, taps,
        _ptr(x), _ptr(conv_w), _ptr(br), _ptr(ar), _ptr(dt), _ptr(rate), _ptr(z), _ptr(gn),
        float(l2_eps), float(eps), _ptr(out), batch, nk, nv, d,
        x_stride if x_stride is not None else C,
        gate_stride if gate_stride is not None else nv,
        z_stride if z_stride is not None else nv * d,
        out_stride if out_stride is not None else nv * d,
        _stream(stream))
    _check("gdn_decode_conv_norm_noalloc", st)


def gdn_decode_chunk2(state, state_mid, q, k, v, alpha, beta, o, *, batch, nk, nv, d,
                      state_pitch=None, mid_pitch=None, state_dtype=None,
                      qk_stride=None, v_stride=None, gb_stride=None, o_stride=None, stream=None):
    """Two tokens per sequence in one launch (token rows 2*b + t); state_mid receives the state
    after the first token, state the state after both; raw fp32 o for both tokens."""
    lib = load()
    sd = _state_dtype(state, state_dtype)
    st = lib.gdn_decode_chunk2(
        _ptr(state), sd, state_pitch if state_pitch is not None else nv * d * d,
        _ptr(state_mid), mid_pitch if mid_pitch is not None else nv * d * d,
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(o),
        batch, nk, nv, d,
        qk_stride if qk_stride is not None else nk * d,
        v_stride if v_stride is not None else nv * d,
        gb_stride if gb_stride is not None else nv,
        o_stride if o_stride is not None else nv * d,
        _stream(stream))
    _check("gdn_decode_chunk2", st)


def _prefill(fn, state, q, k, v, alpha, beta, o, *, batch, seq_len, nk, nv, d,
             state_pitch=None, state_dtype=None,
             qk_stride=None, v_stride=None, gb_stride=None, o_stride=None, stream=None):
    lib = load()
    sd = _state_dtype(state, state_dtype)
    st = getattr(lib, fn)(
        _ptr(state), sd, state_pitch if state_pitch is not None else nv * d * d,
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(o),
        batch, seq_len, nk, nv, d,
        qk_stride if qk_stride is not None else nk * d,
        v_stride if v_stride is not None else nv * d,
        gb_stride if gb_stride is not None else nv,
        o_stride if o_stride is not None else nv * d,
        _stream(stream))
    _check(fn, st)


def gdn_prefill_seq(state, q, k, v, alpha, beta, o, **kw):
    """seq_len tokens per sequence in one launch (token rows b*seq_len + t), token by token; raw fp32 o."""
    _prefill("gdn_prefill_seq", state, q, k, v, alpha, beta, o, **kw)


def gdn_prefill_chunked(state, q, k, v, alpha, beta, o, **kw):
    """gdn_prefill_seq regrouped into chunks of 64 tokens on the tensor cores (D = 128); same arguments."""
    _prefill("gdn_prefill_chunked", state, q, k, v, alpha, beta, o, **kw)


def gdn_set_wait_polls(polls: int) -> None:
    """Polls of an MMA or tensor-copy completion before a tensor-core kernel gives up (0: at once, to
    test that path)."""
    load().gdn_set_wait_polls(polls)


def gdn_set_mma_wait_polls(polls: int) -> None:
    """As gdn_set_wait_polls for the MMA waits only (the tensor-copy waits keep their bound)."""
    load().gdn_set_mma_wait_polls(polls)


def gdn_device_wait_timeouts() -> int:
    """Bounded MMA-completion waits that ran out on the current device (0 when healthy); synchronises."""
    c = ctypes.c_uint(0)
    _check("gdn_device_wait_timeouts", load().gdn_device_wait_timeouts(ctypes.byref(c)))
    return c.value


def gdn_h_f32_to_f16(src, dst, n=None, stream=None):
    """n h-state elements fp32 -> fp16 (round to nearest even)."""
    lib = load()
    n = src.numel() if n is None else n
    _check("gdn_h_f32_to_f16", lib.gdn_h_f32_to_f16(_ptr(src), _ptr(dst), n, _stream(stream)))


def gdn_h_f16_to_f32(src, dst, n=None, stream=None):
    """n h-state elements fp16 -> fp32 (exact)."""
    lib = load()
    n = src.numel() if n is None else n
    _check("gdn_h_f16_to_f32", lib.gdn_h_f16_to_f32(_ptr(src), _ptr(dst), n, _stream(stream)))


def gdn_status_str(status: int) -> str:
    return load().gdn_status_str(status).decode()


def gdn_last_cuda_error() -> int:
    return load().gdn_last_cuda_error()
