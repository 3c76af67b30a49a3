"""Shared helpers for the GPU parity tests: strided device buffers with guard
bands, the parity metrics, and runners that drive the CUDA path (through the
C-ABI binding) and the fp64 oracle on the same seeded inputs.

Every device buffer is allocated with sentinel-filled guard bands around it
and, for strided rows, sentinel-filled row padding; the runners check that all
of it is bit-unchanged after the calls (nothing is written out of bounds)."""
from __future__ import annotations

import numpy as np
import torch

import gdn_synth as gs
import gated_deltanet_linear_16_gb300 as gdn
import oracle

GUARD = 256                      # elements of sentinel before and after every buffer
SENT32 = np.int32(0x7FBADBAD)    # quiet-NaN bit pattern
SENT16 = np.int16(0x7DAD)        # binary16 / bf16 NaN bit pattern
SENT8 = 0x5A                     # int8 codes: a value the tests never expect in padding

# Parity bars (stated for the method): fp32 results within 1e-4 of the largest
# reference magnitude; fp16 state and bf16 output within 2e-2 relative L2.
TOL_F32 = 1e-4
TOL_REL_L2 = 2e-2


def max_rel_err(got, ref):
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    scale = np.max(np.abs(ref))
    if scale == 0:
        return float(np.max(np.abs(got)))
    return float(np.max(np.abs(got - ref)) / scale)


def rel_l2(got, ref):
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


def bf16_to_f64(bits):
    """bf16 bit patterns (uint16/int16 array) -> float64."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


class Rows:
    """`rows` rows of `length` elements, `stride` apart, inside a guarded device buffer.

    dtype is a torch dtype (float32, float16, int16 for bf16 bits, or int8).  Padding
    between rows and the guard bands hold the sentinel.  `misalign` shifts the
    payload by that many elements (to force the general kernels)."""

    def __init__(self, rows, length, stride=None, dtype=torch.float32, misalign=0):
        self.rows, self.length = rows, length
        self.stride = length if stride is None else stride
        self.dtype = dtype
        self.nelem = (rows - 1) * self.stride + length if rows > 0 else 0
        self.off = GUARD + misalign
        total = self.off + self.nelem + GUARD
        if dtype == torch.float32:
            ibits, sent = torch.int32, int(SENT32)
        elif dtype == torch.int8:
            ibits, sent = torch.int8, SENT8
        else:
            ibits, sent = torch.int16, int(SENT16)
        self.raw = torch.full((total,), sent, dtype=ibits, device="cuda")
        self.buf = self.raw.view(dtype) if dtype not in (torch.int16, torch.int8) else self.raw
        self.sentinel = sent
        self.ibits = ibits

    @property
    def ptr(self):
        return self.buf[self.off:].data_ptr()

    def _index(self):
        r = torch.arange(self.rows, device="cuda")[:, None] * self.stride
        c = torch.arange(self.length, device="cuda")[None, :]
        return (self.off + r + c).reshape(-1)

    def write(self, arr):
        a = np.ascontiguousarray(arr).reshape(self.rows, self.length)
        t = torch.from_numpy(a).to("cuda")
        if self.dtype == torch.int16 and t.dtype != torch.int16:
            t = t.view(torch.int16)
        self.buf[self._index()] = t.reshape(-1).to(self.buf.dtype) if t.dtype != self.buf.dtype else t.reshape(-1)

    def read(self):
        return self.buf[self._index()].reshape(self.rows, self.length).cpu().numpy()

    def intact(self):
        """Guard bands and row padding still hold the sentinel."""
        mask = torch.ones(self.raw.numel(), dtype=torch.bool, device="cuda")
        mask[self._index()] = False
        return bool(torch.all(self.raw[mask] == self.sentinel).item())


def state_pool(B, NV, D, f16, pad=0, misalign=0):
    """Slots of NV*D*D state elements with `pad` sentinel elements of slot padding."""
    return Rows(B, NV * D * D, NV * D * D + pad, torch.float16 if f16 else torch.float32, misalign)


def to_f64_state(pool, B, NV, D, f16):
    x = pool.read()
    x = x.astype(np.float64)
    return x.reshape(B, NV, D, D)


def run_decode_case(B, NK, NV, D, T, *, f16=False, norm=True, seed=0, init="normal", eps=1e-6,
                    pad=(0, 0, 0, 0, 0), pitch_pad=0, misalign=0, alpha=None, beta=None):
    """T decode steps on the GPU and in the oracle; returns a dict of error metrics.

    pad = extra elements per row for (qk, v, gb, z, out/o)."""
    sdt = np.float16 if f16 else np.float32
    if init == "zero":
        S0 = np.zeros((B, NV, D, D), sdt)
    else:
        S0 = gs.state_heads(seed, range(B), range(NV), D, dtype=sdt)
    gn = gs.norm_weight(seed, D)
    pool = state_pool(B, NV, D, f16, pitch_pad, misalign)
    pool.write(S0.reshape(B, -1))
    ref = S0.astype(np.float64)
    mis = misalign
    qb = Rows(B, NK * D, NK * D + pad[0], misalign=mis)
    kb = Rows(B, NK * D, NK * D + pad[0], misalign=mis)
    vb = Rows(B, NV * D, NV * D + pad[1])
    ab = Rows(B, NV, NV + pad[2])
    bb = Rows(B, NV, NV + pad[2])
    zb = Rows(B, NV * D, NV * D + pad[3])
    gnb = Rows(1, D)
    gnb.write(gn)
    if norm:
        ob = Rows(B, NV * D, NV * D + pad[4], torch.int16)
    else:
        ob = Rows(B, NV * D, NV * D + pad[4])
    worst_out = 0.0          # bf16 out: relative L2; raw o: max error over max |ref|
    worst_out_l2 = 0.0       # raw o: relative L2 (the bar when the state is fp16)
    for t in range(T):
        x = gs.decode_inputs(seed, B, NK, NV, D, step=t)
        if alpha is not None:
            x["alpha"][:] = alpha
        if beta is not None:
            x["beta"][:] = beta
        qb.write(x["q"]); kb.write(x["k"]); vb.write(x["v"])
        ab.write(x["alpha"]); bb.write(x["beta"]); zb.write(x["z"])
        common = dict(batch=B, nk=NK, nv=NV, d=D, state_pitch=pool.stride,
                      state_dtype=gdn.GDN_STATE_F16 if f16 else gdn.GDN_STATE_F32,
                      qk_stride=qb.stride, v_stride=vb.stride, gb_stride=ab.stride)
        if norm:
            gdn.gdn_decode_norm(pool.ptr, qb.ptr, kb.ptr, vb.ptr, ab.ptr, bb.ptr, zb.ptr, gnb.ptr, ob.ptr,
                                eps=eps, z_stride=zb.stride, out_stride=ob.stride, **common)
        else:
            gdn.gdn_decode(pool.ptr, qb.ptr, kb.ptr, vb.ptr, ab.ptr, bb.ptr, ob.ptr, o_stride=ob.stride, **common)
        o_ref = oracle.decode(ref, x["q"], x["k"], x["v"], x["alpha"], x["beta"], NK)
        torch.cuda.synchronize()
        if norm:
            out_ref = oracle.gated_rmsnorm(o_ref.reshape(B * NV, D), x["z"].reshape(B * NV, D), gn, eps)
            got = bf16_to_f64(ob.read()).reshape(B * NV, D)
            worst_out = max(worst_out, rel_l2(got, out_ref))
        else:
            got = ob.read().astype(np.float64)
            worst_out = max(worst_out, max_rel_err(got, o_ref))
            worst_out_l2 = max(worst_out_l2, rel_l2(got, o_ref))
    S_gpu = to_f64_state(pool, B, NV, D, f16)
    res = {
        "state_max_rel": max_rel_err(S_gpu, ref),
        "state_rel_l2": rel_l2(S_gpu, ref),
        "out_worst": worst_out,
        "out_worst_rel_l2": worst_out_l2,
        "intact": all(b.intact() for b in (pool, qb, kb, vb, ab, bb, zb, gnb, ob)),
        "S_gpu": S_gpu, "S_ref": ref,
    }
    return res


def check_decode(res, f16, norm):
    assert res["intact"], "guard band or padding overwritten"
    if f16:
        assert res["state_rel_l2"] <= TOL_REL_L2, res["state_rel_l2"]
    else:
        assert res["state_max_rel"] <= TOL_F32, res["state_max_rel"]
    if norm:
        assert res["out_worst"] <= TOL_REL_L2, res["out_worst"]
    elif f16:
        # o read out of a state that is rounded to fp16 every step carries that state's
        # error, so it is held to the fp16-state bar
        assert res["out_worst_rel_l2"] <= TOL_REL_L2, res["out_worst_rel_l2"]
    else:
        assert res["out_worst"] <= TOL_F32, res["out_worst"]


def run_prefill_case(B, NK, NV, D, T, *, seed=0, init="zero", pad=(0, 0, 0, 0), pitch_pad=0, misalign=0,
                     splits=None, alpha=None, beta=None, f16=False, chunked=False):
    """Prefill of T tokens on the GPU (one call, or per-sequence calls over `splits`)
    and in the oracle; returns error metrics.  chunked: through gdn_prefill_chunked."""
    prefill = gdn.gdn_prefill_chunked if chunked else gdn.gdn_prefill_seq
    sdt = np.float16 if f16 else np.float32
    if init == "zero":
        S0 = np.zeros((B, NV, D, D), sdt)
    else:
        S0 = gs.state_heads(seed, range(B), range(NV), D, dtype=sdt)
    x = gs.prefill_inputs(seed, B, T, NK, NV, D)
    if alpha is not None:          # host-side override of the drawn gates (array or scalar)
        x["alpha"][...] = alpha
    if beta is not None:
        x["beta"][...] = beta
    pool = state_pool(B, NV, D, f16, pitch_pad, misalign)
    pool.write(S0.reshape(B, -1))
    R = B * T
    qb = Rows(R, NK * D, NK * D + pad[0], misalign=misalign)
    kb = Rows(R, NK * D, NK * D + pad[0], misalign=misalign)
    vb = Rows(R, NV * D, NV * D + pad[1])
    ab = Rows(R, NV, NV + pad[2])
    bb = Rows(R, NV, NV + pad[2])
    ob = Rows(R, NV * D, NV * D + pad[3])
    qb.write(x["q"].reshape(R, -1)); kb.write(x["k"].reshape(R, -1)); vb.write(x["v"].reshape(R, -1))
    ab.write(x["alpha"].reshape(R, -1)); bb.write(x["beta"].reshape(R, -1))
    common = dict(nk=NK, nv=NV, d=D, state_pitch=pool.stride,
                  state_dtype=gdn.GDN_STATE_F16 if f16 else gdn.GDN_STATE_F32,
                  qk_stride=qb.stride, v_stride=vb.stride, gb_stride=ab.stride, o_stride=ob.stride)
    if splits is None:
        prefill(pool.ptr, qb.ptr, kb.ptr, vb.ptr, ab.ptr, bb.ptr, ob.ptr, batch=B, seq_len=T, **common)
    else:
        e32, es = 4, (2 if f16 else 4)
        for b in range(B):
            t0 = 0
            for n in splits:
                row = b * T + t0
                prefill(pool.ptr + b * pool.stride * es,
                        qb.ptr + row * qb.stride * e32, kb.ptr + row * kb.stride * e32,
                        vb.ptr + row * vb.stride * e32, ab.ptr + row * ab.stride * e32,
                        bb.ptr + row * bb.stride * e32, ob.ptr + row * ob.stride * e32,
                        batch=1, seq_len=n, **common)
                t0 += n
            assert t0 == T
    ref = S0.astype(np.float64)
    o_ref = oracle.prefill(ref, x["q"], x["k"], x["v"], x["alpha"], x["beta"], NK)
    torch.cuda.synchronize()
    o_gpu = ob.read().astype(np.float64).reshape(B, T, NV * D)
    S_gpu = to_f64_state(pool, B, NV, D, f16)
    return {
        "state_max_rel": max_rel_err(S_gpu, ref),
        "state_rel_l2": rel_l2(S_gpu, ref),
        "o_max_rel": max_rel_err(o_gpu, o_ref),
        "o_rel_l2": rel_l2(o_gpu, o_ref),
        "intact": all(b.intact() for b in (pool, qb, kb, vb, ab, bb, ob)),
        "S_gpu": S_gpu, "S_ref": ref,
    }
