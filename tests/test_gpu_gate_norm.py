"""GPU parity: gdn_gate_norm / gdn_gate_norm_q8 (the gated RMS norm as its own call, gdn.rs
`gdn_gate_norm` and `gdn_gate_norm_q`) against the fp64 oracle, alone and after a prefill call.

bf16 output: relative L2 against the oracle's fp64 norm (the bf16 bar).  int8: the fp32 values y
the kernel writes are held to the fp32 bar, and the oracle's fp32 quantiser applied to them must
give the kernel's codes and scales bit for bit.  Strided rows, guard bands, D = 5 ... 256 and an
all-zero head (gate input 0) are covered."""
import numpy as np
import pytest
import torch

import gdn_synth as gs
import gated_deltanet_linear_16_gb300 as gdn
import oracle
from tests.gpu_helpers import TOL_F32, TOL_REL_L2, Rows, bf16_to_f64, max_rel_err, rel_l2

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _inputs(rows, nv, d, seed):
    rng = np.random.default_rng(seed)
    o = (rng.standard_normal((rows, nv * d)) * rng.choice([1e-3, 0.1, 3.0], size=(rows, 1))).astype(np.float32)
    z = rng.standard_normal((rows, nv * d)).astype(np.float32)
    z[0, (nv - 1) * d:] = 0.0                         # one all-zero head: silu(0) = 0
    gn = gs.norm_weight(seed, d)
    return o, z, gn


def _ref(o, z, gn, nv, d):
    rows = o.shape[0]
    return oracle.gated_rmsnorm(o.astype(np.float64).reshape(rows * nv, d), z.reshape(rows * nv, d), gn,
                                EPS).reshape(rows, nv * d)


@pytest.mark.parametrize("rows,nv,d,pad", [(5, 3, 128, 3), (5, 3, 128, 4), (1000, 48, 128, 0), (9, 1, 128, 0), (33, 2, 64, 4),
                                            (4, 3, 5, 0), (3, 2, 256, 8), (1, 48, 128, 4)])
def test_bf16(rows, nv, d, pad):
    """pad = 0 or a multiple of 4 keeps D = 128 rows 16-byte aligned (the vector kernel); 3 does not."""
    o, z, gn = _inputs(rows, nv, d, seed=300 + d + pad)
    hv = nv * d
    ob, zb, gb = Rows(rows, hv, hv + pad), Rows(rows, hv, hv + 2 * pad), Rows(1, d)
    out = Rows(rows, hv, hv + 4 * pad, torch.int16)
    ob.write(o); zb.write(z); gb.write(gn)
    gdn.gdn_gate_norm(ob.ptr, zb.ptr, gb.ptr, out.ptr, rows=rows, nv=nv, d=d, eps=EPS, o_stride=ob.stride,
                      z_stride=zb.stride, out_stride=out.stride)
    torch.cuda.synchronize()
    got = bf16_to_f64(out.read())
    assert rel_l2(got, _ref(o, z, gn, nv, d)) <= TOL_REL_L2
    assert not got[0, (nv - 1) * d:].any()
    assert all(b.intact() for b in (ob, zb, gb, out)), "guard band or padding overwritten"


@pytest.mark.parametrize("rows,nv,d,with_y,pad", [(6, 3, 128, True, 4), (6, 3, 128, True, 1), (777, 48, 128, True, 0),
                                                  (5, 1, 128, True, 4), (7, 2, 128, False, 0),
                                                  (9, 2, 64, True, 4), (2, 4, 32, True, 4), (3, 2, 256, True, 4),
                                                  (6, 3, 128, False, 4)])
def test_q8(rows, nv, d, with_y, pad):
    """pad 4 / 0: the D = 128 vector kernel (a quarter-warp per (row, head), so NV = 1 or 2 puts
    several rows' heads in one warp; an int8 group over 2 lanes); pad 1: the general kernel."""
    o, z, gn = _inputs(rows, nv, d, seed=400 + d + pad)
    hv = nv * d
    ob, zb, gb = Rows(rows, hv, hv + pad), Rows(rows, hv, hv + pad), Rows(1, d)
    xq, xs = Rows(rows, hv, hv + 16, torch.int8), Rows(rows, hv // 32, hv // 32 + 2)
    yb = Rows(rows, hv, hv + 4) if with_y else None
    ob.write(o); zb.write(z); gb.write(gn)
    gdn.gdn_gate_norm_q8(ob.ptr, zb.ptr, gb.ptr, xq.ptr, xs.ptr, yb.ptr if yb else None, rows=rows, nv=nv, d=d,
                         eps=EPS, o_stride=ob.stride, z_stride=zb.stride, xq_stride=xq.stride,
                         xs_stride=xs.stride, y_stride=yb.stride if yb else 0)
    torch.cuda.synchronize()
    ref = _ref(o, z, gn, nv, d).reshape(-1)
    codes = xq.read().reshape(-1).astype(np.int64)
    scales = xs.read().reshape(-1)
    step = np.repeat(scales.astype(np.float64), 32)
    assert np.all(np.abs(codes * step - ref) <= 0.5 * step * (1 + 1e-6) + TOL_F32 * np.max(np.abs(ref)))
    g0 = ((nv - 1) * d) // 32
    assert np.all(scales[g0:g0 + d // 32] == 1.0) and not codes[(nv - 1) * d:nv * d].any()
    if yb is not None:
        y = yb.read().reshape(-1)
        assert max_rel_err(y, ref) <= TOL_F32, max_rel_err(y, ref)
        c_ref, s_ref = oracle.quant_q8(y)
        assert np.array_equal(codes, c_ref.astype(np.int64)), "codes differ from the fp32 quantiser's"
        assert np.array_equal(scales.view(np.uint32), s_ref.view(np.uint32)), "scales differ"
    bufs = [ob, zb, gb, xq, xs] + ([yb] if yb else [])
    assert all(b.intact() for b in bufs), "guard band or padding overwritten"


def test_prefill_then_norm():
    """gdn_prefill_seq's raw o for every token, normed by gdn_gate_norm: against the oracle's prefill
    followed by its norm."""
    B, NK, NV, D, T = 2, 2, 6, 128, 20
    rows = B * T
    x = gs.prefill_inputs(7, B, T, NK, NV, D)
    z = np.stack([gs.decode_inputs(7, B, NK, NV, D, step=t)["z"] for t in range(T)], axis=1).reshape(rows, NV * D)
    gn = gs.norm_weight(7, D)
    S0 = gs.state_heads(7, range(B), range(NV), D)
    dev = torch.device("cuda")
    t = {k: torch.from_numpy(np.ascontiguousarray(v.reshape(rows, -1))).to(dev) for k, v in x.items()}
    S = torch.from_numpy(S0).to(dev)
    o = torch.empty((rows, NV * D), device=dev)
    gdn.gdn_prefill_seq(S, t["q"], t["k"], t["v"], t["alpha"], t["beta"], o, batch=B, seq_len=T, nk=NK, nv=NV, d=D)
    out = torch.empty((rows, NV * D), dtype=torch.int16, device=dev)
    gdn.gdn_gate_norm(o, torch.from_numpy(z).to(dev), torch.from_numpy(gn).to(dev), out, rows=rows, nv=NV, d=D,
                      eps=EPS)
    torch.cuda.synchronize()
    o_ref = oracle.prefill(S0.astype(np.float64), x["q"], x["k"], x["v"], x["alpha"], x["beta"], NK)
    ref = oracle.gated_rmsnorm(o_ref.reshape(rows * NV, D), z.reshape(rows * NV, D), gn, EPS)
    assert rel_l2(bf16_to_f64(out.cpu().numpy()).reshape(rows * NV, D), ref) <= TOL_REL_L2


@pytest.mark.parametrize("pad,offset,scale", [(0, 0.0, 1.0), (1, 0.0, 1.0), (0, 2.0 ** -15, 1.0), (0, 2.0 ** -14, 1.0),
                                              (0, 2.0 ** -13, 1.0), (1, 2.0 ** -14, 1.0), (0, 0.0, 1e-34),
                                              (0, 2.0 ** -14, 1e-34)])
def test_q8_near_ties(pad, offset, scale):
    """Quotients y / scale planted within a few ulp of half-integers (the ties and near-ties of
    round-half-even), on the vector kernel (pad 0) and the general one (pad 1): with z = 20
    (silu(20) = 20 in fp32) and gn = 1, y is o times one per-head factor up to rounding, so o =
    +-(k + 1/2 + e) / 127 next to a group maximum of 1 puts 127 y / max|y| next to k + 1/2 + e.
    e = 0, or +-offset at random (2^-15 .. 2^-13: quotients a few hundred ulp from a tie).  scale
    multiplies o: at 1e-34 the norm's eps dominates and the
    groups' scales fall far below 2^-60, where the vector kernel's quotients come from the IEEE
    division instead of the corrected reciprocal.  Codes and scales must equal the oracle's fp32
    quantiser (IEEE quotients) on the kernel's own y bit for bit."""
    rows, nv, d = 4, 3, 128
    hv = nv * d
    rng = np.random.default_rng(77 + int(offset * 2 ** 20))
    k = rng.integers(0, 127, size=(rows, hv // 32, 32)).astype(np.float64)
    e = rng.choice([-1.0, 1.0], size=k.shape) * offset
    o = rng.choice([-1.0, 1.0], size=k.shape) * (k + 0.5 + e) / 127.0
    o[:, :, 0] = rng.choice([-1.0, 1.0], size=(rows, hv // 32))       # the group maximum, |o| = 1
    o = (o.reshape(rows, hv) * scale).astype(np.float32)
    z = np.full((rows, hv), 20.0, np.float32)
    gn = np.ones(d, np.float32)
    ob, zb, gb = Rows(rows, hv, hv + pad), Rows(rows, hv, hv + pad), Rows(1, d)
    xq, xs, yb = Rows(rows, hv, hv + 16, torch.int8), Rows(rows, hv // 32, hv // 32 + 2), Rows(rows, hv, hv + 4)
    ob.write(o); zb.write(z); gb.write(gn)
    gdn.gdn_gate_norm_q8(ob.ptr, zb.ptr, gb.ptr, xq.ptr, xs.ptr, yb.ptr, rows=rows, nv=nv, d=d, eps=EPS,
                         o_stride=ob.stride, z_stride=zb.stride, xq_stride=xq.stride, xs_stride=xs.stride,
                         y_stride=yb.stride)
    torch.cuda.synchronize()
    y = yb.read().reshape(-1)
    codes = xq.read().reshape(-1).astype(np.int64)
    scales = xs.read().reshape(-1)
    q = y.reshape(-1, 32).astype(np.float64) / scales[:, None].astype(np.float64)
    near = np.abs(np.abs(q) - np.floor(np.abs(q)) - 0.5) < 1e-3
    assert near[:, 1:].mean() > 0.9, "the planted quotients did not land next to half-integers"
    c_ref, s_ref = oracle.quant_q8(y)
    assert np.array_equal(scales.view(np.uint32), s_ref.view(np.uint32)), "scales differ"
    assert np.array_equal(codes, c_ref.astype(np.int64)), "codes differ from the fp32 quantiser's"
    assert all(b.intact() for b in (ob, zb, gb, xq, xs, yb)), "guard band or padding overwritten"
