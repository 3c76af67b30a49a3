"""GPU parity: gdn_decode_norm_q8 (decode + gated norm + int8 groups of 32, gdn.rs
`gdn_gate_norm_q`) against the fp64 oracle.

Three checks per call:
* the fp32 normed values y the kernel also writes, against the oracle's fp64 norm output
  (fp32-state bar, or the fp16-state relative-L2 bar);
* the quantisation itself, bit for bit: the oracle's fp32 group quantiser applied to the
  kernel's own y must give exactly the kernel's codes and scales (the codes are integers
  decided by fp32 arithmetic, so both sides decide in fp32 from the same values);
* the dequantised codes against the oracle's fp64 y: within half a quantisation step plus the
  value tolerance.
The D = 128 kernel's three load variants (one CTA per SM or fewer, register batches, staged)
and the general kernel (D = 32, 64, a misaligned state) all run; one head's gate input is zero,
so its groups are all zero (scale 1, codes 0)."""
import numpy as np
import pytest
import torch

import gdn_synth as gs
import gated_deltanet_linear_16_gb300 as gdn
import oracle
from tests.gpu_helpers import TOL_F32, TOL_REL_L2, Rows, max_rel_err, rel_l2, state_pool

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def run_q8(B, NK, NV, D, f16, seed, T=2, misalign=0, with_y=True, zero_head=True):
    sdt = np.float16 if f16 else np.float32
    S0 = gs.state_heads(seed, range(B), range(NV), D, dtype=sdt)
    gn = gs.norm_weight(seed, D)
    pool = state_pool(B, NV, D, f16, 8, misalign)
    pool.write(S0.reshape(B, -1))
    ref = S0.astype(np.float64)
    qb, kb = Rows(B, NK * D, NK * D + 4), Rows(B, NK * D, NK * D + 4)
    vb, zb = Rows(B, NV * D, NV * D + 4), Rows(B, NV * D, NV * D + 8)
    ab, bb = Rows(B, NV, NV + 1), Rows(B, NV, NV + 1)
    gnb = Rows(1, D)
    gnb.write(gn)
    hv = NV * D
    xq = Rows(B, hv, hv + 16, torch.int8)
    xs = Rows(B, hv // 32, hv // 32 + 2)
    yb = Rows(B, hv, hv + 4) if with_y else None
    res = {"codes": [], "scales": []}
    for t in range(T):
        x = gs.decode_inputs(seed, B, NK, NV, D, step=t)
        if zero_head:
            x["z"][0, (NV - 1) * D:] = 0.0          # last head of sequence 0: silu(0) = 0, all-zero groups
        qb.write(x["q"]); kb.write(x["k"]); vb.write(x["v"])
        ab.write(x["alpha"]); bb.write(x["beta"]); zb.write(x["z"])
        gdn.gdn_decode_norm_q8(pool.ptr, qb.ptr, kb.ptr, vb.ptr, ab.ptr, bb.ptr, zb.ptr, gnb.ptr, xq.ptr, xs.ptr,
                               yb.ptr if yb else None, batch=B, nk=NK, nv=NV, d=D, eps=EPS,
                               state_pitch=pool.stride, state_dtype=gdn.GDN_STATE_F16 if f16 else gdn.GDN_STATE_F32,
                               qk_stride=qb.stride, v_stride=vb.stride, gb_stride=ab.stride, z_stride=zb.stride,
                               xq_stride=xq.stride, xs_stride=xs.stride, y_stride=yb.stride if yb else 0)
        o_ref = oracle.decode(ref, x["q"], x["k"], x["v"], x["alpha"], x["beta"], NK)
        y_ref = oracle.gated_rmsnorm(o_ref.reshape(B * NV, D), x["z"].reshape(B * NV, D), gn, EPS).reshape(-1)
        torch.cuda.synchronize()
        codes = xq.read().reshape(-1).astype(np.int64)
        scales = xs.read().reshape(-1)
        res["codes"].append(codes)
        res["scales"].append(scales)
        step = np.repeat(scales.astype(np.float64), 32)
        deq = codes * step
        if f16:
            assert rel_l2(deq, y_ref) <= TOL_REL_L2, (t, rel_l2(deq, y_ref))
        else:
            bound = 0.5 * step * (1 + 1e-6) + TOL_F32 * np.max(np.abs(y_ref))
            assert np.all(np.abs(deq - y_ref) <= bound), (t, np.max(np.abs(deq - y_ref) - bound))
        if zero_head:
            g0 = ((NV - 1) * D) // 32
            assert np.all(scales[g0:g0 + D // 32] == 1.0) and not codes[(NV - 1) * D:NV * D].any()
        if yb is not None:
            y_gpu = yb.read().reshape(-1)
            if f16:
                assert rel_l2(y_gpu, y_ref) <= TOL_REL_L2
            else:
                assert max_rel_err(y_gpu, y_ref) <= TOL_F32, max_rel_err(y_gpu, y_ref)
            c_ref, s_ref = oracle.quant_q8(y_gpu)
            assert np.array_equal(codes, c_ref.astype(np.int64)), "codes differ from the fp32 quantiser's"
            assert np.array_equal(scales.view(np.uint32), s_ref.view(np.uint32)), "scales differ"
    S_gpu = pool.read().astype(np.float64).reshape(B, NV, D, D)
    if f16:
        assert rel_l2(S_gpu, ref) <= TOL_REL_L2
    else:
        assert max_rel_err(S_gpu, ref) <= TOL_F32
    bufs = [pool, qb, kb, vb, ab, bb, zb, gnb, xq, xs] + ([yb] if yb else [])
    assert all(b.intact() for b in bufs), "guard band or padding overwritten"
    return res


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("B,NK,NV", [(3, 2, 6), (2, 16, 48), (8, 16, 48), (32, 16, 48)])
def test_d128_variants(f16, B, NK, NV):
    """Grids of 18, 96, 384 and 1536 CTAs: the all-in-registers (18, 96), register-batched and
    staged loads."""
    run_q8(B, NK, NV, 128, f16, seed=100 + B, T=2 if B < 32 else 1)


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("NK,NV,D,misalign", [(2, 4, 64, 0), (1, 3, 32, 0), (2, 6, 128, 1)])
def test_general_kernel(f16, NK, NV, D, misalign):
    run_q8(2, NK, NV, D, f16, seed=110 + D, misalign=misalign)


def test_without_y_gives_the_same_codes():
    a = run_q8(4, 2, 6, 128, False, seed=120, with_y=True)
    b = run_q8(4, 2, 6, 128, False, seed=120, with_y=False)
    for ca, cb, sa, sb in zip(a["codes"], b["codes"], a["scales"], b["scales"]):
        assert np.array_equal(ca, cb) and np.array_equal(sa.view(np.uint32), sb.view(np.uint32))
