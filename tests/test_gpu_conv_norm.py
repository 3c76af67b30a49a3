"""GPU parity: gdn_decode_conv_norm (conv ring + silu, q/k L2 norm, gates from logits, the step,
the gated norm, in one launch) against the fp64 oracle composed from its parts.

The conv state update is a pure data move (shift by one, append the token), so it is compared bit
for bit; the h-state and the bf16 output use the fp32 / fp16-state / bf16 bars of the other tests.
NV/NK = 1, 3, 8 and 9 run on the D = 128 kernels: fp32 (and fp16 with NV/NK = 9) on the one with a
CTA per value head, where the last reader of a key head's q/k ring rows writes them; fp16 with
NV/NK <= 8 on the one with a CTA per key head.  D != 128 and a misaligned state run on the general
kernel.  The workspace counters must be zero again after every call."""
import numpy as np
import pytest
import torch

import gdn_synth as gs
import gated_deltanet_linear_16_gb300 as gdn
import oracle
from tests.gpu_helpers import TOL_F32, TOL_REL_L2, Rows, bf16_to_f64, max_rel_err, rel_l2, state_pool

pytestmark = pytest.mark.gpu
EPS, L2_EPS = 1e-6, 1e-6


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def run(B, NK, NV, D, taps, f16, seed, steps=2, misalign=0, pad=(0, 0, 0, 0), ring_pad=0):
    C = (2 * NK + NV) * D
    sdt = np.float16 if f16 else np.float32
    S0 = gs.state_heads(seed, range(B), range(NV), D, dtype=sdt)
    first = gs.conv_decode_inputs(seed, B, NK, NV, D, taps, step=0)
    gn = gs.norm_weight(seed, D)
    pool = state_pool(B, NV, D, f16, 32, misalign)
    pool.write(S0.reshape(B, -1))
    ring = Rows(B, taps * C, taps * C + ring_pad)
    ring.write(first["ring"].reshape(B, -1))
    xb = Rows(B, C, C + pad[0])
    wb = Rows(1, taps * C)
    wb.write(first["conv_w"])
    brb, arb = Rows(B, NV, NV + pad[1]), Rows(B, NV, NV + pad[1])
    dtb, rateb = Rows(1, NV), Rows(1, NV)
    dtb.write(first["dt"]); rateb.write(first["rate"])
    zb = Rows(B, NV * D, NV * D + pad[2])
    gnb = Rows(1, D)
    gnb.write(gn)
    ob = Rows(B, NV * D, NV * D + pad[3], torch.int16)
    ws = torch.zeros(B * NK + 64, dtype=torch.int32, device="cuda")     # counters + a guard tail
    ws[B * NK:] = 12345

    ring_ref = first["ring"].copy()
    S_ref = S0.astype(np.float64)
    worst_out = 0.0
    for t in range(steps):
        x = gs.conv_decode_inputs(seed, B, NK, NV, D, taps, step=t)
        xb.write(x["x"]); brb.write(x["br"]); arb.write(x["ar"]); zb.write(x["z"])
        gdn.gdn_decode_conv_norm(pool.ptr, ring.ptr, xb.ptr, wb.ptr, brb.ptr, arb.ptr, dtb.ptr, rateb.ptr, zb.ptr,
                                 gnb.ptr, ob.ptr, ws, batch=B, nk=NK, nv=NV, d=D, taps=taps, eps=EPS, l2_eps=L2_EPS,
                                 state_dtype=gdn.GDN_STATE_F16 if f16 else gdn.GDN_STATE_F32,
                                 state_pitch=pool.stride, conv_pitch=ring.stride, x_stride=xb.stride,
                                 gate_stride=brb.stride, z_stride=zb.stride, out_stride=ob.stride)
        torch.cuda.synchronize()
        assert torch.count_nonzero(ws[:B * NK]).item() == 0, "workspace not left zero"
        assert torch.all(ws[B * NK:] == 12345).item()
        got = bf16_to_f64(ob.read()).reshape(B, NV, D)
        for b in range(B):
            y = oracle.conv_silu(ring_ref[b], x["x"][b], first["conv_w"])
            q = oracle.l2norm_heads(y[:NK * D], D, L2_EPS)
            k = oracle.l2norm_heads(y[NK * D:2 * NK * D], D, L2_EPS)
            v = y[2 * NK * D:]
            beta, alpha = oracle.gates(x["br"][b], x["ar"][b], first["dt"], first["rate"])
            o = oracle.decode_f64(S_ref[b:b + 1], q, k, v, alpha, beta, NK)
            ref = oracle.gated_rmsnorm(o.reshape(NV, D), x["z"][b].reshape(NV, D), gn, EPS)
            worst_out = max(worst_out, rel_l2(got[b], ref))
    S_gpu = pool.read().astype(np.float64).reshape(B, NV, D, D)
    intact = all(r.intact() for r in (pool, ring, xb, wb, brb, arb, dtb, rateb, zb, gnb, ob))
    return {"out": worst_out, "S_gpu": S_gpu, "S_ref": S_ref, "ring": ring.read(),
            "ring_ref": ring_ref.reshape(B, -1), "intact": intact}


def check(r, f16):
    assert r["intact"], "guard band or padding overwritten"
    assert np.array_equal(r["ring"], r["ring_ref"]), "conv state update differs"
    if f16:
        assert rel_l2(r["S_gpu"], r["S_ref"]) <= TOL_REL_L2
    else:
        assert max_rel_err(r["S_gpu"], r["S_ref"]) <= TOL_F32, max_rel_err(r["S_gpu"], r["S_ref"])
    assert r["out"] <= TOL_REL_L2, r["out"]


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("NK,NV", [(2, 6), (4, 4), (1, 8), (1, 9)])
def test_d128_kernel(f16, NK, NV):
    check(run(2, NK, NV, 128, 4, f16, seed=51 + NV, steps=3, pad=(4, 1, 2, 6), ring_pad=16), f16)


@pytest.mark.parametrize("taps", [1, 2, 3, 4, 5, 8])
def test_taps(taps):
    """Up to 4 taps the per-value-head kernel holds a channel's ring entries in 3-entry register
    arrays, above that in 7-entry ones (conv_norm_d128<float, ..., MT = 4 | 8>)."""
    check(run(2, 2, 6, 128, taps, False, seed=60 + taps), False)


@pytest.mark.parametrize("taps", [2, 6])
def test_taps_f16_per_value_head(taps):
    """fp16 with NV / NK = 9 > 8 takes the per-value-head kernel (conv_norm_d128<__half, ...>) for
    both tap bounds."""
    check(run(2, 1, 9, 128, taps, True, seed=90 + taps), True)


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("NK,NV,D,misalign", [(2, 4, 64, 0), (2, 6, 128, 1), (1, 2, 5, 0)])
def test_general_kernel(f16, NK, NV, D, misalign):
    check(run(2, NK, NV, D, 4, f16, seed=70 + D + NV, misalign=misalign), f16)


def test_full_layer():
    """One Qwen3.8-27B-shaped layer at batch 32: 1536 CTAs, three readers per key head."""
    check(run(32, 16, 48, 128, 4, False, seed=80, steps=2), False)
