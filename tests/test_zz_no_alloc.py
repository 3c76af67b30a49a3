"""GPU: gdn_decode_conv_norm_noalloc, the decode from projections for callers that cannot allocate
device memory, against gdn_decode_conv_norm (caller's workspace) on the same seeded inputs, two
calls in a row.

The allocation-free entry runs exactly the kernels of the workspace entry on identical inputs, with
only the counters' home changed (a static array inside the library), so the state, the bf16 output
and the conv ring must agree bit for bit after every call.  The second call only agrees if the first
left the static counters at zero: otherwise the wrong block would take itself for the last reader of
a key head's q/k ring rows and the ring would go stale.  Both entries are also checked once against
the fp64 oracle composed from its parts (the one tolerance in this file).

This file is named to run after every other test, so it also covers a process in which the other
entry points ran first; it passes on its own in a fresh process as well."""
import numpy as np
import pytest
import torch

import gdn_synth as gs
import gated_deltanet_linear_16_gb300 as gdn
import oracle
from tests.gpu_helpers import TOL_F32, TOL_REL_L2, bf16_to_f64, max_rel_err, rel_l2

pytestmark = pytest.mark.gpu
EPS, L2_EPS = 1e-6, 1e-6


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _inputs(B, NK, NV, D, taps, f16, seed, steps=2):
    dev = torch.device("cuda")
    sdt = np.float16 if f16 else np.float32
    S0_np = gs.state_heads(seed, range(B), range(NV), D, dtype=sdt)
    S0 = torch.from_numpy(S0_np.reshape(B, -1)).to(dev)
    host = [gs.conv_decode_inputs(seed, B, NK, NV, D, taps, step=t) for t in range(steps)]
    ring0 = torch.from_numpy(host[0]["ring"].reshape(B, -1)).to(dev)
    fixed = {k: torch.from_numpy(host[0][k]).to(dev) for k in ("conv_w", "dt", "rate")}
    per = [{k: torch.from_numpy(s[k]).to(dev) for k in ("x", "br", "ar", "z")} for s in host]
    gn_np = gs.norm_weight(seed, D)
    gn = torch.from_numpy(gn_np).to(dev)
    return S0, ring0, fixed, per, gn, (S0_np, host, gn_np)


def _oracle_step(S_ref, ring_ref, h, gn_np, NK, NV, D):
    """One step of the oracle for every sequence; S_ref, ring_ref updated in place; bf16-bar output."""
    B = S_ref.shape[0]
    out = np.empty((B, NV, D))
    for b in range(B):
        y = oracle.conv_silu(ring_ref[b], h["x"][b], h["conv_w"])
        q = oracle.l2norm_heads(y[:NK * D], D, L2_EPS)
        k = oracle.l2norm_heads(y[NK * D:2 * NK * D], D, L2_EPS)
        v = y[2 * NK * D:]
        beta, alpha = oracle.gates(h["br"][b], h["ar"][b], h["dt"], h["rate"])
        o = oracle.decode_f64(S_ref[b:b + 1], q, k, v, alpha, beta, NK)
        out[b] = oracle.gated_rmsnorm(o.reshape(NV, D), h["z"][b].reshape(NV, D), gn_np, EPS)
    return out


@pytest.mark.parametrize("B,NK,NV,D,f16", [
    (32, 16, 48, 128, False),      # one full layer: three value-head blocks share each key-head counter
    (4, 16, 48, 128, False),
    (3, 2, 6, 128, True),          # fp16: one block per key head (counters unused)
    (2, 2, 4, 64, False),          # general kernel
])
def test_matches_workspace_entry_two_calls(B, NK, NV, D, f16):
    taps = 4
    S0, ring0, fixed, per, gn, (S0_np, host, gn_np) = _inputs(B, NK, NV, D, taps, f16, seed=90 + D + NV + B)
    sd = gdn.GDN_STATE_F16 if f16 else gdn.GDN_STATE_F32
    S_a, ring_a = S0.clone(), ring0.clone()
    S_b, ring_b = S0.clone(), ring0.clone()
    ws = torch.zeros(B * NK, dtype=torch.int32, device="cuda")
    kw = dict(batch=B, nk=NK, nv=NV, d=D, taps=taps, eps=EPS, l2_eps=L2_EPS, state_dtype=sd)
    S_ref = S0_np.astype(np.float64)
    ring_ref = host[0]["ring"].copy()
    for t in range(2):
        out_a = torch.full((B, NV * D), 0x7F7F, dtype=torch.int16, device="cuda")
        out_b = torch.full((B, NV * D), 0x7F7F, dtype=torch.int16, device="cuda")
        p = per[t]
        gdn.gdn_decode_conv_norm(S_a, ring_a, p["x"], fixed["conv_w"], p["br"], p["ar"], fixed["dt"],
                                 fixed["rate"], p["z"], gn, out_a, ws, **kw)
        gdn.gdn_decode_conv_norm_noalloc(S_b, ring_b, p["x"], fixed["conv_w"], p["br"], p["ar"], fixed["dt"],
                                         fixed["rate"], p["z"], gn, out_b, **kw)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: identical bits
        assert torch.equal(out_b, out_a), f"bf16 output differs after call {t + 1}"
        assert torch.equal(ring_b, ring_a), f"conv state differs after call {t + 1}"
        assert torch.equal(S_b.view(torch.int16 if f16 else torch.int32),
                           S_a.view(torch.int16 if f16 else torch.int32)), f"state differs after call {t + 1}"
        assert torch.count_nonzero(ws).item() == 0
        # and both against the fp64 oracle
        h = dict(host[t], conv_w=host[0]["conv_w"], dt=host[0]["dt"], rate=host[0]["rate"])
        out_ref = _oracle_step(S_ref, ring_ref, h, gn_np, NK, NV, D)
        got = bf16_to_f64(out_b.cpu().numpy()).reshape(B, NV, D)
        assert rel_l2(got, out_ref) <= TOL_REL_L2, (t, rel_l2(got, out_ref))
        assert np.array_equal(ring_b.cpu().numpy(), ring_ref.reshape(B, -1)), t
    S_got = S_b.double().cpu().numpy().reshape(S_ref.shape)
    if f16:
        assert rel_l2(S_got, S_ref) <= TOL_REL_L2
    else:
        assert max_rel_err(S_got, S_ref) <= TOL_F32, max_rel_err(S_got, S_ref)


def test_rejects_batch_beyond_static_counters():
    """batch * NK above the static array's size is refused before anything runs."""
    B, NK, NV, D, taps = 2, 16, 48, 128, 4
    S0, ring0, fixed, per, gn, _ = _inputs(B, NK, NV, D, taps, False, seed=7, steps=1)
    out = torch.full((B, NV * D), 0x1234, dtype=torch.int16, device="cuda")
    S, ring = S0.clone(), ring0.clone()
    big = gdn.GDN_NOALLOC_MAX_KEY_HEADS // NK + 1
    p = per[0]
    with pytest.raises(gdn.GdnError) as err:
        gdn.gdn_decode_conv_norm_noalloc(S, ring, p["x"], fixed["conv_w"], p["br"], p["ar"], fixed["dt"],
                                         fixed["rate"], p["z"], gn, out, batch=big, nk=NK, nv=NV, d=D,
                                         taps=taps, state_dtype=gdn.GDN_STATE_F32)
    assert err.value.status == 2        # GDN_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.equal(S, S0) and torch.equal(ring, ring0)
    assert torch.all(out == 0x1234).item()
