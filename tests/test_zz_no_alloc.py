"""GPU: gdn_decode_conv_norm_noalloc (counters in the library's static device memory) against
gdn_decode_conv_norm (caller's workspace) on the same seeded inputs, two calls in a row.

The second call only matches if the first left the static counters at zero (otherwise the wrong
CTA would take itself for the last reader of a key head's ring rows and the ring would go stale).
This file is named to run after every other test, so it also covers a process in which the other
entry points ran first; it passes on its own as well."""
import numpy as np
import pytest
import torch

import gdn_synth as gs
import gated_deltanet_linear_16_gb300 as gdn
from tests.gpu_helpers import TOL_F32, TOL_REL_L2, bf16_to_f64, max_rel_err, rel_l2

pytestmark = pytest.mark.gpu
EPS, L2_EPS = 1e-6, 1e-6


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _inputs(B, NK, NV, D, taps, f16, seed):
    dev = torch.device("cuda")
    sdt = np.float16 if f16 else np.float32
    S0 = torch.from_numpy(gs.state_heads(seed, range(B), range(NV), D, dtype=sdt).reshape(B, -1)).to(dev)
    steps = [gs.conv_decode_inputs(seed, B, NK, NV, D, taps, step=t) for t in range(2)]
    ring0 = torch.from_numpy(steps[0]["ring"].reshape(B, -1)).to(dev)
    fixed = {k: torch.from_numpy(steps[0][k]).to(dev) for k in ("conv_w", "dt", "rate")}
    per = [{k: torch.from_numpy(s[k]).to(dev) for k in ("x", "br", "ar", "z")} for s in steps]
    gn = torch.from_numpy(gs.norm_weight(seed, D)).to(dev)
    return S0, ring0, fixed, per, gn


@pytest.mark.parametrize("B,NK,NV,D,f16", [(4, 16, 48, 128, False), (3, 2, 6, 128, True), (2, 2, 4, 64, False)])
def test_matches_workspace_entry_two_calls(B, NK, NV, D, f16):
    taps = 4
    S0, ring0, fixed, per, gn = _inputs(B, NK, NV, D, taps, f16, seed=90 + D + NV)
    sd = gdn.GDN_STATE_F16 if f16 else gdn.GDN_STATE_F32
    S_a, ring_a = S0.clone(), ring0.clone()
    S_b, ring_b = S0.clone(), ring0.clone()
    ws = torch.zeros(B * NK, dtype=torch.int32, device="cuda")
    kw = dict(batch=B, nk=NK, nv=NV, d=D, taps=taps, eps=EPS, l2_eps=L2_EPS, state_dtype=sd)
    for t in range(2):
        out_a = torch.empty((B, NV * D), dtype=torch.int16, device="cuda")
        out_b = torch.full((B, NV * D), 0x7F7F, dtype=torch.int16, device="cuda")
        p = per[t]
        gdn.gdn_decode_conv_norm(S_a, ring_a, p["x"], fixed["conv_w"], p["br"], p["ar"], fixed["dt"],
                                 fixed["rate"], p["z"], gn, out_a, ws, **kw)
        gdn.gdn_decode_conv_norm_noalloc(S_b, ring_b, p["x"], fixed["conv_w"], p["br"], p["ar"], fixed["dt"],
                                         fixed["rate"], p["z"], gn, out_b, **kw)
        torch.cuda.synchronize()
        assert rel_l2(bf16_to_f64(out_b.cpu().numpy()), bf16_to_f64(out_a.cpu().numpy())) <= TOL_REL_L2, t
        assert torch.equal(ring_b, ring_a), f"conv state differs after call {t + 1}"
        sa = S_a.double().cpu().numpy()
        sb = S_b.double().cpu().numpy()
        if f16:
            assert rel_l2(sb, sa) <= TOL_REL_L2, t
        else:
            assert max_rel_err(sb, sa) <= TOL_F32, t
    assert torch.count_nonzero(ws).item() == 0


def test_rejects_batch_beyond_static_counters():
    """batch * NK above the static array's size is refused before anything runs."""
    B, NK, NV, D, taps = 2, 16, 48, 128, 4
    S0, ring0, fixed, per, gn = _inputs(B, NK, NV, D, taps, False, seed=7)
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
