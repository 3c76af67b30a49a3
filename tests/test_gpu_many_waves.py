"""GPU parity for the kernel instances that grids of more than four waves take.

The D = 128 launchers of gdn_decode*, gdn_decode_chunk2 and the fp32
gdn_decode_conv_norm launch a kernel early (programmatic stream serialisation
with a partial L2 prefetch) only while its grid is at most four waves of
resident CTAs.  Above that they take a separate template instance with a plain
launch and none of the grid-dependency code.  Each test here sizes its batch
from the GPU's SM count so that the grid is past that threshold, names the
instance it reaches, and checks it against the fp64 oracle at the bars of the
other parity tests (fp32 state and raw o within 1e-4 of max |ref|; fp16
state, raw o from an fp16 state and bf16 out within 2e-2 relative L2).  Where
the whole batch is too large for the oracle, it checks seeded sample slots
element by element (their inputs drawn by the counter-based generator, the
other slots filled by torch's generator at the same distribution: heads never
interact) and whole-grid properties: finite results, untouched slot padding,
and bit-identity with the single-token kernel where the header promises it."""
import math

import numpy as np
import pytest
import torch

import gdn_synth as gs
import gated_deltanet_linear_16_gb300 as gdn
import oracle
from tests.gpu_helpers import TOL_F32, TOL_REL_L2, bf16_to_f64, check_decode, max_rel_err, rel_l2, run_decode_case
from tests.test_gpu_chunk2 import run as run_chunk2
from tests.test_gpu_conv_norm import check as check_conv, run as run_conv
from tests.test_gpu_q8 import run_q8

pytestmark = pytest.mark.gpu

NK, NV, D = 16, 48, 128
EPS, L2_EPS = 1e-6, 1e-6
EARLY_MAX_WAVES = 4           # the launchers' early-launch limit, in waves


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield cuda_lib
    torch.cuda.empty_cache()


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def batch_past_early(ctas_per_sm, at_least):
    """Smallest batch whose grid of B * NV CTAs exceeds four waves of `ctas_per_sm` CTAs per SM
    (and at least `at_least`)."""
    return max(at_least, math.floor(EARLY_MAX_WAVES * sms() * ctas_per_sm / NV) + 1)


# ------------------------------------------------------------------ single-token decode

@pytest.mark.parametrize("norm", [False, True])
def test_decode_fp32_plain_staged(norm):
    """fp32 state, 3 staged CTAs per SM, grid > 4 waves (B = 40 on 152 SMs: 1920 CTAs):
    decode_d128<float, kEpiRaw | kEpiBf16, STAGED = true, NB = 1, MINB = 3, EARLY = false>."""
    B = batch_past_early(3, 40)
    r = run_decode_case(B, NK, NV, D, 2, f16=False, norm=norm, seed=300 + norm)
    check_decode(r, f16=False, norm=norm)


def test_decode_fp32_plain_staged_int8():
    """fp32 state, int8 epilogue, grid > 4 waves:
    decode_d128<float, kEpiQ8, true, 1, 3, false>."""
    run_q8(batch_past_early(3, 40), NK, NV, D, False, seed=302, T=1)


@pytest.mark.parametrize("norm", [False, True])
def test_decode_fp16_plain_staged(norm):
    """fp16 state, 4 staged CTAs per SM, grid > 4 waves (B = 64 on 152 SMs: 3072 CTAs):
    decode_d128<__half, kEpiRaw | kEpiBf16, true, 1, 4, false>."""
    B = batch_past_early(4, 64)
    r = run_decode_case(B, NK, NV, D, 2, f16=True, norm=norm, seed=304 + norm, pitch_pad=4096)
    check_decode(r, f16=True, norm=norm)


def test_decode_fp16_plain_staged_int8():
    """fp16 state, int8 epilogue, grid > 4 waves:
    decode_d128<__half, kEpiQ8, true, 1, 4, false>."""
    run_q8(batch_past_early(4, 64), NK, NV, D, True, seed=306, T=1)


# ------------------------------------------------------------------ two-token verify

def test_chunk2_fp32_plain_staged():
    """fp32 state, grid > 4 waves (B = 40): chunk2_d128<float, 8, STAGED = true, 1, 3, EARLY = false>,
    against the oracle and bit for bit against two gdn_decode calls (decode_d128<float, kEpiRaw,
    true, 1, 3, false>)."""
    B = batch_past_early(3, 40)
    got, two, (ref_mid, ref_S, ref_o), intact, bufs = run_chunk2(B, NK, NV, D, False, seed=310, pitch_pad=64)
    assert intact, "guard band or padding overwritten"
    pool, mid, ob = bufs
    assert np.array_equal(pool.read(), two["S"])
    assert np.array_equal(mid.read(), two["M"])
    assert np.array_equal(ob.read(), two["o"])
    assert max_rel_err(got["M"], ref_mid) <= TOL_F32
    assert max_rel_err(got["S"], ref_S) <= TOL_F32
    assert max_rel_err(got["o"], ref_o) <= TOL_F32


def test_chunk2_fp16_pool_256_slots():
    """The two-token row of the benchmark: 256-slot fp16 pool, slot pitch 48*128*128 + 4096 halves
    (12288 CTAs): chunk2_d128<__half, 8, true, 1, 4, false>.  The whole pool bit for bit against two
    gdn_decode calls (decode_d128<__half, kEpiRaw, true, 1, 4, false>); sample slots against the
    oracle; the slot padding of the state and of the intermediate pool stays zero."""
    PB, seed = 256, 311
    hs = NV * D * D
    pitch = hs + 4096
    dev = torch.device("cuda")
    pool = torch.zeros((PB, pitch), dtype=torch.float16, device=dev)
    pool[:, :hs].normal_(0.0, 0.02)
    sample = [0, 131, 255]
    S0 = {}
    for b in sample:
        s0 = gs.state_heads(seed, [b], range(NV), D, dtype=np.float16)[0]
        pool[b, :hs] = torch.from_numpy(s0.reshape(-1)).to(dev)
        S0[b] = s0.astype(np.float64)[None]
    x0 = gs.decode_inputs(seed, PB, NK, NV, D, step=0)
    x1 = gs.decode_inputs(seed, PB, NK, NV, D, step=1)
    inter = {n: torch.from_numpy(np.stack([x0[n], x1[n]], axis=1).reshape(2 * PB, -1)).to(dev)
             for n in ("q", "k", "v", "alpha", "beta")}
    pool2 = pool.clone()
    mid = torch.zeros_like(pool)
    o = torch.empty((2 * PB, NV * D), device=dev)
    gdn.gdn_decode_chunk2(pool, mid, inter["q"], inter["k"], inter["v"], inter["alpha"], inter["beta"], o,
                          batch=PB, nk=NK, nv=NV, d=D, state_pitch=pitch, mid_pitch=pitch)
    # two single-token calls on the same pool layout: token t's rows are every other row
    o2 = torch.empty_like(o)
    e = 4
    for t in range(2):
        gdn.gdn_decode(pool2, inter["q"].data_ptr() + t * NK * D * e, inter["k"].data_ptr() + t * NK * D * e,
                       inter["v"].data_ptr() + t * NV * D * e, inter["alpha"].data_ptr() + t * NV * e,
                       inter["beta"].data_ptr() + t * NV * e, o2.data_ptr() + t * NV * D * e,
                       batch=PB, nk=NK, nv=NV, d=D, state_pitch=pitch, qk_stride=2 * NK * D, v_stride=2 * NV * D,
                       gb_stride=2 * NV, o_stride=2 * NV * D)
        if t == 0:
            torch.cuda.synchronize()
            assert torch.equal(mid[:, :hs].view(torch.int16), pool2[:, :hs].view(torch.int16)), \
                "intermediate state differs from one gdn_decode call"
    torch.cuda.synchronize()
    assert torch.equal(pool.view(torch.int16), pool2.view(torch.int16)), "final state differs from two calls"
    assert torch.equal(o.view(torch.int32), o2.view(torch.int32)), "outputs differ from two calls"
    assert torch.count_nonzero(pool[:, hs:]).item() == 0, "slot padding of the state was written"
    assert torch.count_nonzero(mid[:, hs:]).item() == 0, "slot padding of the intermediate pool was written"
    assert torch.isfinite(pool).all().item() and torch.isfinite(o).all().item()
    for b in sample:
        ref = S0[b].copy()
        sl = slice(b, b + 1)
        o_a = oracle.decode(ref, x0["q"][sl], x0["k"][sl], x0["v"][sl], x0["alpha"][sl], x0["beta"][sl], NK)
        ref_mid = ref.copy()
        o_b = oracle.decode(ref, x1["q"][sl], x1["k"][sl], x1["v"][sl], x1["alpha"][sl], x1["beta"][sl], NK)
        got_mid = mid[b, :hs].double().cpu().numpy().reshape(1, NV, D, D)
        got_s = pool[b, :hs].double().cpu().numpy().reshape(1, NV, D, D)
        got_o = o[2 * b:2 * b + 2].double().cpu().numpy()
        assert rel_l2(got_mid, ref_mid) <= TOL_REL_L2
        assert rel_l2(got_s, ref) <= TOL_REL_L2
        assert rel_l2(got_o, np.concatenate([o_a, o_b], axis=0)) <= TOL_REL_L2


# ------------------------------------------------------------------ decode from projections

def test_conv_norm_fp32_plain():
    """fp32 state, one CTA per value head at 4 CTAs per SM, grid > 4 waves (B = 64: 3072 CTAs):
    conv_norm_d128<float, STAGED = false, NB = 4, MINB = 4, EARLY = false>; three readers per
    key-head counter, the counters left zero."""
    B = batch_past_early(4, 64)
    check_conv(run_conv(B, NK, NV, D, 4, False, seed=320, steps=2), False)


def test_conv_norm_kh_fp16_pool_256_slots():
    """The fp16 row of the benchmark: 256-slot pool, pitch 48*128*128 + 4096 halves, 4096 CTAs of
    conv_norm_kh<__half, 5> (one per (sequence, key head)).  Sample slots against the oracle composed
    from its parts; the whole conv ring against its data move (shift by one, append the token), bit for
    bit; slot padding untouched; the workspace (not used by this kernel) left zero."""
    PB, taps, seed = 256, 4, 321
    C = (2 * NK + NV) * D
    hs = NV * D * D
    pitch = hs + 4096
    dev = torch.device("cuda")
    pool = torch.zeros((PB, pitch), dtype=torch.float16, device=dev)
    pool[:, :hs].normal_(0.0, 0.02)
    sample = [0, 100, 255]
    S = {}
    for b in sample:
        s0 = gs.state_heads(seed, [b], range(NV), D, dtype=np.float16)[0]
        pool[b, :hs] = torch.from_numpy(s0.reshape(-1)).to(dev)
        S[b] = s0.astype(np.float64)[None]
    first = gs.conv_decode_inputs(seed, PB, NK, NV, D, taps, step=0)
    ring = torch.from_numpy(first["ring"].reshape(PB, -1)).to(dev)
    ring_ref = first["ring"].reshape(PB, taps, C).copy()
    w = torch.from_numpy(first["conv_w"]).to(dev)
    dt = torch.from_numpy(first["dt"]).to(dev)
    rate = torch.from_numpy(first["rate"]).to(dev)
    gn_np = gs.norm_weight(seed, D)
    gn = torch.from_numpy(gn_np).to(dev)
    ws = torch.zeros(PB * NK, dtype=torch.int32, device=dev)
    out = torch.empty((PB, NV * D), dtype=torch.int16, device=dev)
    for t in range(2):
        x = gs.conv_decode_inputs(seed, PB, NK, NV, D, taps, step=t)
        dx = {n: torch.from_numpy(x[n]).to(dev) for n in ("x", "br", "ar", "z")}
        gdn.gdn_decode_conv_norm(pool, ring, dx["x"], w, dx["br"], dx["ar"], dt, rate, dx["z"], gn, out, ws,
                                 batch=PB, nk=NK, nv=NV, d=D, taps=taps, eps=EPS, l2_eps=L2_EPS, state_pitch=pitch)
        torch.cuda.synchronize()
        got = bf16_to_f64(out.cpu().numpy()).reshape(PB, NV, D)
        for b in sample:
            y = oracle.conv_silu(ring_ref[b].copy(), x["x"][b], first["conv_w"])   # the shift is checked below
            q = oracle.l2norm_heads(y[:NK * D], D, L2_EPS)
            k = oracle.l2norm_heads(y[NK * D:2 * NK * D], D, L2_EPS)
            v = y[2 * NK * D:]
            beta, alpha = oracle.gates(x["br"][b], x["ar"][b], first["dt"], first["rate"])
            o = oracle.decode_f64(S[b], q, k, v, alpha, beta, NK)
            ref = oracle.gated_rmsnorm(o.reshape(NV, D), x["z"][b].reshape(NV, D), gn_np, EPS)
            assert rel_l2(got[b], ref) <= TOL_REL_L2, (t, b)
        # the ring's update is a pure data move for every slot
        ring_ref = np.concatenate([ring_ref[:, 1:], x["x"][:, None, :]], axis=1)
        assert np.array_equal(ring.cpu().numpy(), ring_ref.reshape(PB, -1)), t
        assert torch.count_nonzero(ws).item() == 0
    for b in sample:
        got_s = pool[b, :hs].double().cpu().numpy().reshape(1, NV, D, D)
        assert rel_l2(got_s, S[b]) <= TOL_REL_L2
    assert torch.count_nonzero(pool[:, hs:]).item() == 0, "slot padding (canary) was written"
    assert torch.isfinite(pool).all().item()
