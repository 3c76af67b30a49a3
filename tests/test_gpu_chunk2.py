"""GPU parity: gdn_decode_chunk2 (two tokens per launch, intermediate state kept for rollback).

Checked two ways on the same seeded inputs: against the fp64 oracle run for two
steps (intermediate state, final state, both outputs), and bit for bit against
two gdn_decode calls on the same kernel path (the contract in include/gdn.h)."""
import numpy as np
import pytest
import torch

import gdn_synth as gs
import gated_deltanet_linear_16_gb300 as gdn
import oracle
from tests.gpu_helpers import TOL_F32, TOL_REL_L2, Rows, max_rel_err, rel_l2, state_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def run(B, NK, NV, D, f16, seed, pad=(0, 0, 0, 0), pitch_pad=0, misalign=0):
    sdt = np.float16 if f16 else np.float32
    S0 = gs.state_heads(seed, range(B), range(NV), D, dtype=sdt)
    x0 = gs.decode_inputs(seed, B, NK, NV, D, step=0)
    x1 = gs.decode_inputs(seed, B, NK, NV, D, step=1)
    # token rows 2b + t
    inter = {n: np.stack([x0[n], x1[n]], axis=1).reshape(2 * B, -1) for n in ("q", "k", "v", "alpha", "beta")}
    sd = gdn.GDN_STATE_F16 if f16 else gdn.GDN_STATE_F32
    esz = 2 if f16 else 4

    pool = state_pool(B, NV, D, f16, pitch_pad, misalign)
    mid = state_pool(B, NV, D, f16, pitch_pad + 8, misalign)
    pool.write(S0.reshape(B, -1))
    bufs = {}
    for n, L, p in (("q", NK * D, pad[0]), ("k", NK * D, pad[0]), ("v", NV * D, pad[1]),
                    ("alpha", NV, pad[2]), ("beta", NV, pad[2])):
        bufs[n] = Rows(2 * B, L, L + p, misalign=misalign if n in "qk" else 0)
        bufs[n].write(inter[n])
    ob = Rows(2 * B, NV * D, NV * D + pad[3])
    gdn.gdn_decode_chunk2(pool.ptr, mid.ptr, bufs["q"].ptr, bufs["k"].ptr, bufs["v"].ptr, bufs["alpha"].ptr,
                          bufs["beta"].ptr, ob.ptr, batch=B, nk=NK, nv=NV, d=D, state_dtype=sd,
                          state_pitch=pool.stride, mid_pitch=mid.stride, qk_stride=bufs["q"].stride,
                          v_stride=bufs["v"].stride, gb_stride=bufs["alpha"].stride, o_stride=ob.stride)
    torch.cuda.synchronize()
    got = {"S": pool.read().astype(np.float64).reshape(B, NV, D, D),
           "M": mid.read().astype(np.float64).reshape(B, NV, D, D),
           "o": ob.read().astype(np.float64).reshape(B, 2, NV * D)}
    intact = all(b.intact() for b in [pool, mid, ob, *bufs.values()])

    # two single-token calls on the same path: rows of token t are every other row (stride doubled)
    pool2 = state_pool(B, NV, D, f16, pitch_pad, misalign)
    pool2.write(S0.reshape(B, -1))
    ob2 = Rows(2 * B, NV * D, NV * D + pad[3])
    mids = []
    for t in range(2):
        gdn.gdn_decode(pool2.ptr, bufs["q"].ptr + t * bufs["q"].stride * 4, bufs["k"].ptr + t * bufs["k"].stride * 4,
                       bufs["v"].ptr + t * bufs["v"].stride * 4, bufs["alpha"].ptr + t * bufs["alpha"].stride * 4,
                       bufs["beta"].ptr + t * bufs["beta"].stride * 4, ob2.ptr + t * ob2.stride * 4,
                       batch=B, nk=NK, nv=NV, d=D, state_dtype=sd, state_pitch=pool2.stride,
                       qk_stride=2 * bufs["q"].stride, v_stride=2 * bufs["v"].stride,
                       gb_stride=2 * bufs["alpha"].stride, o_stride=2 * ob2.stride)
        torch.cuda.synchronize()
        mids.append(pool2.read().copy())
    two = {"S": mids[1], "M": mids[0], "o": ob2.read()}

    ref = S0.astype(np.float64)
    o0 = oracle.decode(ref, x0["q"], x0["k"], x0["v"], x0["alpha"], x0["beta"], NK)
    ref_mid = ref.copy()
    o1 = oracle.decode(ref, x1["q"], x1["k"], x1["v"], x1["alpha"], x1["beta"], NK)
    return got, two, (ref_mid, ref, np.stack([o0, o1], axis=1)), intact, (pool, mid, ob)


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("D,misalign", [(128, 0), (128, 1), (64, 0), (5, 0)])
def test_chunk2_matches_oracle_and_two_single_steps(f16, D, misalign):
    got, two, (ref_mid, ref_S, ref_o), intact, bufs = run(3, 2, 5, D, f16, seed=31 + D, misalign=misalign,
                                                         pad=(4 if misalign == 0 else 1, 4, 1, 2), pitch_pad=64)
    assert intact, "guard band or padding overwritten"
    pool, mid, ob = bufs
    # bit for bit equal to two single-token calls on the same kernel path
    assert np.array_equal(pool.read(), two["S"])
    assert np.array_equal(mid.read(), two["M"])
    assert np.array_equal(ob.read(), two["o"])
    # against the fp64 oracle
    if f16:
        assert rel_l2(got["M"], ref_mid) <= TOL_REL_L2
        assert rel_l2(got["S"], ref_S) <= TOL_REL_L2
        assert rel_l2(got["o"], ref_o) <= TOL_REL_L2
    else:
        assert max_rel_err(got["M"], ref_mid) <= TOL_F32
        assert max_rel_err(got["S"], ref_S) <= TOL_F32
        assert max_rel_err(got["o"], ref_o) <= TOL_F32


def test_chunk2_full_layer():
    """One Qwen3.8-27B-shaped layer at batch 32: 1536 CTAs on the vector path."""
    got, two, (ref_mid, ref_S, ref_o), intact, bufs = run(32, 16, 48, 128, False, seed=33)
    assert intact
    assert np.array_equal(bufs[0].read(), two["S"]) and np.array_equal(bufs[1].read(), two["M"])
    assert max_rel_err(got["S"], ref_S) <= TOL_F32 and max_rel_err(got["o"], ref_o) <= TOL_F32
