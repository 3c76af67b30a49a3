"""GPU: calls enqueued back to back on one state, with no host synchronisation between them.

The D = 128 decode, two-token and decode-from-projections kernels on grids of a few waves, and the
general decode kernel on one-wave grids, are launched with programmatic stream serialisation: a kernel may become resident while the one before it in the stream is still
draining, asks the L2 for its state block, and waits for its predecessor's completion before it
reads or writes anything.  Every call here reads the state (and conv ring) that the call before it
wrote, and the first call reads a state that a torch copy has just written, so a wait in the wrong
place would read stale values.  Each chain is checked bit for bit against the same calls with a
device synchronisation after each one, eagerly and replayed from a CUDA graph; the decode chain
also against the fp64 oracle."""
import numpy as np
import pytest
import torch

import gdn_synth as gs
import gated_deltanet_linear_16_gb300 as gdn
import oracle
from tests.gpu_helpers import TOL_F32, TOL_REL_L2, bf16_to_f64, max_rel_err, rel_l2

pytestmark = pytest.mark.gpu
NK, NV, D = 16, 48, 128
EPS = 1e-6


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _run_three_ways(issue, bufs):
    """issue(sync) enqueues the chain; returns {mode: {name: host copy of each buffer}}."""
    res = {}
    for mode in ("synced", "back_to_back", "graph"):
        for b in bufs.values():
            b.zero_()
        torch.cuda.synchronize()
        if mode == "graph":
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                issue(False)
            for b in bufs.values():
                b.zero_()
            torch.cuda.synchronize()
            g.replay()
        else:
            issue(mode == "synced")
        torch.cuda.synchronize()
        res[mode] = {n: b.cpu().clone() for n, b in bufs.items()}
    return res


def _assert_bitwise(res):
    for mode in ("back_to_back", "graph"):
        for n, ref in res["synced"].items():
            assert torch.equal(res[mode][n].view(torch.uint8), ref.view(torch.uint8)), f"{mode}: {n} differs"


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("B,NK,NV,D", [(1, NK, NV, D), (2, NK, NV, D), (8, NK, NV, D), (32, NK, NV, D), (1, 1, 2, 4),
                                        (3, 2, 3, 40)])
def test_decode_chain(B, NK, NV, D, f16):
    """Six steps alternating the bf16-normed and raw decode; at D = 128, B = 1 and 2 take the
    all-in-registers loads and B = 8, 32 the register-batched (fp32) or staged, and staged kernels;
    D = 4 (the tiny configuration) and D = 40 take the general kernel, also launched early for
    one-wave grids."""
    T, seed = 6, 900 + B + D
    S0 = gs.state_heads(seed, range(B), range(NV), D, dtype=np.float16 if f16 else np.float32)
    xs = [gs.decode_inputs(seed, B, NK, NV, D, step=t) for t in range(T)]
    gn = _t(gs.norm_weight(seed, D))
    dx = {n: _t(np.stack([x[n] for x in xs])) for n in ("q", "k", "v", "alpha", "beta", "z")}
    src = _t(S0)
    bufs = {"state": torch.empty_like(src),
            "bf16": torch.empty((T, B, NV * D), dtype=torch.int16, device="cuda"),
            "o": torch.empty((T, B, NV * D), dtype=torch.float32, device="cuda")}

    def issue(sync):
        bufs["state"].copy_(src)                 # a plain torch kernel writes the state just before
        for t in range(T):
            a = (bufs["state"], dx["q"][t], dx["k"][t], dx["v"][t], dx["alpha"][t], dx["beta"][t])
            if t % 2 == 0:
                gdn.gdn_decode_norm(*a, dx["z"][t], gn, bufs["bf16"][t], batch=B, nk=NK, nv=NV, d=D, eps=EPS)
            else:
                gdn.gdn_decode(*a, bufs["o"][t], batch=B, nk=NK, nv=NV, d=D)
            if sync:
                torch.cuda.synchronize()

    res = _run_three_ways(issue, bufs)
    _assert_bitwise(res)

    ref = S0.astype(np.float64)
    got = res["synced"]
    gn_h = gs.norm_weight(seed, D)
    for t, x in enumerate(xs):
        o_ref = oracle.decode(ref, x["q"], x["k"], x["v"], x["alpha"], x["beta"], NK)
        if t % 2 == 0:
            out_ref = oracle.gated_rmsnorm(o_ref.reshape(B * NV, D), x["z"].reshape(B * NV, D), gn_h, EPS)
            assert rel_l2(bf16_to_f64(got["bf16"][t].numpy()).reshape(B * NV, D), out_ref) <= TOL_REL_L2
        elif f16:
            assert rel_l2(got["o"][t].numpy(), o_ref) <= TOL_REL_L2
        else:
            assert max_rel_err(got["o"][t].numpy(), o_ref) <= TOL_F32
    S = got["state"].numpy().astype(np.float64)
    if f16:
        assert rel_l2(S, ref) <= TOL_REL_L2
    else:
        assert max_rel_err(S, ref) <= TOL_F32


@pytest.mark.parametrize("f16", [False, True])
def test_mixed_chain(f16):
    """decode_norm, the two-token step, the decode from projections (workspace entry), the int8
    epilogue, the allocation-free decode from projections and a raw decode, each on the state the
    one before left; B = 32 (fp32: the per-value-head conv kernel with its last-reader counters;
    fp16: the per-key-head one)."""
    B, seed, taps = 32, 950, 4
    C = (2 * NK + NV) * D
    S0 = gs.state_heads(seed, range(B), range(NV), D, dtype=np.float16 if f16 else np.float32)
    xs = [gs.decode_inputs(seed, B, NK, NV, D, step=t) for t in range(5)]
    cv = [gs.conv_decode_inputs(seed, B, NK, NV, D, taps=taps, step=s) for s in (3, 5)]
    gn = _t(gs.norm_weight(seed, D))
    dx = {n: _t(np.stack([x[n] for x in xs])) for n in ("q", "k", "v", "alpha", "beta", "z")}
    pair = {n: _t(np.stack([xs[1][n], xs[2][n]], axis=1).reshape(2 * B, -1))     # token rows 2b + t
            for n in ("q", "k", "v", "alpha", "beta")}
    dc = [{n: _t(c[n]) for n in ("x", "conv_w", "br", "ar", "dt", "rate", "z")} for c in cv]
    src, ring0 = _t(S0), _t(cv[0]["ring"])
    bufs = {"state": torch.empty_like(src), "mid": torch.empty_like(src), "ring": torch.empty_like(ring0),
            "out0": torch.empty((B, NV * D), dtype=torch.int16, device="cuda"),
            "o2": torch.empty((2 * B, NV * D), dtype=torch.float32, device="cuda"),
            "out3": torch.empty((B, NV * D), dtype=torch.int16, device="cuda"),
            "xq4": torch.empty((B, NV * D), dtype=torch.int8, device="cuda"),
            "xs4": torch.empty((B, NV * D // 32), dtype=torch.float32, device="cuda"),
            "out5": torch.empty((B, NV * D), dtype=torch.int16, device="cuda"),
            "o6": torch.empty((B, NV * D), dtype=torch.float32, device="cuda")}
    ws = torch.zeros(B * NK, dtype=torch.int32, device="cuda")
    dims = dict(batch=B, nk=NK, nv=NV, d=D)

    def one(t):
        return (bufs["state"], dx["q"][t], dx["k"][t], dx["v"][t], dx["alpha"][t], dx["beta"][t])

    def conv(entry, c, out):
        args = (bufs["state"], bufs["ring"], c["x"], c["conv_w"], c["br"], c["ar"], c["dt"], c["rate"], c["z"], gn,
                out)
        if entry == "ws":
            gdn.gdn_decode_conv_norm(*args, ws, taps=taps, eps=EPS, **dims)
        else:
            gdn.gdn_decode_conv_norm_noalloc(*args, taps=taps, eps=EPS, **dims)

    def issue(sync):
        steps = [
            lambda: (bufs["state"].copy_(src), bufs["ring"].copy_(ring0)),
            lambda: gdn.gdn_decode_norm(*one(0), dx["z"][0], gn, bufs["out0"], eps=EPS, **dims),
            lambda: gdn.gdn_decode_chunk2(bufs["state"], bufs["mid"], pair["q"], pair["k"], pair["v"],
                                          pair["alpha"], pair["beta"], bufs["o2"], **dims),
            lambda: conv("ws", dc[0], bufs["out3"]),
            lambda: gdn.gdn_decode_norm_q8(*one(3), dx["z"][3], gn, bufs["xq4"], bufs["xs4"], eps=EPS, **dims),
            lambda: conv("noalloc", dc[1], bufs["out5"]),
            lambda: gdn.gdn_decode(*one(4), bufs["o6"], **dims),
        ]
        for s in steps:
            s()
            if sync:
                torch.cuda.synchronize()

    res = _run_three_ways(issue, bufs)
    _assert_bitwise(res)
    assert int(ws.abs().sum().item()) == 0, "workspace counters not left zero"
    got = res["synced"]
    assert torch.isfinite(got["state"].float()).all() and torch.isfinite(got["o6"]).all()
    assert not torch.equal(got["state"], src.cpu()), "the chain left the state unchanged"
