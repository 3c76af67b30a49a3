"""The seeded input generator: deterministic, sliceable, and drawing the stated distributions."""
import numpy as np

import gdn_synth as gs


def test_splitmix64_reference_values():
    # SplitMix64 started at state 0 (published generator; first outputs of the seed-0 stream)
    x = gs.stream_u64(np.uint64(0), 3)
    assert [int(v) for v in x] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_sliceable():
    a = gs.decode_inputs(0, 6, 2, 5, 8, layer=3, step=7)
    b = gs.decode_inputs(0, 6, 2, 5, 8, layer=3, step=7)
    for n in a:
        assert np.array_equal(a[n], b[n])
    part = gs.decode_inputs(0, 6, 2, 5, 8, layer=3, step=7, seqs=[4, 1])
    for n in a:
        assert np.array_equal(part[n], a[n][[4, 1]])
    c = gs.decode_inputs(1, 6, 2, 5, 8, layer=3, step=7)
    assert not np.array_equal(a["v"], c["v"])
    s_full = gs.state_heads(0, [0, 1, 2], [0, 1, 2, 3], 8)
    s_one = gs.state_heads(0, [2], [3], 8)
    assert np.array_equal(s_full[2, 3], s_one[0, 0])


def test_prefill_tokens_are_decode_steps():
    p = gs.prefill_inputs(0, 2, 5, 2, 3, 4)
    for t in range(5):
        d = gs.decode_inputs(0, 2, 2, 3, 4, step=t)
        for n in ("q", "k", "v", "alpha", "beta"):
            assert np.array_equal(p[n][:, t], d[n])


def test_distributions():
    x = gs.decode_inputs(0, 64, 16, 48, 128)
    qn = np.linalg.norm(x["q"].reshape(64, 16, 128).astype(np.float64), axis=-1)
    assert np.allclose(qn, 1.0, atol=1e-6)
    v = x["v"].astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
    a = x["alpha"].astype(np.float64)
    assert 0.0 < a.min() and a.max() < 1.0 and abs(a.mean() - 0.8413) < 0.01   # E[sigmoid(N(2,1))] = 0.841
    b = x["beta"].astype(np.float64)
    assert abs(b.mean() - 0.5) < 0.02
    gn = gs.norm_weight(0, 4096).astype(np.float64)
    assert abs(gn.mean() - 1.0) < 0.01 and abs(gn.std() - 0.1) < 0.01
    s = gs.state_heads(0, [0], list(range(8)), 128).astype(np.float64)
    assert abs(s.std() - 0.02) < 0.001
