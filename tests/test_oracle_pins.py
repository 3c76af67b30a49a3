"""Pins for the fp64 oracle, against things other than the oracle itself.

The oracle writes the gated delta rule as its matrix definition
(logicaffeine_compile/codegen_cuda/gdn.rs, kernel `gdn_step`):
    S <- alpha S + beta (v - alpha S k) k^T,   o = S q / sqrt(D)
and the gated norm as RMS-norm-then-silu-gate (same page, `gdn_gate_norm`).
None of the checks below re-types that formula.  Each one fixes the result by a
route a plausible slip would break:

* closed form of the first step from S = 0 (catches a wrong key-head pairing
  or a missing 1/sqrt(D));
* the delta-rule property along the key, S_new k = (1-beta) alpha S k + beta v
  for a unit key (catches a dropped alpha or a sign slip in the correction);
* the decay-only action off the key, S_new x = alpha S x for x orthogonal to k
  (catches a transposed outer product);
* the read-out assembled from those two by linearity;
* invariants: beta = 0 gives alpha S exactly, alpha = 1 & beta = 0 leaves S
  bit-identical, T steps of beta = 0 give (prod alpha) S;
* the textbook special case D = 1, where the rule is the scalar recurrence
  s_t = (1 - beta_t) alpha_t s_{t-1} + beta_t v_t k_t (k_t = +-1);
* the classic delta-rule overwrite (alpha = beta = 1: a second write with the
  same key replaces the value);
* the page's own alternative row form (u, w, kq, coef), in plain Python loops;
* hand-worked D = 2 steps with exact small numbers;
* the norm: RMS of the normalised output is 1, sign follows o, silu taken from
  scipy's logistic function, norm-before-gate ordering;
* binary16 conversion: the IEEE boundary table in tests/golden, numpy's own
  binary16 conversion on random bit patterns, exhaustive widening.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle

RNG = np.random.default_rng(1234)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_case(B, nk, nv, d, rng=RNG, s_scale=0.3):
    S = rng.normal(size=(B, nv, d, d)) * s_scale
    q = unit(rng.normal(size=(B, nk, d))).astype(np.float32).reshape(B, nk * d)
    k = unit(rng.normal(size=(B, nk, d))).astype(np.float32).reshape(B, nk * d)
    v = rng.normal(size=(B, nv * d)).astype(np.float32)
    a = rng.uniform(0.3, 0.99, size=(B, nv)).astype(np.float32)
    b = rng.uniform(0.05, 0.95, size=(B, nv)).astype(np.float32)
    return S, q, k, v, a, b


# ---------------------------------------------------------------- recurrence

@pytest.mark.parametrize("B,nk,nv,d", [(1, 1, 1, 1), (2, 1, 2, 4), (1, 2, 3, 5), (2, 2, 5, 8), (1, 3, 7, 16)])
def test_first_step_closed_form_from_zero(B, nk, nv, d):
    """From S = 0 one step gives S = beta v k^T and o = beta (k.q) v / sqrt(D), with g = h mod NK."""
    _, q, k, v, a, b = rand_case(B, nk, nv, d)
    S = np.zeros((B, nv, d, d))
    o = oracle.decode(S, q, k, v, a, b, nk)
    q3 = q.astype(np.float64).reshape(B, nk, d)
    k3 = k.astype(np.float64).reshape(B, nk, d)
    v3 = v.astype(np.float64).reshape(B, nv, d)
    for bb in range(B):
        for h in range(nv):
            g = h % nk      # tiled pairing stated on the page, not h // (nv // nk)
            want_S = float(b[bb, h]) * np.outer(v3[bb, h], k3[bb, g])
            want_o = float(b[bb, h]) * float(k3[bb, g] @ q3[bb, g]) * v3[bb, h] / math.sqrt(d)
            np.testing.assert_allclose(S[bb, h], want_S, rtol=0, atol=1e-15)
            np.testing.assert_allclose(o.reshape(B, nv, d)[bb, h], want_o, rtol=1e-13, atol=1e-15)


def test_key_head_pairing_is_tiled():
    """NV = 3, NK = 2: heads 0,1,2 read key heads 0,1,0 (mod), not 0,0,1 (repeat-interleave)."""
    d = 4
    q = np.zeros((1, 2 * d), np.float32)
    k = np.zeros((1, 2 * d), np.float32)
    k[0, 0] = 1.0            # key head 0 = e0
    k[0, d + 1] = 1.0        # key head 1 = e1
    q[:] = k
    v = np.ones((1, 3 * d), np.float32)
    a = np.ones((1, 3), np.float32)
    b = np.ones((1, 3), np.float32)
    S = np.zeros((1, 3, d, d))
    oracle.decode(S, q, k, v, a, b, nk=2)
    assert np.all(S[0, 0][:, 0] == 1) and np.all(S[0, 0][:, 1] == 0)
    assert np.all(S[0, 1][:, 1] == 1) and np.all(S[0, 1][:, 0] == 0)
    assert np.all(S[0, 2][:, 0] == 1) and np.all(S[0, 2][:, 1] == 0)


@pytest.mark.parametrize("d", [2, 3, 8, 17])
def test_delta_rule_along_key(d):
    """For a unit key, S_new k = (1 - beta) alpha S k + beta v (the delta rule's defining property)."""
    S, q, k, v, a, b = rand_case(3, 2, 4, d)
    S0 = S.copy()
    oracle.decode(S, q, k, v, a, b, nk=2)
    k64 = k.astype(np.float64).reshape(3, 2, d)
    k64 = unit(k64)   # fp32 rounding leaves |k| = 1 +- 1e-7; use the exact unit vector below
    for bb in range(3):
        for h in range(4):
            kk = k.astype(np.float64).reshape(3, 2, d)[bb, h % 2]
            n2 = float(kk @ kk)
            # general identity for any k: S_new k = alpha S k + beta (v - alpha S k) |k|^2
            lhs = S[bb, h] @ kk
            Sk = S0[bb, h] @ kk
            vv = v.astype(np.float64).reshape(3, 4, d)[bb, h]
            rhs = (1.0 - float(b[bb, h]) * n2) * float(a[bb, h]) * Sk + float(b[bb, h]) * n2 * vv
            np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("d", [3, 8, 16])
def test_decay_only_off_key(d):
    """For x orthogonal to k, S_new x = alpha S x: the write touches only the key direction."""
    S, q, k, v, a, b = rand_case(2, 1, 3, d)
    S0 = S.copy()
    oracle.decode(S, q, k, v, a, b, nk=1)
    for bb in range(2):
        kk = k.astype(np.float64)[bb]
        for _ in range(3):
            x = RNG.normal(size=d)
            x -= (x @ kk) / (kk @ kk) * kk
            for h in range(3):
                np.testing.assert_allclose(S[bb, h] @ x, float(a[bb, h]) * (S0[bb, h] @ x), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("d", [4, 8, 33])
def test_readout_by_linearity(d):
    """o = [ (q.k)/|k|^2 * S_new k + alpha S (q - (q.k)/|k|^2 k) ] / sqrt(D), from the two properties above."""
    S, q, k, v, a, b = rand_case(2, 2, 5, d)
    S0 = S.copy()
    o = oracle.decode(S, q, k, v, a, b, nk=2).reshape(2, 5, d)
    for bb in range(2):
        for h in range(5):
            kk = k.astype(np.float64).reshape(2, 2, d)[bb, h % 2]
            qq = q.astype(np.float64).reshape(2, 2, d)[bb, h % 2]
            vv = v.astype(np.float64).reshape(2, 5, d)[bb, h]
            n2 = kk @ kk
            c = (qq @ kk) / n2
            Sk = S0[bb, h] @ kk
            along = (1.0 - float(b[bb, h]) * n2) * float(a[bb, h]) * Sk + float(b[bb, h]) * n2 * vv   # S_new k
            off = float(a[bb, h]) * (S0[bb, h] @ (qq - c * kk))
            want = (c * along + off) / math.sqrt(d)
            np.testing.assert_allclose(o[bb, h], want, rtol=1e-11, atol=1e-13)


def test_beta_zero_is_pure_decay():
    S, q, k, v, a, b = rand_case(2, 2, 3, 6)
    b[:] = 0.0
    S0 = S.copy()
    o = oracle.decode(S, q, k, v, a, b, nk=2)
    for bb in range(2):
        for h in range(3):
            assert np.array_equal(S[bb, h], np.float64(a[bb, h]) * S0[bb, h])   # exact: alpha*S + 0
    # read-out of a pure decay: alpha S q / sqrt(D)
    q3 = q.astype(np.float64).reshape(2, 2, 6)
    for bb in range(2):
        for h in range(3):
            want = float(a[bb, h]) * (S0[bb, h] @ q3[bb, h % 2]) / math.sqrt(6)
            np.testing.assert_allclose(o.reshape(2, 3, 6)[bb, h], want, rtol=1e-12)


def test_alpha_one_beta_zero_is_identity_bitwise():
    S, q, k, v, a, b = rand_case(1, 1, 2, 7)
    a[:] = 1.0
    b[:] = 0.0
    S0 = S.copy()
    oracle.decode(S, q, k, v, a, b, nk=1)
    assert np.array_equal(S, S0)


def test_delta_rule_overwrite():
    """alpha = beta = 1, unit key, S = 0: write (k, v1) then (k, v2) -> S = v2 k^T and S k = v2."""
    d = 8
    k = np.zeros((1, d), np.float32)
    k[0, 3] = 1.0                      # exactly unit in fp32
    q = k.copy()
    v1 = RNG.normal(size=(1, d)).astype(np.float32)
    v2 = RNG.normal(size=(1, d)).astype(np.float32)
    one = np.ones((1, 1), np.float32)
    S = np.zeros((1, 1, d, d))
    oracle.decode(S, q, k, v1, one, one, nk=1)
    oracle.decode(S, q, k, v2, one, one, nk=1)
    np.testing.assert_array_equal(S[0, 0], np.outer(v2[0].astype(np.float64), k[0].astype(np.float64)))
    np.testing.assert_array_equal(S[0, 0] @ k[0].astype(np.float64), v2[0].astype(np.float64))


def test_hand_worked_d2_steps():
    """Three D = 2 steps worked by hand from the definition (see the arithmetic in the comments)."""
    d = 2
    S = np.zeros((1, 1, 2, 2))
    # step 1: S = 0, k = (1,0), q = (0.6,0.8), v = (2,-1), alpha = 0.9, beta = 0.5
    #   S1 = 0.5 * v k^T = [[1, 0], [-0.5, 0]];  o = S1 q / sqrt2 = (0.6, -0.3)/sqrt2
    o = oracle.decode(S, np.array([[0.6, 0.8]], np.float32), np.array([[1, 0]], np.float32),
                      np.array([[2, -1]], np.float32), np.array([[0.9]], np.float32),
                      np.array([[0.5]], np.float32), 1)
    np.testing.assert_allclose(S[0, 0], [[1, 0], [-0.5, 0]], atol=1e-7)
    np.testing.assert_allclose(o[0], np.array([0.6, -0.3]) / math.sqrt(2), atol=1e-7)
    # step 2: k = (0,1), q = (1,0), v = (1,1), alpha = 0.5, beta = 1
    #   S k = (0, 0); r = (1, 1); S2 = 0.5 S1 + r k^T = [[0.5, 1], [-0.25, 1]]; o = (0.5, -0.25)/sqrt2
    o = oracle.decode(S, np.array([[1, 0]], np.float32), np.array([[0, 1]], np.float32),
                      np.array([[1, 1]], np.float32), np.array([[0.5]], np.float32),
                      np.array([[1.0]], np.float32), 1)
    np.testing.assert_allclose(S[0, 0], [[0.5, 1], [-0.25, 1]], atol=1e-7)
    np.testing.assert_allclose(o[0], np.array([0.5, -0.25]) / math.sqrt(2), atol=1e-7)
    # step 3: k = (0.6,0.8), q = (0.8,-0.6), v = (0,0), alpha = 1, beta = 0.5
    #   S2 k = (1.1, 0.65); r = 0.5 * (0 - S2 k) = (-0.55, -0.325)
    #   S3 = S2 + r k^T = [[0.17, 0.56], [-0.445, 0.74]];  o = S3 q / sqrt2 = (-0.2, -0.8)/sqrt2
    o = oracle.decode(S, np.array([[0.8, -0.6]], np.float32), np.array([[0.6, 0.8]], np.float32),
                      np.array([[0, 0]], np.float32), np.array([[1.0]], np.float32),
                      np.array([[0.5]], np.float32), 1)
    np.testing.assert_allclose(S[0, 0], [[0.17, 0.56], [-0.445, 0.74]], atol=1e-6)
    np.testing.assert_allclose(o[0], np.array([-0.2, -0.8]) / math.sqrt(2), atol=1e-6)


def _page_row_form(S, q, k, v, a, b, nk):
    """The page's per-row rearrangement (gdn.rs, `gdn_step`): u = S[a].k, w = S[a].q, kq = k.q,
    coef = beta (v[a] - alpha u), o[a] = (alpha w + coef kq)/sqrt(D), S[a][b] = alpha S[a][b] + coef k[b].
    A different formula from the oracle's (read-out from the OLD state plus a kq term), plain loops."""
    B, nv, d, _ = S.shape
    o = np.zeros((B, nv * d))
    for bb in range(B):
        for h in range(nv):
            g = h % nk
            kk = [float(x) for x in k[bb, g * d:(g + 1) * d]]
            qq = [float(x) for x in q[bb, g * d:(g + 1) * d]]
            kq = sum(x * y for x, y in zip(kk, qq))
            al, be = float(a[bb, h]), float(b[bb, h])
            for r in range(d):
                row = S[bb, h, r]
                u = sum(row[c] * kk[c] for c in range(d))
                w = sum(row[c] * qq[c] for c in range(d))
                coef = be * (float(v[bb, h * d + r]) - al * u)
                o[bb, h * d + r] = (al * w + coef * kq) / math.sqrt(d)
                for c in range(d):
                    row[c] = al * row[c] + coef * kk[c]
    return o


@pytest.mark.parametrize("B,nk,nv,d", [(1, 1, 2, 4), (2, 2, 3, 5), (1, 3, 4, 9)])
def test_matches_page_row_form(B, nk, nv, d):
    S, q, k, v, a, b = rand_case(B, nk, nv, d)
    S2 = S.copy()
    for _ in range(4):
        o = oracle.decode(S, q, k, v, a, b, nk)
        o2 = _page_row_form(S2, q, k, v, a, b, nk)
        np.testing.assert_allclose(S, S2, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(o, o2, rtol=1e-11, atol=1e-14)
        _, q, k, v, a, b = rand_case(B, nk, nv, d)


# ---------------------------------------------------------------- prefill

def test_scalar_recurrence_d1():
    """D = 1: k_t = +-1 (k_t^2 = 1), so the rule is s_t = (1 - beta_t) alpha_t s_{t-1} + beta_t v_t k_t, o_t = s_t q_t."""
    T = 50
    rng = np.random.default_rng(7)
    k = np.sign(rng.normal(size=(1, T, 1))).astype(np.float32)
    q = np.sign(rng.normal(size=(1, T, 1))).astype(np.float32)
    v = rng.normal(size=(1, T, 1)).astype(np.float32)
    a = rng.uniform(0.5, 1.0, size=(1, T, 1)).astype(np.float32)
    b = rng.uniform(0.0, 1.0, size=(1, T, 1)).astype(np.float32)
    S = np.full((1, 1, 1, 1), 0.25)
    o = oracle.prefill(S, q, k, v, a, b, nk=1)
    s = 0.25
    for t in range(T):
        s = (1.0 - float(b[0, t, 0])) * float(a[0, t, 0]) * s + float(b[0, t, 0]) * float(v[0, t, 0]) * float(k[0, t, 0])
        assert o[0, t, 0] == pytest.approx(s * float(q[0, t, 0]), rel=1e-13, abs=1e-15)
    assert S[0, 0, 0, 0] == pytest.approx(s, rel=1e-13)


def test_prefill_beta_zero_is_product_of_decays():
    rng = np.random.default_rng(3)
    B, T, nk, nv, d = 2, 12, 2, 3, 5
    S = rng.normal(size=(B, nv, d, d))
    S0 = S.copy()
    q = rng.normal(size=(B, T, nk * d)).astype(np.float32)
    k = rng.normal(size=(B, T, nk * d)).astype(np.float32)
    v = rng.normal(size=(B, T, nv * d)).astype(np.float32)
    a = rng.uniform(0.5, 1.0, size=(B, T, nv)).astype(np.float32)
    b = np.zeros((B, T, nv), np.float32)
    oracle.prefill(S, q, k, v, a, b, nk)
    for bb in range(B):
        for h in range(nv):
            want = np.prod(a[bb, :, h].astype(np.float64)) * S0[bb, h]
            np.testing.assert_allclose(S[bb, h], want, rtol=1e-13)


def test_prefill_equals_steps_and_splits():
    """Prefill over T = T1 + T2 tokens equals T single steps, and two prefills of T1 and T2."""
    rng = np.random.default_rng(5)
    B, T, nk, nv, d = 2, 9, 2, 5, 6
    S = rng.normal(size=(B, nv, d, d)) * 0.1
    q = rng.normal(size=(B, T, nk * d)).astype(np.float32)
    k = unit(rng.normal(size=(B, T, nk, d))).reshape(B, T, nk * d).astype(np.float32)
    v = rng.normal(size=(B, T, nv * d)).astype(np.float32)
    a = rng.uniform(0.5, 1.0, size=(B, T, nv)).astype(np.float32)
    b = rng.uniform(0.0, 1.0, size=(B, T, nv)).astype(np.float32)
    Sa, Sb, Sc = S.copy(), S.copy(), S.copy()
    oa = oracle.prefill(Sa, q, k, v, a, b, nk)
    ob = np.stack([oracle.decode(Sb, q[:, t], k[:, t], v[:, t], a[:, t], b[:, t], nk) for t in range(T)], axis=1)
    o1 = oracle.prefill(Sc, q[:, :4], k[:, :4], v[:, :4], a[:, :4], b[:, :4], nk)
    o2 = oracle.prefill(Sc, q[:, 4:], k[:, 4:], v[:, 4:], a[:, 4:], b[:, 4:], nk)
    assert np.array_equal(Sa, Sb) and np.array_equal(oa, ob)
    assert np.array_equal(Sa, Sc) and np.array_equal(oa, np.concatenate([o1, o2], axis=1))


# ---------------------------------------------------------------- gated norm

def test_norm_rms_is_one_and_sign_follows_o():
    rng = np.random.default_rng(11)
    heads, d = 6, 32
    o = rng.normal(size=(heads, d)) * 0.3
    z = rng.normal(size=(heads, d)).astype(np.float32) * 2
    gn = (1 + 0.1 * rng.normal(size=d)).astype(np.float32)
    out = oracle.gated_rmsnorm(o, z, gn, eps=0.0)
    z64 = z.astype(np.float64)
    silu = z64 * expit(z64)                      # scipy's logistic function
    y = out / (gn.astype(np.float64) * silu)     # should be o / rms(o)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-12)
    assert np.all(np.sign(y) == np.sign(o))
    # norm then gate, NOT gate then norm: scaling one head's o leaves out unchanged (eps = 0)
    out2 = oracle.gated_rmsnorm(o * 7.5, z, gn, eps=0.0)
    np.testing.assert_allclose(out2, out, rtol=1e-12)


def test_norm_eps_and_hand_value():
    """D = 2, o = (3, 4): mean square 12.5; gn = (1, 2); z = (0, 2) -> out = (0, 2*4/sqrt(12.5+eps)*2*sigmoid(2))."""
    eps = 1e-6
    out = oracle.gated_rmsnorm(np.array([[3.0, 4.0]]), np.array([[0.0, 2.0]], np.float32),
                               np.array([1.0, 2.0], np.float32), eps)
    want1 = 2 * 4 / math.sqrt(12.5 + eps) * 2.0 / (1.0 + math.exp(-2.0))
    assert out[0, 0] == 0.0
    assert out[0, 1] == pytest.approx(want1, rel=1e-14)
    # eps dominates a tiny head: o ~ 1e-6 -> out ~ o / sqrt(eps), not o / rms(o)
    tiny = oracle.gated_rmsnorm(np.array([[1e-6, -1e-6]]), np.array([[30.0, 30.0]], np.float32),
                                np.array([1.0, 1.0], np.float32), 1e-6)
    np.testing.assert_allclose(tiny[0], np.array([1e-6, -1e-6]) / math.sqrt(1e-12 + 1e-6) * 30 * expit(30.0), rtol=1e-12)


# ---------------------------------------------------------------- converters

def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "binary16_rne.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                a, b = line.split()
                rows.append((int(a, 16), int(b, 16)))
    return rows


def test_f32_to_f16_golden_table():
    rows = _golden_rows()
    assert len(rows) >= 20
    src = np.array([r[0] for r in rows], np.uint32)
    want = np.array([r[1] for r in rows], np.uint16)
    got = oracle.f32_to_f16_bits(src)
    assert [hex(x) for x in got] == [hex(x) for x in want]


def test_f32_to_f16_matches_numpy_on_random_bits():
    rng = np.random.default_rng(99)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    # add every exponent near the binary16 range with random fractions, and exact ties
    e = rng.integers(100, 145, size=500_000).astype(np.uint32)
    fr = rng.integers(0, 2 ** 23, size=500_000).astype(np.uint32)
    near = (e << 23) | fr
    ties = (e << 23) | (fr & ~np.uint32(0x1fff)) | np.uint32(0x1000)
    bits = np.concatenate([bits, near, ties])
    f = bits.view(np.float32)
    got = oracle.f32_to_f16_bits(bits)
    with np.errstate(over="ignore"):
        want = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], want[~nan])
    g16 = got[nan]
    assert np.all(((g16 & 0x7c00) == 0x7c00) & ((g16 & 0x3ff) != 0))   # NaN stays NaN


def test_f16_to_f32_exhaustive():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32_bits(h)
    want = h.view(np.float16).astype(np.float32).view(np.uint32)
    nan = np.isnan(h.view(np.float16))
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(got[nan].view(np.float32)))
    # round trip binary16 -> binary32 -> binary16 is the identity on every non-NaN pattern
    back = oracle.f32_to_f16_bits(got)
    assert np.array_equal(back[~nan], h[~nan])


# ---------------------------------------------------------------- producers (conv, L2, gates)

def test_conv_is_causal_convolution_then_silu():
    """Fed a stream from a zero ring, the conv pre-activation is numpy's full convolution with the
    taps reversed (newest tap last), and the output is that through silu (scipy's logistic)."""
    rng = np.random.default_rng(41)
    taps, C, n = 4, 7, 12
    w = rng.normal(size=(taps, C)).astype(np.float32)
    xs = rng.normal(size=(n, C)).astype(np.float32)
    ring = np.zeros((taps, C), np.float32)
    ys = np.stack([oracle.conv_silu(ring, xs[t], w) for t in range(n)])
    for c in range(C):
        pre = np.convolve(xs[:, c].astype(np.float64), w[::-1, c].astype(np.float64))[:n]
        np.testing.assert_allclose(ys[:, c], pre * expit(pre), rtol=1e-12, atol=1e-14)
    # the ring holds the last `taps` inputs, oldest first
    np.testing.assert_array_equal(ring, xs[-taps:])


def test_conv_with_a_unit_newest_tap_is_silu_of_the_input():
    taps, C = 4, 5
    w = np.zeros((taps, C), np.float32)
    w[taps - 1] = 1.0
    ring = np.full((taps, C), 3.0, np.float32)
    x = np.array([-2.0, -0.5, 0.0, 0.5, 2.0], np.float32)
    y = oracle.conv_silu(ring, x, w)
    np.testing.assert_allclose(y, x * expit(x.astype(np.float64)), rtol=1e-14)


def test_l2norm_heads():
    rng = np.random.default_rng(42)
    y = rng.normal(size=(3, 8))
    out = oracle.l2norm_heads(y.reshape(-1), 8, 0.0).reshape(3, 8)
    np.testing.assert_allclose(np.linalg.norm(out, axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(out * np.linalg.norm(y, axis=1, keepdims=True), y, rtol=1e-13)
    # eps is added to the sum of squares: (3, 4) with eps 11 -> (3, 4) / 6
    np.testing.assert_allclose(oracle.l2norm_heads(np.array([3.0, 4.0]), 2, 11.0), [0.5, 4.0 / 6.0], rtol=1e-15)


def test_gates_closed_forms():
    rng = np.random.default_rng(43)
    n = 64
    br, ar, dt = (rng.normal(size=n).astype(np.float32) for _ in range(3))
    rate = (-np.exp(rng.normal(size=n) - 3.0)).astype(np.float32)   # negative rates, |rate| < 0.1 typical
    beta, alpha = oracle.gates(br, ar, dt, rate)
    np.testing.assert_allclose(beta, expit(br.astype(np.float64)), rtol=1e-14)
    # alpha = exp(rate * softplus(ar + dt)), softplus from numpy's logaddexp
    sp = np.logaddexp(0.0, ar.astype(np.float64) + dt.astype(np.float64))
    np.testing.assert_allclose(alpha, np.exp(rate.astype(np.float64) * sp), rtol=1e-13)
    assert np.all((alpha > 0) & (alpha < 1))
    # rate = -1, ar + dt = 0: alpha = 1/2 exactly
    b1, a1 = oracle.gates(*(np.array([v], np.float32) for v in (0.0, 0.0, 0.0, -1.0)))
    assert a1[0] == 0.5 and b1[0] == 0.5


def test_decode_f64_matches_decode_on_f32_representable_inputs():
    S, q, k, v, a, b = rand_case(2, 2, 3, 8)
    S2 = S.copy()
    o1 = oracle.decode(S, q, k, v, a, b, 2)
    o2 = oracle.decode_f64(S2, q.astype(np.float64), k.astype(np.float64), v.astype(np.float64),
                           a.astype(np.float64), b.astype(np.float64), 2)
    assert np.array_equal(S, S2) and np.array_equal(o1, o2)


# ---- int8 activation groups (gdn.rs `gdn_gate_norm_q`) -------------------------------------

def test_q8_ties_round_to_even_at_unit_scale():
    """A group whose largest magnitude is 127 has scale exactly 1, so the codes are the values
    rounded half to even: 63.5 -> 64, 0.5 -> 0, 1.5 -> 2, 2.5 -> 2, 126.5 -> 126."""
    y = np.zeros(32, np.float32)
    y[:10] = [127, 63.5, -63.5, 0.5, 1.5, 2.5, -2.5, 126.5, -0.5, 3.25]
    code, scale = oracle.quant_q8(y)
    assert scale.tolist() == [1.0]
    assert code[:10].tolist() == [127, 64, -64, 0, 2, 2, -2, 126, 0, 3]
    assert not code[10:].any()


def test_q8_scale_is_group_max_over_127():
    """Largest magnitude 254 (negative here) gives scale 2: 3 -> 1.5 -> 2, 5 -> 2.5 -> 2,
    -7 -> -3.5 -> -4, and the largest value itself maps to -127."""
    y = np.zeros(32, np.float32)
    y[:4] = [3, 5, -7, -254]
    code, scale = oracle.quant_q8(y)
    assert scale.tolist() == [2.0]
    assert code[:4].tolist() == [2, 2, -4, -127]


def test_q8_zero_group_has_unit_scale():
    code, scale = oracle.quant_q8(np.zeros(64, np.float32))
    assert scale.tolist() == [1.0, 1.0] and not code.any()


def test_q8_groups_are_32_consecutive_values():
    """Each group of 32 gets its own scale: a large value in the second group leaves the first
    group's codes alone."""
    y = np.zeros(96, np.float32)
    y[5], y[40], y[70] = 12.7, -1270.0, 0.127
    code, scale = oracle.quant_q8(y)
    assert np.allclose(scale, [0.1, 10.0, 0.001], rtol=1e-6)
    assert (code[5], code[40], code[70]) == (127, -127, 127)


def test_q8_bounds_on_random_groups():
    """Any group: |code| <= 127, the largest magnitude maps to +-127, and code * scale is within
    half a step of the value."""
    rng = np.random.default_rng(3)
    y = (rng.standard_normal(32 * 200) * rng.choice([1e-3, 1.0, 50.0], size=32 * 200)).astype(np.float32)
    code, scale = oracle.quant_q8(y)
    g = y.reshape(-1, 32).astype(np.float64)
    c = code.reshape(-1, 32).astype(np.int64)
    s = scale.astype(np.float64)[:, None]
    assert np.abs(c).max() <= 127
    top = np.argmax(np.abs(g), axis=1)
    assert np.all(np.abs(c[np.arange(len(top)), top]) == 127)
    assert np.all(np.abs(c * s - g) <= 0.5 * s * (1 + 1e-6))
