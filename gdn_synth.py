"""Seeded synthetic inputs for the gated delta rule workloads.

This module only *draws* inputs: it holds none of the recurrence's arithmetic,
and it is the one piece of code that both the fp64 oracle (``oracle/``) and the
CUDA path (``gated_deltanet_linear_16_gb300``) are fed from, so both sides see
bit-identical inputs.

Generator
---------
Counter-based, so any slice (one sequence, one head, one token) can be drawn on
its own without drawing the rest of the tensor:

* every draw is addressed by the words ``(seed, tensor, layer, step, seq,
  head)`` plus an element index;
* the words are folded into a 64-bit key with the SplitMix64 output function
  (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014): ``key = mix(key ^ word)`` for each word in turn;
* element ``n`` of a stream is ``mix(key + (n + 1) * GAMMA)``, i.e. the n-th
  output of a SplitMix64 generator started at ``key``;
* a 64-bit output becomes a uniform in (0, 1) from its top 53 bits
  (``((x >> 11) + 0.5) * 2**-53``), and two uniforms become one standard
  normal by the Box-Muller transform, ``sqrt(-2 ln u1) * cos(2 pi u2)``,
  evaluated in fp64.

Distributions (per value head h, key head g, sequence b, step/token t), as the
workloads state them:

* q, k ~ N(0, 1), then L2-normalised per key head in fp64 (the upstream
  producer normalises q and k before the recurrence, so the recurrence sees
  unit-norm keys and queries);
* v, z ~ N(0, 1);
* alpha = sigmoid(N(2, 1)), beta = sigmoid(N(0, 1)), one value per head per
  step;
* gn = 1 + 0.1 * N(0, 1), one vector of D per layer (shared by all heads);
* initial state S0 = 0.02 * N(0, 1) (standard deviation 0.02) or zero.

Everything is rounded to fp32 at the end (state for an fp16 pool is rounded to
binary16 by numpy's own conversion).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "GAMMA", "mix64", "key_of", "stream_u64", "normals",
    "TENSOR_IDS", "decode_inputs", "prefill_inputs", "norm_weight",
    "state_heads", "head_normals", "conv_decode_inputs",
]

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# One id per drawn tensor, so streams of different tensors never coincide.
TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "z": 4, "alpha": 5, "beta": 6, "gn": 7, "state": 8,
              "x": 9, "ring": 10, "conv_w": 11, "br": 12, "ar": 13, "dt": 14, "a_log": 15}


def mix64(z):
    """SplitMix64 output function on uint64 numpy values (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def key_of(seed, *words):
    """Fold (seed, *words) into one 64-bit stream key; words may be arrays (broadcast)."""
    k = mix64(np.uint64(seed) + GAMMA)
    for w in words:
        k = mix64(k ^ np.asarray(w, dtype=np.uint64))
    return k


def stream_u64(key, n):
    """First n outputs of the SplitMix64 stream at each key: shape key.shape + (n,)."""
    key = np.asarray(key, dtype=np.uint64)
    idx = np.arange(1, n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        states = key[..., None] + idx * GAMMA
    return mix64(states)


def normals(key, n):
    """n standard normals per key (fp64), two stream outputs per normal."""
    x = stream_u64(key, 2 * n)
    u = ((x >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    u1 = u[..., 0::2]
    u2 = u[..., 1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def _sigmoid64(x):
    return 1.0 / (1.0 + np.exp(-x))


def head_normals(seed, tensor, layer, step, seqs, heads, n):
    """Normals for a (seq, head) grid: shape (len(seqs), len(heads), n)."""
    seqs = np.asarray(seqs, dtype=np.uint64)[:, None]
    heads = np.asarray(heads, dtype=np.uint64)[None, :]
    key = key_of(seed, TENSOR_IDS[tensor], layer, step, seqs, heads)
    return normals(key, n)


def _unit_rows(x):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))


def decode_inputs(seed, batch, nk, nv, d, layer=0, step=0, seqs=None):
    """One decode step's token inputs, contiguous fp32.

    Returns dict with q, k: [B][NK*D]; v, z: [B][NV*D]; alpha, beta: [B][NV].
    ``seqs`` selects which sequence indices to draw (default 0..batch-1), so a
    sample of a large batch can be drawn alone.
    """
    seqs = np.arange(batch) if seqs is None else np.asarray(seqs)
    B = len(seqs)
    kh = np.arange(nk)
    vh = np.arange(nv)
    q = _unit_rows(head_normals(seed, "q", layer, step, seqs, kh, d))
    k = _unit_rows(head_normals(seed, "k", layer, step, seqs, kh, d))
    v = head_normals(seed, "v", layer, step, seqs, vh, d)
    z = head_normals(seed, "z", layer, step, seqs, vh, d)
    a = _sigmoid64(2.0 + head_normals(seed, "alpha", layer, step, seqs, vh, 1)[..., 0])
    b = _sigmoid64(head_normals(seed, "beta", layer, step, seqs, vh, 1)[..., 0])
    f32 = np.float32
    return {
        "q": q.reshape(B, nk * d).astype(f32),
        "k": k.reshape(B, nk * d).astype(f32),
        "v": v.reshape(B, nv * d).astype(f32),
        "z": z.reshape(B, nv * d).astype(f32),
        "alpha": a.astype(f32),
        "beta": b.astype(f32),
    }


def prefill_inputs(seed, batch, seq_len, nk, nv, d, layer=0, seqs=None, t0=0):
    """Token inputs for tokens t0..t0+seq_len-1, token-major fp32.

    Returns dict with q, k: [B][T][NK*D]; v: [B][T][NV*D]; alpha, beta: [B][T][NV].
    Token t uses step index t, so a prefill over T tokens sees exactly the
    inputs of T consecutive decode steps.
    """
    seqs = np.arange(batch) if seqs is None else np.asarray(seqs)
    out = {n: [] for n in ("q", "k", "v", "alpha", "beta")}
    for t in range(t0, t0 + seq_len):
        x = decode_inputs(seed, batch, nk, nv, d, layer=layer, step=t, seqs=seqs)
        for n in out:
            out[n].append(x[n])
    return {n: np.ascontiguousarray(np.stack(v, axis=1)) for n, v in out.items()}


def norm_weight(seed, d, layer=0):
    """Gated-RMSNorm weight gn = 1 + 0.1 N(0,1): [D] fp32."""
    key = key_of(seed, TENSOR_IDS["gn"], layer)
    return (1.0 + 0.1 * normals(key, d)).astype(np.float32)


def state_heads(seed, seqs, heads, d, layer=0, std=0.02, dtype=np.float32):
    """Initial state S0 = std * N(0,1) for the given (seq, head) grid.

    Shape (len(seqs), len(heads), d, d); row a is the value index, column b the
    key index. ``dtype`` np.float16 rounds with numpy's binary16 conversion.
    """
    x = head_normals(seed, "state", layer, 0, seqs, heads, d * d) * std
    x = x.reshape(len(seqs), len(heads), d, d)
    return x.astype(dtype)


def conv_decode_inputs(seed, batch, nk, nv, d, taps=4, layer=0, step=0):
    """Inputs of the fused decode from projections (conv, L2, gates, step, norm), fp32.

    x: [B][C] projection of this token, C = 2*NK*D + NV*D laid out [q heads | k heads | v heads],
    ~ N(0,1); ring: [B][taps][C] conv state (the previous tokens' projections) ~ N(0,1);
    conv_w: [taps][C] ~ N(0, 0.5^2); br, ar: [B][NV] gate logits ~ N(0,1);
    dt: [NV] ~ N(0,1); rate: [NV] = -exp(a_log), a_log ~ N(-3, 1) (a negative decay rate, as a
    checkpoint stores it); z: [B][NV*D] ~ N(0,1).
    """
    C = 2 * nk * d + nv * d
    seqs = np.arange(batch)
    one = np.arange(1)
    x = head_normals(seed, "x", layer, step, seqs, one, C)[:, 0]
    ring = head_normals(seed, "ring", layer, step, seqs, one, taps * C)[:, 0].reshape(batch, taps, C)
    w = 0.5 * head_normals(seed, "conv_w", layer, 0, one, one, taps * C)[0, 0].reshape(taps, C)
    br = head_normals(seed, "br", layer, step, seqs, np.arange(nv), 1)[..., 0]
    ar = head_normals(seed, "ar", layer, step, seqs, np.arange(nv), 1)[..., 0]
    dt = head_normals(seed, "dt", layer, 0, one, np.arange(nv), 1)[0, :, 0]
    rate = -np.exp(head_normals(seed, "a_log", layer, 0, one, np.arange(nv), 1)[0, :, 0] - 3.0)
    z = head_normals(seed, "z", layer, step, seqs, np.arange(nv), d).reshape(batch, nv * d)
    f32 = np.float32
    return {"x": x.astype(f32), "ring": ring.astype(f32), "conv_w": w.astype(f32), "br": br.astype(f32),
            "ar": ar.astype(f32), "dt": dt.astype(f32), "rate": rate.astype(f32), "z": z.astype(f32)}
