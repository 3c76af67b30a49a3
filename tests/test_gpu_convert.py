"""GPU parity: h-state converters, bit-exact against the oracle's integer IEEE rounding."""
import os

import numpy as np
import pytest
import torch

import gated_deltanet_linear_16_gb300 as gdn
import oracle

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "binary16_rne.txt")


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def f32_to_f16_gpu(bits32, offset=0):
    n = bits32.size
    src = torch.zeros(n + 16, dtype=torch.int32, device="cuda")
    src[offset:offset + n] = torch.from_numpy(bits32.view(np.int32)).cuda()
    dst = torch.full((n + 16,), 0x7DAD, dtype=torch.int16, device="cuda")
    gdn.gdn_h_f32_to_f16(src[offset:].data_ptr(), dst[offset:].data_ptr(), n)
    torch.cuda.synchronize()
    out = dst.cpu().numpy().view(np.uint16)
    assert np.all(out[:offset] == 0x7DAD) and np.all(out[offset + n:] == 0x7DAD), "guard overwritten"
    return out[offset:offset + n]


def f16_to_f32_gpu(bits16, offset=0):
    n = bits16.size
    src = torch.zeros(n + 16, dtype=torch.int16, device="cuda")
    src[offset:offset + n] = torch.from_numpy(bits16.view(np.int16)).cuda()
    dst = torch.full((n + 16,), 0x7FBADBAD, dtype=torch.int32, device="cuda")
    gdn.gdn_h_f16_to_f32(src[offset:].data_ptr(), dst[offset:].data_ptr(), n)
    torch.cuda.synchronize()
    out = dst.cpu().numpy().view(np.uint32)
    assert np.all(out[:offset] == 0x7FBADBAD) and np.all(out[offset + n:] == 0x7FBADBAD), "guard overwritten"
    return out[offset:offset + n]


def same_or_both_nan16(got, want):
    nan = ((want & 0x7C00) == 0x7C00) & ((want & 0x3FF) != 0)
    assert np.array_equal(got[~nan], want[~nan])
    g = got[nan]
    assert np.all(((g & 0x7C00) == 0x7C00) & ((g & 0x3FF) != 0))


def random_bits(n, seed):
    """n bit patterns: half uniform over all 2^32, half with exponents near the binary16 range."""
    rng = np.random.default_rng(seed)
    m = n // 2
    bits = rng.integers(0, 2 ** 32, size=n - m, dtype=np.uint64).astype(np.uint32)
    near = ((rng.integers(100, 145, size=m).astype(np.uint32) << 23) |
            rng.integers(0, 2 ** 23, size=m).astype(np.uint32))
    out = np.concatenate([bits, near])
    rng.shuffle(out)
    return out


@pytest.mark.parametrize("n,offset", [(1, 0), (7, 0), (8, 0), (1_000_003, 0), (1_000_003, 1), (4096, 3)])
def test_f32_to_f16_bit_exact(n, offset):
    bits = random_bits(n, n + offset)
    same_or_both_nan16(f32_to_f16_gpu(bits, offset), oracle.f32_to_f16_bits(bits))


def test_f32_to_f16_golden_boundaries():
    rows = [l.split("#")[0].split() for l in open(GOLDEN) if l.split("#")[0].strip()]
    src = np.array([int(a, 16) for a, _ in rows], np.uint32)
    want = np.array([int(b, 16) for _, b in rows], np.uint16)
    assert np.array_equal(f32_to_f16_gpu(src), want)


@pytest.mark.parametrize("offset", [0, 1])
def test_f16_to_f32_exhaustive(offset):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = f16_to_f32_gpu(h, offset)
    want = oracle.f16_to_f32_bits(h)
    nan = np.isnan(h.view(np.float16))
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(got[nan].view(np.float32)))


def test_round_trip_identity():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    back = f32_to_f16_gpu(f16_to_f32_gpu(h))
    nan = np.isnan(h.view(np.float16))
    assert np.array_equal(back[~nan], h[~nan])


def test_alias_rejected():
    x = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_h_f32_to_f16(x.data_ptr(), x.data_ptr() + 16, 32)
    assert e.value.status == 4
