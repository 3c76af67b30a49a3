"""GPU parity: gdn_decode / gdn_decode_norm (fp32 and fp16 h-state) against the fp64 oracle.

Sizes are small enough for the oracle to finish in seconds yet span several
CTAs, ragged head counts (NV not a multiple of NK), strided rows with padding,
padded slot pitches, tiny and odd D (general kernel) and D = 128 (vector
kernel), and misaligned bases that force the general kernel at D = 128."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_16_gb300 as gdn
from tests.gpu_helpers import check_decode, run_decode_case, Rows, state_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


@pytest.mark.parametrize("norm", [True, False])
def test_tiny_config_64_steps(norm):
    """Batch 1, NK = 1, NV = 2, D = 4, 64 sequential steps from a zero state."""
    r = run_decode_case(1, 1, 2, 4, 64, norm=norm, init="zero")
    check_decode(r, f16=False, norm=norm)


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("norm", [True, False])
def test_d128_vector_path(f16, norm):
    r = run_decode_case(3, 2, 5, 128, 6, f16=f16, norm=norm, seed=1)
    check_decode(r, f16=f16, norm=norm)


@pytest.mark.parametrize("f16", [False, True])
def test_d128_strided_rows_and_padded_pitch(f16):
    """Row padding on every operand (multiples of 4 floats keep the vector path) and 4096 slot padding."""
    r = run_decode_case(4, 2, 6, 128, 4, f16=f16, norm=True, seed=2, pad=(8, 4, 3, 12, 6), pitch_pad=4096)
    check_decode(r, f16=f16, norm=True)


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("norm", [True, False])
def test_d128_misaligned_takes_general_kernel(f16, norm):
    r = run_decode_case(2, 2, 3, 128, 3, f16=f16, norm=norm, seed=3, misalign=1, pad=(1, 0, 0, 0, 0))
    check_decode(r, f16=f16, norm=norm)


@pytest.mark.parametrize("D", [1, 2, 5, 31, 33, 64, 96, 127, 200, 256])
@pytest.mark.parametrize("f16", [False, True])
def test_general_kernel_any_d(D, f16):
    r = run_decode_case(2, 2, 3, D, 3, f16=f16, norm=True, seed=D)
    check_decode(r, f16=f16, norm=True)


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("B", [1, 2, 8, 32])
def test_every_load_variant(B, norm, f16):
    """NV = 48: grids of 48, 96, 384 and 1536 CTAs take the all-in-registers (48, 96),
    register-batched (fp32; fp16 is staged there) and staged loads of the D = 128 kernel."""
    r = run_decode_case(B, 16, 48, 128, 1, f16=f16, norm=norm, seed=200 + B)
    check_decode(r, f16=f16, norm=norm)


def test_many_heads_several_waves():
    """B * NV = 640 CTAs: several waves over the SMs, with NV = 40 not a multiple of NK = 16."""
    r = run_decode_case(16, 16, 40, 128, 2, f16=False, norm=True, seed=4)
    check_decode(r, f16=False, norm=True)


@pytest.mark.parametrize("f16", [False, True])
def test_alpha_one_beta_zero_leaves_state_bitwise(f16):
    """alpha = 1, beta = 0: coef = 0 and S <- fma(0, k, 1 * S) = S exactly, on both kernels."""
    for D in (128, 48):
        r = run_decode_case(2, 2, 3, D, 3, f16=f16, norm=True, seed=5, alpha=1.0, beta=0.0)
        assert r["intact"]
        assert np.array_equal(r["S_gpu"], r["S_ref"])


def test_beta_zero_is_pure_decay_on_gpu():
    """beta = 0: S_T = (prod alpha) S_0 up to fp32 rounding of the products."""
    r = run_decode_case(2, 2, 4, 128, 5, norm=False, seed=6, beta=0.0)
    check_decode(r, f16=False, norm=False)


def test_empty_batch_is_a_no_op():
    st = state_pool(1, 2, 128, False)
    before = st.raw.clone()
    q = Rows(1, 256)
    gdn.gdn_decode(st.ptr, q.ptr, q.ptr, q.ptr, q.ptr, q.ptr, Rows(1, 256).ptr, batch=0, nk=2, nv=2, d=128,
                   state_dtype=gdn.GDN_STATE_F32)
    torch.cuda.synchronize()
    assert torch.equal(before, st.raw)


def test_rejected_call_raises_and_touches_nothing():
    st = state_pool(1, 2, 128, False)
    before = st.raw.clone()
    q = Rows(1, 256)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_decode(st.ptr, q.ptr, q.ptr, q.ptr, q.ptr, q.ptr, st.ptr + 64, batch=1, nk=2, nv=2, d=128,
                       state_dtype=gdn.GDN_STATE_F32)
    assert e.value.status == 4           # output inside the state
    torch.cuda.synchronize()
    assert torch.equal(before, st.raw)


@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("B", [1, 32])
def test_outputs_in_pinned_host_memory(B, norm):
    """Outputs may live in pinned host memory, which the kernels write directly over the host link (as
    the end-to-end benchmark does): the same bits as outputs in device memory, from the same state and
    inputs.  B = 1 runs the one-wave decode_d128 (16 warps, norm finished by four warps), B = 32 the
    staged one."""
    NK, NV, D = 16, 48, 128
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(900 + B)
    st = torch.randn((B, NV, D, D), device=dev, generator=g) * 0.02
    q = torch.nn.functional.normalize(torch.randn((B, NK, D), device=dev, generator=g), dim=-1).reshape(B, NK * D)
    k = torch.nn.functional.normalize(torch.randn((B, NK, D), device=dev, generator=g), dim=-1).reshape(B, NK * D)
    v = torch.randn((B, NV * D), device=dev, generator=g)
    z = torch.randn((B, NV * D), device=dev, generator=g)
    a = torch.sigmoid(torch.randn((B, NV), device=dev, generator=g) + 2.0)
    b = torch.sigmoid(torch.randn((B, NV), device=dev, generator=g))
    gn = 1.0 + 0.1 * torch.randn(D, device=dev, generator=g)
    dt = torch.int16 if norm else torch.float32
    outs, states = [], []
    for host in (False, True):
        s = st.clone()
        out = torch.full((B, NV * D), -1, dtype=dt).pin_memory() if host else torch.full((B, NV * D), -1, dtype=dt, device=dev)
        if norm:
            gdn.gdn_decode_norm(s, q, k, v, a, b, z, gn, out, batch=B, nk=NK, nv=NV, d=D, eps=1e-6)
        else:
            gdn.gdn_decode(s, q, k, v, a, b, out, batch=B, nk=NK, nv=NV, d=D)
        torch.cuda.synchronize()
        outs.append(out.cpu())
        states.append(s)
    assert torch.equal(outs[0].view(torch.int16 if norm else torch.int32), outs[1].view(torch.int16 if norm else torch.int32))
    assert torch.equal(states[0].view(torch.int32), states[1].view(torch.int32))
    assert not torch.equal(outs[1], torch.full_like(outs[1], -1)), "nothing written"


@pytest.mark.parametrize("B", [1, 32])
def test_int8_outputs_in_pinned_host_memory(B):
    """The int8 epilogue's codes, scales and fp32 y written into pinned host memory: the same bits as
    into device memory (B = 1: one warp per group of 32 on the one-wave path; B = 32: staged)."""
    NK, NV, D = 16, 48, 128
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(950 + B)
    st = torch.randn((B, NV, D, D), device=dev, generator=g) * 0.02
    q = torch.nn.functional.normalize(torch.randn((B, NK, D), device=dev, generator=g), dim=-1).reshape(B, NK * D)
    k = torch.nn.functional.normalize(torch.randn((B, NK, D), device=dev, generator=g), dim=-1).reshape(B, NK * D)
    v = torch.randn((B, NV * D), device=dev, generator=g)
    z = torch.randn((B, NV * D), device=dev, generator=g)
    a = torch.sigmoid(torch.randn((B, NV), device=dev, generator=g) + 2.0)
    b = torch.sigmoid(torch.randn((B, NV), device=dev, generator=g))
    gn = 1.0 + 0.1 * torch.randn(D, device=dev, generator=g)
    res = []
    for host in (False, True):
        s = st.clone()
        mk = (lambda *shape, dtype: torch.full(shape, -1, dtype=dtype).pin_memory()) if host else \
             (lambda *shape, dtype: torch.full(shape, -1, dtype=dtype, device=dev))
        xq, xs, y = mk(B, NV * D, dtype=torch.int8), mk(B, NV * D // 32, dtype=torch.float32), mk(B, NV * D, dtype=torch.float32)
        gdn.gdn_decode_norm_q8(s, q, k, v, a, b, z, gn, xq, xs, y, batch=B, nk=NK, nv=NV, d=D, eps=1e-6)
        torch.cuda.synchronize()
        res.append((xq.cpu(), xs.cpu().view(torch.int32), y.cpu().view(torch.int32), s))
    for i in range(3):
        assert torch.equal(res[0][i], res[1][i])
    assert torch.equal(res[0][3].view(torch.int32), res[1][3].view(torch.int32))
    assert not torch.equal(res[1][0], torch.full_like(res[1][0], -1)), "nothing written"


@pytest.mark.parametrize("f16", [False, True])
def test_load_paths_bitwise_identical(f16):
    """The same heads (sequence 0's state and inputs) stepped inside grids of 48, 384 and 1920 CTAs: the
    one-wave path (a lane's 8 rows in one reduce-scatter), register batches (fp32) or staging (fp16),
    and staging at many waves (4 rows a group) give the same raw o and new state bit for bit, since
    every reduction keeps the butterfly's association."""
    NK, NV, D = 16, 48, 128
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    Bmax = 40
    dt = torch.float16 if f16 else torch.float32
    st = (torch.randn((Bmax, NV, D, D), device=dev, generator=g) * 0.02).to(dt)
    q = torch.nn.functional.normalize(torch.randn((Bmax, NK, D), device=dev, generator=g), dim=-1).reshape(Bmax, NK * D)
    k = torch.nn.functional.normalize(torch.randn((Bmax, NK, D), device=dev, generator=g), dim=-1).reshape(Bmax, NK * D)
    v = torch.randn((Bmax, NV * D), device=dev, generator=g)
    a = torch.sigmoid(torch.randn((Bmax, NV), device=dev, generator=g) + 2.0)
    b = torch.sigmoid(torch.randn((Bmax, NV), device=dev, generator=g))
    res = []
    for B in (1, 8, Bmax):
        s = st[:B].clone()
        o = torch.empty((B, NV * D), device=dev)
        gdn.gdn_decode(s, q[:B], k[:B], v[:B], a[:B], b[:B], o, batch=B, nk=NK, nv=NV, d=D)
        torch.cuda.synchronize()
        res.append((o[0].view(torch.int32).clone(), s[0].view(torch.int16 if f16 else torch.int32).clone()))
    for o_, s_ in res[1:]:
        assert torch.equal(o_, res[0][0]), "raw o differs between load paths"
        assert torch.equal(s_, res[0][1]), "state differs between load paths"
