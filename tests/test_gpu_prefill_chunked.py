"""GPU parity: gdn_prefill_chunked (the prefill regrouped into chunks of 64 tokens, products on the
tensor cores with operands split into two TF32 parts) against the fp64 oracle's token-sequential
prefill, at the fp32 bar (1e-4 of max |ref| for o and the final state).

Token counts straddle the chunk (1, 63, 64, 65, 130, 200: one partial chunk, exact chunks, ragged
tails); the decays cover the typical ~0.86, decays small enough that products over a chunk underflow
fp32, and exact zeros; alpha = 1, beta = 0 must leave the state bit for bit unchanged (every delta is
then exactly zero).  No call may end with a timed-out MMA wait."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_16_gb300 as gdn
from tests.gpu_helpers import TOL_F32, TOL_REL_L2, run_prefill_case

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(request, cuda_lib):
    before = gdn.gdn_device_wait_timeouts()
    yield cuda_lib
    if "timeout_path" not in request.node.name:         # the two give-up tests count their own events
        assert gdn.gdn_device_wait_timeouts() == before, "a bounded MMA wait ran out"


def check(r):
    assert r["intact"], "guard band or padding overwritten"
    assert r["state_max_rel"] <= TOL_F32, r["state_max_rel"]
    assert r["o_max_rel"] <= TOL_F32, r["o_max_rel"]


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 200])
def test_chunk_boundaries(T):
    """NV = 3 over NK = 2, random initial state."""
    check(run_prefill_case(2, 2, 3, 128, T, seed=400 + T, init="normal", chunked=True))


def test_from_zero_state_with_strides_and_pitch():
    check(run_prefill_case(2, 2, 5, 128, 97, seed=410, pad=(4, 8, 1, 3), pitch_pad=4096, chunked=True))


@pytest.mark.parametrize("pad", [(0, 0, 0, 8), (4, 8, 1, 3)])
def test_o_row_padding(pad):
    """o rows padded by 8 floats (a 16-byte multiple: the outputs leave by one tensor store per chunk,
    clipped at the sequence's end) and by 3 (plain stores); the padding must stay untouched."""
    check(run_prefill_case(3, 2, 3, 128, 150, seed=416 + pad[3], init="normal", pad=pad, chunked=True))


def test_v_rows_of_any_pitch():
    """v rows padded by one float (rows not 16-byte aligned): v is read by plain loads either way."""
    check(run_prefill_case(2, 2, 3, 128, 70, seed=417, init="normal", pad=(0, 1, 0, 0), chunked=True))


def test_long_sequence():
    check(run_prefill_case(1, 2, 4, 128, 1000, seed=411, init="normal", chunked=True))


def test_split_calls_equal_one_call():
    """Consecutive calls per sequence (70 + 59 tokens, chunk boundaries inside both) match the
    oracle's single pass."""
    check(run_prefill_case(2, 2, 3, 128, 129, seed=412, init="normal", splits=(70, 59), chunked=True))


def test_low_and_zero_decay():
    """Decays in [1e-3, 0.3] (a chunk's product underflows fp32 many times over) with exact zeros."""
    rng = np.random.default_rng(413)
    B, NV, T = 2, 3, 200
    a = rng.uniform(1e-3, 0.3, size=(B, T, NV)).astype(np.float32)
    a[:, ::7, :] = 0.0
    check(run_prefill_case(B, 2, NV, 128, T, seed=413, init="normal", alpha=a, chunked=True))


def test_alpha_one_beta_zero_leaves_state_bitwise():
    r = run_prefill_case(2, 2, 3, 128, 100, seed=414, init="normal", alpha=1.0, beta=0.0, chunked=True)
    assert r["intact"]
    assert np.array_equal(r["S_gpu"], r["S_ref"])
    assert r["o_max_rel"] <= TOL_F32


def test_many_heads():
    """B * NV = 320 CTAs (more than one per SM in turn), NV = 80 over NK = 16."""
    check(run_prefill_case(4, 16, 80, 128, 70, seed=415, init="normal", chunked=True))


@pytest.mark.parametrize("T", [1, 64, 150])
def test_f16_state(T):
    """fp16 state: widened once, carried in fp32 across the call, rounded once on store."""
    r = run_prefill_case(2, 2, 3, 128, T, seed=420 + T, init="normal", f16=True, pitch_pad=4096, chunked=True)
    assert r["intact"]
    assert r["state_rel_l2"] <= TOL_REL_L2, r["state_rel_l2"]
    assert r["state_max_rel"] <= 2.0 ** -10, r["state_max_rel"]
    assert r["o_max_rel"] <= TOL_F32, r["o_max_rel"]


@pytest.mark.parametrize("D,misalign", [(64, 0), (128, 1)])
def test_other_shapes_take_the_token_kernels(D, misalign):
    check(run_prefill_case(2, 2, 3, D, 40, seed=430 + D, init="normal", misalign=misalign,
                           pad=(1 if misalign else 0, 0, 0, 0), chunked=True))


def test_matches_token_kernel_closely():
    """Both kernels on the same inputs: far inside the bar of each other."""
    a = run_prefill_case(2, 2, 3, 128, 150, seed=440, init="normal", chunked=True)
    b = run_prefill_case(2, 2, 3, 128, 150, seed=440, init="normal", chunked=False)
    scale = np.max(np.abs(a["S_ref"]))
    assert np.max(np.abs(a["S_gpu"] - b["S_gpu"])) <= TOL_F32 * scale


def test_wait_timeout_path_reports_and_leaves_the_context_usable():
    """With the poll bound at 0 every CTA's first wait (for its k, q tensor copies) gives up at once:
    the kernel lets its copies finish, writes NaN to its state and counts one event per CTA; nothing
    faults, and with the default bound restored the next call is correct again."""
    B, NK, NV, D, T = 1, 2, 3, 128, 70
    before = gdn.gdn_device_wait_timeouts()
    dev = torch.device("cuda")
    S = torch.zeros((B, NV, D, D), device=dev)
    q = torch.nn.functional.normalize(torch.randn((B * T, NK, D), device=dev), dim=-1).reshape(B * T, NK * D)
    k = torch.nn.functional.normalize(torch.randn((B * T, NK, D), device=dev), dim=-1).reshape(B * T, NK * D)
    v = torch.randn((B * T, NV * D), device=dev)
    a = torch.full((B * T, NV), 0.9, device=dev)
    b = torch.full((B * T, NV), 0.5, device=dev)
    o = torch.zeros((B * T, NV * D), device=dev)
    try:
        gdn.gdn_set_wait_polls(0)
        gdn.gdn_prefill_chunked(S, q, k, v, a, b, o, batch=B, seq_len=T, nk=NK, nv=NV, d=D)
        torch.cuda.synchronize()
    finally:
        gdn.gdn_set_wait_polls(gdn.GDN_DEFAULT_WAIT_POLLS)
    assert gdn.gdn_device_wait_timeouts() == before + B * NV
    assert torch.isnan(S).all().item()
    r = run_prefill_case(2, 2, 3, 128, 65, seed=450, init="normal", chunked=True)
    check(r)
    assert gdn.gdn_device_wait_timeouts() == before + B * NV


def test_mma_wait_timeout_path_drains_the_mmas_in_flight():
    """With only the MMA waits bounded at 0 the k, q copies are awaited normally and the first wait to
    give up is the one for G (MMA-1's G and Y in flight): the kernel lets them finish before it frees
    tensor memory, writes NaN to its state and counts one event per CTA; nothing faults, and with the
    default bound restored the next call is correct again."""
    B, NK, NV, D, T = 1, 2, 3, 128, 70
    before = gdn.gdn_device_wait_timeouts()
    dev = torch.device("cuda")
    S = torch.zeros((B, NV, D, D), device=dev)
    q = torch.nn.functional.normalize(torch.randn((B * T, NK, D), device=dev), dim=-1).reshape(B * T, NK * D)
    k = torch.nn.functional.normalize(torch.randn((B * T, NK, D), device=dev), dim=-1).reshape(B * T, NK * D)
    v = torch.randn((B * T, NV * D), device=dev)
    a = torch.full((B * T, NV), 0.9, device=dev)
    b = torch.full((B * T, NV), 0.5, device=dev)
    o = torch.zeros((B * T, NV * D), device=dev)
    try:
        gdn.gdn_set_mma_wait_polls(0)
        gdn.gdn_prefill_chunked(S, q, k, v, a, b, o, batch=B, seq_len=T, nk=NK, nv=NV, d=D)
        torch.cuda.synchronize()
    finally:
        gdn.gdn_set_wait_polls(gdn.GDN_DEFAULT_WAIT_POLLS)
    assert gdn.gdn_device_wait_timeouts() == before + B * NV
    assert torch.isnan(S).all().item()
    r = run_prefill_case(2, 2, 3, 128, 65, seed=451, init="normal", chunked=True)
    check(r)
    assert gdn.gdn_device_wait_timeouts() == before + B * NV
