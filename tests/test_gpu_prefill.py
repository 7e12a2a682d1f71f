"""GPU parity of la_prefill against the fp64 oracle, through the C ABI.

Inputs come from the seeded generators; the oracle receives the exact values
the GPU receives (bf16/fp32 widened to float64).  Tolerance: max|gpu - ref| /
max|ref| over the whole tensor, 1e-5 for fp32 inputs, 2e-2 for bf16 inputs,
applied to o and to the final S and z separately.
"""
import json
import os

import numpy as np
import pytest
import torch

from conftest import golden
from helpers import f64, relmax, tol_for, TOL_F32, TOL_BF16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrent_gb300 import build, api
    build.build()
    api.load()
    return api


def _gen(B, H, N, dk, dv, dtype, seed, scale=1.0):
    from fixed_state_recurrent_gb300 import inputs
    return inputs.la_inputs(B, H, N, dk, dv, dtype, seed, scale)


def _state(B, H, dk, dv, seed):
    g = torch.Generator().manual_seed(seed)
    S0 = torch.randn((B, H, dk, dv), generator=g) * 3.0
    z0 = torch.rand((B, H, dk), generator=g) * 20.0 + 1.0
    return S0, z0


def _check(la, orc, q, k, v, S0=None, z0=None, eps=1e-6, chunk=0):
    dev = torch.device("cuda")
    args = [x.to(dev) for x in (q, k, v)]
    S0d = S0.to(dev) if S0 is not None else None
    z0d = z0.to(dev) if z0 is not None else None
    o, S, z = la.prefill(*args, eps=eps, S0=S0d, z0=z0d, chunk=chunk)
    torch.cuda.synchronize()
    ro, rS, rz = orc.la_recurrent(f64(q), f64(k), f64(v), eps=eps,
                                  S0=None if S0 is None else f64(S0),
                                  z0=None if z0 is None else f64(z0))
    tol = tol_for(q.dtype)
    eo, eS, ez = relmax(f64(o), ro), relmax(f64(S), rS), relmax(f64(z), rz)
    assert eo <= tol and eS <= tol and ez <= tol, (eo, eS, ez, tol)
    return eo, eS, ez


def test_pr1_fp32_config(la, orc):
    # B=1 H=1 N=256 dk=dv=64, fp32 N(0,1), zero state, eps = 1e-6
    q, k, v = _gen(1, 1, 256, 64, 64, torch.float32, 7)
    _check(la, orc, q, k, v)


def test_p1_seed7_printed_run_on_gpu(la):
    g = golden("p1_seed7_run.json")
    rng = np.random.default_rng(g["seed"])
    q = torch.tensor(rng.normal(size=(8, 4)), dtype=torch.float32)[None, None].cuda()
    k = torch.tensor(rng.normal(size=(8, 4)), dtype=torch.float32)[None, None].cuda()
    v = torch.tensor(rng.normal(size=(8, 3)), dtype=torch.float32)[None, None].cuda()
    o, _, _ = la.prefill(q, k, v, eps=g["eps"])
    o = f64(o)[0, 0]
    # fp32 inputs are the float64 draw rounded once: compare at 1e-5 of max|o|
    np.testing.assert_allclose(o[:2], g["first_two_outputs"], rtol=0, atol=2e-5)
    assert abs(o.min() - g["output_min"]) < 2e-5
    assert abs(o.max() - g["output_max"]) < 2e-5


SMALL = [
    # B, H, N, dk, dv
    (1, 1, 1, 1, 1),
    (2, 3, 37, 5, 3),
    (1, 2, 100, 64, 64),
    (1, 1, 300, 128, 128),
    (2, 1, 129, 17, 128),
    (1, 1, 257, 128, 31),
    (3, 1, 64, 64, 64),
    (1, 1, 127, 64, 64),
    (1, 1, 129, 64, 64),
    (1, 2, 385, 128, 128),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("shape", SMALL, ids=[str(s) for s in SMALL])
@pytest.mark.parametrize("with_state", [False, True], ids=["zero", "state"])
def test_prefill_small_shapes(la, orc, dtype, shape, with_state):
    B, H, N, dk, dv = shape
    q, k, v = _gen(B, H, N, dk, dv, dtype, seed=100 + N)
    S0, z0 = _state(B, H, dk, dv, 5) if with_state else (None, None)
    _check(la, orc, q, k, v, S0, z0)


@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.5])
def test_prefill_eps_values(la, orc, eps):
    q, k, v = _gen(1, 2, 200, 64, 64, torch.bfloat16, seed=3)
    _check(la, orc, q, k, v, eps=eps)


def test_prefill_config_bf16_full(la, orc):
    # B=4 H=8 N=4096 dk=dv=64, bf16 N(0,1): every head against the oracle
    q, k, v = _gen(4, 8, 4096, 64, 64, torch.bfloat16, 1)
    _check(la, orc, q, k, v)


def test_long_config_full(la, orc):
    # B=1 H=16 N=65536 dk=dv=64, bf16 N(0,1)*0.5: every head, every token
    # against the oracle (threaded over the heads)
    q, k, v = _gen(1, 16, 65536, 64, 64, torch.bfloat16, 2, scale=0.5)
    _check(la, orc, q, k, v)


@pytest.mark.parametrize("d,B,H,N", [(64, 2, 5, 3000), (64, 1, 4, 51200), (128, 2, 5, 3000)],
                         ids=["prefix_d64", "three_launch_d64", "chunked_d128"])
def test_prefill_workspace_needs_only_its_status_word_zeroed(la, orc, d, B, H, N):
    # Only the 256-byte header (the status word) of a workspace must be zero
    # before its first use; the rest may hold anything (NaN here), because
    # every call writes what it reads (both d = 64 forms: the two-launch one
    # up to 1536 chunks, the three-launch one above).
    q, k, v = _gen(B, H, N, d, d, torch.bfloat16, seed=26)
    S0, z0 = _state(B, H, d, d, 27)
    need = la.prefill_workspace_bytes(B, H, N, d, d)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # all-ones bytes: NaN floats
    ws[:256] = 0
    o, S, z = la.prefill(q.cuda(), k.cuda(), v.cuda(), S0=S0.cuda(), z0=z0.cuda(), ws=ws)
    assert la.read_device_status(ws) == 0
    ro, rS, rz = orc.la_recurrent(f64(q), f64(k), f64(v), S0=f64(S0), z0=f64(z0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16 and relmax(f64(z), rz) <= TOL_BF16


@pytest.mark.parametrize("N", [16384, 16385], ids=["1536_chunks", "1548_chunks"])
def test_d64_forms_either_side_of_the_l2_limit(la, orc, N):
    # 12 heads of 16384 tokens are 1536 chunks, the most the two-launch form
    # takes; one more token per head (a one-token last chunk) takes the
    # three-launch form.  Both against the oracle, with an initial state.
    B, H, d = 1, 12, 64
    q, k, v = _gen(B, H, N, d, d, torch.bfloat16, seed=28)
    S0, z0 = _state(B, H, d, d, 29)
    o, S, z = la.prefill(q.cuda(), k.cuda(), v.cuda(), S0=S0.cuda(), z0=z0.cuda())
    ro, rS, rz = orc.la_recurrent(f64(q), f64(k), f64(v), S0=f64(S0), z0=f64(z0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16 and relmax(f64(z), rz) <= TOL_BF16


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_causality_bit_identical(la, dtype):
    # perturbing q, k, v after t0 leaves o[:t0+1] bit-identical, within and
    # across chunks (page LinearMem, section 04, future_leak_error = 0)
    B, H, N, d = 1, 2, 700, 64
    q, k, v = _gen(B, H, N, d, d, dtype, seed=9)
    base = la.prefill(q.cuda(), k.cuda(), v.cuda())[0].cpu()
    for t0 in (0, 63, 127, 128, 300, 698):
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        q2[:, :, t0 + 1:] += 1.0
        k2[:, :, t0 + 1:] -= 1.0
        v2[:, :, t0 + 1:] += 100.0
        pert = la.prefill(q2.cuda(), k2.cuda(), v2.cuda())[0].cpu()
        assert torch.equal(base[:, :, :t0 + 1], pert[:, :, :t0 + 1]), t0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_split_stream_equals_whole(la, orc, dtype):
    # prefill(N1) then prefill(N2, S0=S_N1, z0=z_N1) == prefill(N1 + N2), and
    # both against the oracle of the whole stream
    B, H, N, d = 2, 2, 1000, 64
    q, k, v = _gen(B, H, N, d, d, dtype, seed=11)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, S, z = la.prefill(qd, kd, vd)
    n1 = 333
    o1, S1, z1 = la.prefill(qd[:, :, :n1].contiguous(), kd[:, :, :n1].contiguous(),
                            vd[:, :, :n1].contiguous())
    o2, S2, z2 = la.prefill(qd[:, :, n1:].contiguous(), kd[:, :, n1:].contiguous(),
                            vd[:, :, n1:].contiguous(), S0=S1, z0=z1)
    ro, rS, rz = orc.la_recurrent(f64(q), f64(k), f64(v))
    tol = tol_for(dtype)
    assert relmax(f64(torch.cat([o1, o2], dim=2)), ro) <= tol
    assert relmax(f64(S2), rS) <= tol and relmax(f64(z2), rz) <= tol
    assert relmax(f64(o), ro) <= tol


def test_state_in_place_alias(la, orc):
    q, k, v = _gen(2, 2, 300, 64, 64, torch.bfloat16, seed=12)
    S0, z0 = _state(2, 2, 64, 64, 13)
    Sd, zd = S0.cuda(), z0.cuda()
    o, S, z = la.prefill(q.cuda(), k.cuda(), v.cuda(), S0=Sd, z0=zd, S_N=Sd, z_N=zd)
    ro, rS, rz = orc.la_recurrent(f64(q), f64(k), f64(v), S0=f64(S0), z0=f64(z0))
    assert S.data_ptr() == Sd.data_ptr()
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(Sd), rS) <= TOL_BF16 and relmax(f64(zd), rz) <= TOL_BF16


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_zero_length_copies_state(la, dtype):
    q = torch.empty((2, 3, 0, 64), dtype=dtype, device="cuda")
    v = torch.empty((2, 3, 0, 64), dtype=dtype, device="cuda")
    S0, z0 = _state(2, 3, 64, 64, 14)
    o, S, z = la.prefill(q, q, v, S0=S0.cuda(), z0=z0.cuda())
    assert o.shape == (2, 3, 0, 64)
    assert torch.equal(S.cpu(), S0) and torch.equal(z.cpu(), z0)
    o, S, z = la.prefill(q, q, v)
    assert torch.count_nonzero(S) == 0 and torch.count_nonzero(z) == 0


def test_first_step_closed_form(la):
    # o_1 = v_1 * s / (s + eps), s = phi(q_1).phi(k_1): the first output is the
    # first value, scaled by a factor within 1e-6 of one
    q, k, v = _gen(3, 4, 5, 64, 64, torch.bfloat16, seed=15)
    o = la.prefill(q.cuda(), k.cuda(), v.cuda())[0].cpu()
    assert relmax(f64(o[:, :, 0]), f64(v[:, :, 0])) < 1e-4


@pytest.mark.parametrize("shape", [(1, 1, 8192, 64), (1, 1, 5000, 128), (2, 3, 1537, 64)],
                         ids=["1head_64pieces", "1head_d128", "ragged_pieces"])
def test_few_heads_many_pieces(la, orc, shape):
    # few heads over many blocks: each head is cut into many pieces whose entry
    # states come from the scan over the earlier pieces' totals
    B, H, N, d = shape
    q, k, v = _gen(B, H, N, d, d, torch.bfloat16, seed=21)
    S0, z0 = _state(B, H, d, d, 22)
    _check(la, orc, q, k, v, S0, z0)


def test_bit_identical_across_runs(la):
    # the carry is a fixed left fold, so results do not depend on block timing
    q, k, v = _gen(2, 3, 3000, 64, 64, torch.bfloat16, seed=23)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    first = [t.clone() for t in la.prefill(qd, kd, vd)]
    for _ in range(5):
        again = la.prefill(qd, kd, vd)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


def test_device_status_clean_after_calls(la):
    q, k, v = _gen(1, 4, 2048, 64, 64, torch.bfloat16, seed=24)
    ws = la.workspace(1, 4, 2048, 64, 64, torch.bfloat16, 0, torch.device("cuda"))
    la.prefill(q.cuda(), k.cuda(), v.cuda(), ws=ws)
    assert la.read_device_status(ws) == 0  # LA_OK


# d = 64 calls of up to 1536 chunks take the two-launch form (prefix tiles,
# outputs), larger ones the three launches (aggregate, scan, outputs)
@pytest.mark.parametrize("d,H,N", [(64, 2, 1024), (64, 4, 51200), (128, 2, 1024)],
                         ids=["prefix_d64", "three_launch_d64", "chunked_d128"])
def test_bounded_wait_reports_timeout(la, orc, monkeypatch, d, H, N):
    # A test hook makes one wait of the kernel wait on something that nothing
    # completes (an mbarrier of the output kernel), with a 2 ms limit: the wait gives up,
    # the kernel drains what it started and finishes, the status word says
    # LA_ERR_TIMEOUT, and the context stays usable.
    q, k, v = _gen(1, H, N, d, d, torch.bfloat16, seed=25)
    ws = torch.zeros(la.prefill_workspace_bytes(1, H, N, d, d), dtype=torch.uint8,
                     device="cuda")
    monkeypatch.setenv("LA_TEST_FORCE_WAIT", "1")
    monkeypatch.setenv("LA_MBAR_TIMEOUT_NS", "2000000")
    la.prefill(q.cuda(), k.cuda(), v.cuda(), ws=ws)
    assert la.read_device_status(ws) == 4  # LA_ERR_TIMEOUT
    assert la.read_device_status(ws) == 0  # reading clears it
    monkeypatch.delenv("LA_TEST_FORCE_WAIT")
    monkeypatch.delenv("LA_MBAR_TIMEOUT_NS")
    o, S, z = la.prefill(q.cuda(), k.cuda(), v.cuda(), ws=ws)
    assert la.read_device_status(ws) == 0
    ro, rS, rz = orc.la_recurrent(f64(q), f64(k), f64(v))
    assert relmax(f64(o), ro) <= TOL_BF16
