"""GPU parity of la_prefill_backward against the fp64 oracle (whose gradient
is pinned to finite differences), through the C ABI."""
import numpy as np
import pytest
import torch

from helpers import f64, relmax, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrent_gb300 import build, api
    build.build()
    api.load()
    return api


SHAPES = [(1, 1, 1, 4, 3), (2, 3, 37, 5, 3), (1, 2, 100, 64, 64), (1, 2, 129, 128, 128),
          (1, 1, 77, 33, 7), (1, 2, 1500, 128, 128), (2, 2, 999, 96, 40)]


# with a workspace (the binding's default) the CUDA-core form cuts the heads
# into chunks run in parallel (and bf16 at d = 64 runs on the tensor cores);
# without one, one block per head
@pytest.mark.parametrize("ws", [None, False], ids=["ws", "nows"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("with_state", [False, True], ids=["zero", "state"])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_backward_matches_oracle(la, orc, dtype, with_state, shape, ws):
    from fixed_state_recurrent_gb300 import inputs
    B, H, N, dk, dv = shape
    q, k, v = inputs.la_inputs(B, H, N, dk, dv, dtype, seed=160 + N)
    g = torch.Generator().manual_seed(161 + N)
    dO = torch.randn((B, H, N, dv), generator=g)
    S0 = z0 = dS = dz = None
    if with_state:
        S0 = torch.rand((B, H, dk, dv), generator=g)
        z0 = torch.rand((B, H, dk), generator=g) + 0.5
        dS = torch.randn((B, H, dk, dv), generator=g)
        dz = torch.randn((B, H, dk), generator=g)
    cu = lambda t: None if t is None else t.cuda()
    got = la.prefill_backward(q.cuda(), k.cuda(), v.cuda(), dO.cuda(), S0=cu(S0), z0=cu(z0),
                              dS_N=cu(dS), dz_N=cu(dz), ws=ws)
    f = lambda t: None if t is None else f64(t)
    want = orc.la_backward(f64(q), f64(k), f64(v), f64(dO), S0=f(S0), z0=f(z0), dS_N=f(dS),
                           dz_N=f(dz))
    tol = 1e-4 if dtype == torch.float32 else tol_for(dtype)
    for name, a, b in zip(("dq", "dk", "dv", "dS0", "dz0"), got, want):
        if N == 1 and not with_state and name in ("dq", "dk"):
            # one token from a zero state: o = v w / (w + eps) with
            # w = phi(q).phi(k), so q and k enter only through eps; the exact
            # gradient is O(eps) and fp32 forms it from O(1) terms that
            # cancel.  Check it in absolute terms against that scale.
            assert np.max(np.abs(f64(a) - b)) <= 1e-5, name
            continue
        assert relmax(f64(a), b) <= tol, name


def test_backward_simt_chunked_repeatable(la):
    # the chunked CUDA-core form sums in a fixed order: bit for bit from run to run
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(1, 3, 1000, 128, 128, torch.float32, seed=170)
    dO = torch.randn((1, 3, 1000, 128), generator=torch.Generator().manual_seed(171)).cuda()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    first = la.prefill_backward(qd, kd, vd, dO)
    for _ in range(5):
        again = la.prefill_backward(qd, kd, vd, dO)
        assert all(torch.equal(a, b) for a, b in zip(first, again))


def test_backward_zero_length_passes_state_gradient(la):
    e = torch.empty((1, 2, 0, 8), device="cuda")
    dS = torch.randn((1, 2, 8, 8), device="cuda")
    dq, dk, dv, dS0, dz0 = la.prefill_backward(e, e, e, e, dS_N=dS)
    assert torch.equal(dS0, dS)
    assert torch.count_nonzero(dz0) == 0


# the tensor-core backward (bf16, dk = dv = 64): a forward and a reverse sweep
# over 128-token chunks, split over every SM when given a workspace (the
# default), one block per head without one (ws=False)
TC_N = [1, 2, 127, 128, 129, 300, 1000]
WS = [None, False]
WS_IDS = ["split", "per_head"]


def _tc_case(la, orc, B, H, N, with_state, ws, seed):
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(B, H, N, 64, 64, torch.bfloat16, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    dO = torch.randn((B, H, N, 64), generator=g)
    S0 = z0 = dS = dz = None
    if with_state:
        S0 = torch.randn((B, H, 64, 64), generator=g) * 0.5
        z0 = torch.rand((B, H, 64), generator=g) * 4 + 0.5
        dS = torch.randn((B, H, 64, 64), generator=g)
        dz = torch.randn((B, H, 64), generator=g)
    cu = lambda t: None if t is None else t.cuda()
    got = la.prefill_backward(q.cuda(), k.cuda(), v.cuda(), dO.cuda(), S0=cu(S0), z0=cu(z0),
                              dS_N=cu(dS), dz_N=cu(dz), ws=ws)
    f = lambda t: None if t is None else f64(t)
    want = orc.la_backward(f64(q), f64(k), f64(v), f64(dO), S0=f(S0), z0=f(z0), dS_N=f(dS),
                           dz_N=f(dz))
    for name, a, b in zip(("dq", "dk", "dv", "dS0", "dz0"), got, want):
        if N == 1 and not with_state and name in ("dq", "dk"):
            # one token from a zero state: the exact gradient is O(eps) (see
            # test_backward_matches_oracle), the difference of two terms of
            # size T = max|phi(k)| |v.dO| / den (dq; phi(q) for dk) that the
            # tensor cores form from bf16 operands, each term within about
            # 3 * 2^-9 of itself: checked against 2^-6 T
            phi = lambda u: np.where(u > 0, u + 1.0, np.exp(np.minimum(u, 0.0)))
            fq, fk = phi(f64(q)[:, :, 0]), phi(f64(k)[:, :, 0])   # [B, H, 64]
            vd = np.abs(np.sum(f64(v)[:, :, 0] * f64(dO)[:, :, 0], axis=-1))
            den = np.sum(fq * fk, axis=-1) + 1e-6
            other = fk if name == "dq" else fq
            T = np.max(np.abs(other).max(axis=-1) * vd / den)
            assert np.max(np.abs(f64(a) - b)) <= 2.0 ** -6 * T, name
            continue
        assert relmax(f64(a), b) <= tol_for(torch.bfloat16), name
    assert la.delta_read_device_status() == 0


@pytest.mark.parametrize("ws", WS, ids=WS_IDS)
@pytest.mark.parametrize("N", TC_N)
@pytest.mark.parametrize("with_state", [False, True], ids=["zero", "state"])
def test_backward_tc_matches_oracle(la, orc, N, with_state, ws):
    _tc_case(la, orc, 1, 3, N, with_state, ws, seed=170 + N)


# the split's pieces: several per head (long heads), runs that cross heads
# (many short heads), a ragged last chunk in each; the last shape has more
# chunks (2188) than the chunk-parallel form takes, so it runs the sweeps over
# the pieces
SPLIT_SHAPES = [(1, 2, 20000), (2, 5, 3000), (3, 40, 333), (1, 1, 40000), (1, 4, 70000)]


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=[str(s) for s in SPLIT_SHAPES])
def test_backward_tc_split_pieces_match_oracle(la, orc, shape):
    B, H, N = shape
    _tc_case(la, orc, B, H, N, True, None, seed=190 + N % 97)


@pytest.mark.parametrize("ws", WS, ids=WS_IDS)
def test_backward_tc_repeatable(la, ws):
    # no atomics and a fixed split: the same bits every call
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(2, 2, 5555, 64, 64, torch.bfloat16, seed=180)
    dO = torch.randn((2, 2, 5555, 64), generator=torch.Generator().manual_seed(181)).cuda()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    first = la.prefill_backward(qd, kd, vd, dO, ws=ws)
    for _ in range(6):
        again = la.prefill_backward(qd, kd, vd, dO, ws=ws)
        assert all(torch.equal(a, b) for a, b in zip(first, again))


def test_backward_tc_explicit_workspace(la, orc):
    # a caller-owned workspace of exactly the asked-for size, whose stale
    # contents (NaN) do not reach the outputs
    from fixed_state_recurrent_gb300 import inputs
    B, H, N = 2, 3, 2500
    q, k, v = inputs.la_inputs(B, H, N, 64, 64, torch.bfloat16, seed=184)
    dO = torch.randn((B, H, N, 64), generator=torch.Generator().manual_seed(185))
    need = la.backward_workspace_bytes(B, H, N, 64, 64)
    assert need > 0 and need % 4 == 0
    ws = torch.full((need // 4,), float("nan"), device="cuda").view(torch.uint8)
    got = la.prefill_backward(q.cuda(), k.cuda(), v.cuda(), dO.cuda(), ws=ws)
    assert la.delta_read_device_status() == 0
    want = orc.la_backward(f64(q), f64(k), f64(v), f64(dO))
    for name, a, b in zip(("dq", "dk", "dv", "dS0", "dz0"), got, want):
        assert relmax(f64(a), b) <= tol_for(torch.bfloat16), name


@pytest.mark.parametrize("ws", WS, ids=WS_IDS)
def test_backward_tc_bounded_wait_reports_timeout(la, orc, monkeypatch, ws):
    # the test hook makes the kernel's MMA issuer wait on an mbarrier that
    # nothing completes (2 ms limit): the launch finishes, the library status
    # word says LA_ERR_TIMEOUT, reading clears it, and the next call is right
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(1, 2, 400, 64, 64, torch.bfloat16, seed=182)
    dO = torch.randn((1, 2, 400, 64), generator=torch.Generator().manual_seed(183))
    qd, kd, vd, dd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    la.delta_read_device_status()
    monkeypatch.setenv("LA_TEST_FORCE_WAIT", "1")
    monkeypatch.setenv("LA_MBAR_TIMEOUT_NS", "2000000")
    la.prefill_backward(qd, kd, vd, dd, ws=ws)
    assert la.delta_read_device_status() == 4  # LA_ERR_TIMEOUT
    assert la.delta_read_device_status() == 0
    monkeypatch.delenv("LA_TEST_FORCE_WAIT")
    monkeypatch.delenv("LA_MBAR_TIMEOUT_NS")
    got = la.prefill_backward(qd, kd, vd, dd, ws=ws)
    assert la.delta_read_device_status() == 0
    want = orc.la_backward(f64(q), f64(k), f64(v), f64(dO))
    for a, b in zip(got[:3], want[:3]):
        assert relmax(f64(a), b) <= tol_for(torch.bfloat16)


@pytest.mark.parametrize("d,seed", [(64, 1), (128, 5)], ids=["d64", "d128"])
def test_backward_bench_shape_full(la, orc, d, seed):
    # B=4 H=8 N=4096, bf16 (d = 64: the chunk-parallel tensor-core form the
    # bench times; d = 128: the CUDA-core form in parallel chunks): every head
    # against the oracle
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(4, 8, 4096, d, d, torch.bfloat16, seed)
    dO = torch.randn((4, 8, 4096, d), generator=torch.Generator().manual_seed(9))
    got = la.prefill_backward(q.cuda(), k.cuda(), v.cuda(), dO.cuda())
    want = orc.la_backward(f64(q), f64(k), f64(v), f64(dO))
    for name, a, b in zip(("dq", "dk", "dv", "dS0", "dz0"), got, want):
        assert relmax(f64(a), b) <= tol_for(torch.bfloat16), name
