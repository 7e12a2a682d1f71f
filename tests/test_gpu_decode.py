"""GPU parity of la_decode_step against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from helpers import f64, relmax, tol_for, TOL_BF16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrent_gb300 import build, api
    build.build()
    api.load()
    return api


def _steps(B, H, dk, dv, T, dtype, seed):
    from fixed_state_recurrent_gb300 import inputs
    return inputs.decode_step_inputs(B, H, dk, dv, T, dtype, seed)


def _run(la, orc, B, H, dk, dv, T, dtype, seed, S0, z0, heads=None):
    """T decode steps on the GPU from (S0, z0) fp32; the oracle runs the same
    steps in fp64 from the same fp32 state (on `heads` only, if given)."""
    qs, ks, vs = _steps(B, H, dk, dv, T, dtype, seed)
    S = S0.cuda().contiguous()
    z = z0.cuda().contiguous()
    sel = (slice(None), slice(None)) if heads is None else heads
    rS, rz = f64(S0)[sel], f64(z0)[sel]
    tol = tol_for(dtype)
    worst = 0.0
    for t in range(T):
        o = la.decode_step(qs[t].cuda(), ks[t].cuda(), vs[t].cuda(), S, z)
        ro, rS, rz = orc.la_decode_step(f64(qs[t])[sel], f64(ks[t])[sel], f64(vs[t])[sel], rS, rz)
        e = relmax(f64(o)[sel], ro)
        worst = max(worst, e)
        assert e <= tol, (t, e)
    torch.cuda.synchronize()
    assert relmax(f64(S)[sel], rS) <= tol
    assert relmax(f64(z)[sel], rz) <= tol
    return worst


SHAPES = [(1, 1, 1, 1), (2, 3, 5, 3), (4, 2, 64, 64), (2, 2, 128, 128), (1, 3, 128, 31),
          (1, 2, 17, 128)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_decode_small(la, orc, dtype, shape):
    B, H, dk, dv = shape
    g = torch.Generator().manual_seed(31)
    S0 = torch.randn((B, H, dk, dv), generator=g) * 10.0
    z0 = torch.rand((B, H, dk), generator=g) * 100.0 + 1.0
    _run(la, orc, B, H, dk, dv, 7, dtype, 32, S0, z0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_from_zero_equals_prefill(la, orc, dtype):
    # T decode steps from the zero state give the prefill of the same T tokens
    B, H, d, T = 2, 3, 64, 20
    qs, ks, vs = _steps(B, H, d, d, T, dtype, 33)
    S = torch.zeros((B, H, d, d), device="cuda")
    z = torch.zeros((B, H, d), device="cuda")
    outs = [la.decode_step(qs[t].cuda(), ks[t].cuda(), vs[t].cuda(), S, z) for t in range(T)]
    o_dec = torch.stack(outs, dim=2)
    q = qs.permute(1, 2, 0, 3).contiguous()
    k = ks.permute(1, 2, 0, 3).contiguous()
    v = vs.permute(1, 2, 0, 3).contiguous()
    o_pre, S_pre, z_pre = la.prefill(q.cuda(), k.cuda(), v.cuda())
    ro, rS, rz = orc.la_recurrent(f64(q), f64(k), f64(v))
    tol = tol_for(dtype)
    assert relmax(f64(o_dec), ro) <= tol and relmax(f64(o_pre), ro) <= tol
    assert relmax(f64(S), rS) <= tol and relmax(f64(z), rz) <= tol


def test_decode_config_full_size(la, orc):
    # B=256 H=32 dk=dv=128, state from a seeded 1024-token bf16 N(0,1) prefix,
    # then 100 steps of fresh bf16 tokens.  The oracle forms the prefix state of
    # the sampled heads (fp64, rounded to fp32); the GPU state of the other
    # heads comes from the GPU prefill, and the sampled heads get the oracle's
    # fp32 state, so both sides start every compared head from the same values.
    from fixed_state_recurrent_gb300 import inputs
    w = inputs.WORKLOADS["decode"]
    B, H, d, P = w.B, w.H, w.dk, w.N
    heads = [(0, 0), (17, 5), (100, 31), (255, 31), (128, 16), (63, 2)]
    S = torch.empty((B, H, d, d), device="cuda")
    z = torch.empty((B, H, d), device="cuda")
    S_or, z_or = {}, {}
    step = 32  # prefix drawn (seeded device generator) and prefilled 32 sequences at a time
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    for b0 in range(0, B, step):
        pq = inputs.gaussian((step, H, P, d), g, torch.bfloat16, device="cuda")
        pk = inputs.gaussian((step, H, P, d), g, torch.bfloat16, device="cuda")
        pv = inputs.gaussian((step, H, P, d), g, torch.bfloat16, device="cuda")
        la.prefill(pq, pk, pv, S_N=S[b0:b0 + step], z_N=z[b0:b0 + step])
        for (b, h) in heads:
            if b0 <= b < b0 + step:
                _, rS, rz = orc.la_recurrent(f64(pq[b - b0:b - b0 + 1, h:h + 1]),
                                             f64(pk[b - b0:b - b0 + 1, h:h + 1]),
                                             f64(pv[b - b0:b - b0 + 1, h:h + 1]))
                S_or[(b, h)] = torch.tensor(rS[0, 0], dtype=torch.float32)
                z_or[(b, h)] = torch.tensor(rz[0, 0], dtype=torch.float32)
    for bh in heads:
        S[bh] = S_or[bh].cuda()
        z[bh] = z_or[bh].cuda()
    qs, ks, vs = inputs.decode_step_inputs(B, H, d, d, w.steps, torch.bfloat16, w.seed)
    bi = np.array([b for b, _ in heads])
    hi = np.array([h for _, h in heads])
    rS = np.stack([S_or[bh].double().numpy() for bh in heads])[None]
    rz = np.stack([z_or[bh].double().numpy() for bh in heads])[None]
    worst = 0.0
    for t in range(w.steps):
        o = la.decode_step(qs[t].cuda(), ks[t].cuda(), vs[t].cuda(), S, z)
        ro, rS, rz = orc.la_decode_step(f64(qs[t])[bi, hi][None], f64(ks[t])[bi, hi][None],
                                        f64(vs[t])[bi, hi][None], rS, rz)
        worst = max(worst, relmax(f64(o)[bi, hi][None], ro))
    torch.cuda.synchronize()
    assert worst <= TOL_BF16
    assert relmax(f64(S)[bi, hi][None], rS) <= TOL_BF16
    assert relmax(f64(z)[bi, hi][None], rz) <= TOL_BF16


def test_prefill_then_decode_chain(la, orc):
    # GPU prefill of a prefix, then GPU decode steps, against the oracle's
    # recurrence over prefix + steps (all on the GPU side, no state injection)
    B, H, d, P, T = 2, 4, 128, 300, 10
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(B, H, P + T, d, d, torch.bfloat16, seed=34)
    _, S, z = la.prefill(q[:, :, :P].contiguous().cuda(), k[:, :, :P].contiguous().cuda(),
                         v[:, :, :P].contiguous().cuda())
    outs = []
    for t in range(P, P + T):
        outs.append(la.decode_step(q[:, :, t].contiguous().cuda(), k[:, :, t].contiguous().cuda(),
                                   v[:, :, t].contiguous().cuda(), S, z))
    ro, rS, rz = orc.la_recurrent(f64(q), f64(k), f64(v))
    assert relmax(f64(torch.stack(outs, dim=2)), ro[:, :, P:]) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16 and relmax(f64(z), rz) <= TOL_BF16
