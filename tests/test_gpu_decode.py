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
    # then 100 steps of fresh bf16 tokens, every head compared at every step.
    # The oracle forms every head's prefix state (fp64, rounded to fp32) and
    # both sides start from that fp32 state; the GPU runs the 100 steps over
    # the whole batch, then the oracle replays them 8 sequences at a time.
    from fixed_state_recurrent_gb300 import inputs
    w = inputs.WORKLOADS["decode"]
    B, H, d, P, T = w.B, w.H, w.dk, w.N, w.steps
    S_or = torch.empty((B, H, d, d), dtype=torch.float32)
    z_or = torch.empty((B, H, d), dtype=torch.float32)
    draw, sub = 32, 8  # prefix drawn 32 sequences at a time, the oracle runs 8 at a time
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    for b0 in range(0, B, draw):
        pq = inputs.gaussian((draw, H, P, d), g, torch.bfloat16, device="cuda").cpu()
        pk = inputs.gaussian((draw, H, P, d), g, torch.bfloat16, device="cuda").cpu()
        pv = inputs.gaussian((draw, H, P, d), g, torch.bfloat16, device="cuda").cpu()
        for s0 in range(0, draw, sub):
            sl = slice(s0, s0 + sub)
            _, rS, rz = orc.la_recurrent(f64(pq[sl]), f64(pk[sl]), f64(pv[sl]))
            S_or[b0 + s0:b0 + s0 + sub] = torch.from_numpy(rS).float()
            z_or[b0 + s0:b0 + s0 + sub] = torch.from_numpy(rz).float()
        del pq, pk, pv
    S = S_or.cuda()
    z = z_or.cuda()
    qs, ks, vs = inputs.decode_step_inputs(B, H, d, d, T, torch.bfloat16, w.seed)
    o_gpu = torch.empty((T, B, H, d), dtype=torch.float32)
    for t in range(T):
        o_gpu[t] = la.decode_step(qs[t].cuda(), ks[t].cuda(), vs[t].cuda(), S, z).cpu()
    torch.cuda.synchronize()
    S_gpu, z_gpu = S.cpu(), z.cpu()
    # maxima over the whole tensors (every sequence, head, step and column)
    err = {"o": 0.0, "S": 0.0, "z": 0.0}
    ref = {"o": 0.0, "S": 0.0, "z": 0.0}

    def acc(name, got, want):
        assert np.all(np.isfinite(got)), name
        err[name] = max(err[name], float(np.max(np.abs(got - want))))
        ref[name] = max(ref[name], float(np.max(np.abs(want))))

    for b0 in range(0, B, sub):
        sl = slice(b0, b0 + sub)
        rS, rz = f64(S_or[sl]), f64(z_or[sl])
        for t in range(T):
            ro, rS, rz = orc.la_decode_step(f64(qs[t, sl]), f64(ks[t, sl]), f64(vs[t, sl]), rS, rz)
            acc("o", f64(o_gpu[t, sl]), ro)
        acc("S", f64(S_gpu[sl]), rS)
        acc("z", f64(z_gpu[sl]), rz)
    rel = {k_: err[k_] / ref[k_] for k_ in err}
    assert all(e <= TOL_BF16 for e in rel.values()), rel


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
