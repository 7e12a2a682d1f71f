"""GPU parity of delta_prefill against the fp64 oracle, through the C ABI,
including the pages' hand-worked delta-memory examples."""
import numpy as np
import pytest
import torch

from conftest import golden
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


def _t(x, dtype=torch.float32):
    return torch.tensor(np.asarray(x), dtype=dtype).cuda()


def test_p3_memory_collision_on_gpu(la):
    g = golden("p3_memory_collision.json")
    k = _t(g["keys"])[None, None]
    v = _t(g["values"])[None, None]
    beta = torch.ones((1, 1, 4), device="cuda")
    reads, S = la.delta_prefill(k, v, beta)
    np.testing.assert_allclose(f64(reads)[0, 0], g["delta_reads_before_write"], atol=1e-6)
    np.testing.assert_allclose(f64(S)[0, 0], np.array(g["delta_S_page_vkT"][3]).T, atol=1e-6)


def test_two_entry_memory_on_gpu(la):
    # S0 = W^T (k v^T layout), beta = 0: the reads are the page's (1,0.6), (0.6,1)
    g = golden("two_entry_memory.json")
    k = _t(g["keys"])[None, None]
    v = torch.zeros((1, 1, 2, 2), device="cuda")
    S0 = _t(np.array(g["W_vkT"]).T)[None, None].contiguous()
    reads, S = la.delta_prefill(k, v, torch.zeros((1, 1, 2), device="cuda"), S0=S0)
    np.testing.assert_allclose(f64(reads)[0, 0], [g["read_A"], g["read_B"]], atol=1e-6)
    assert torch.equal(S, S0)


def test_p1_delta_memory_on_gpu(la):
    g = golden("p1_delta_memory.json")
    key = np.array(g["key"])
    vals = np.concatenate([np.array(g["values"]), np.zeros((1, 2))])
    for beta, want in ((1.0, g["delta_beta1_read"]), (0.5, g["delta_beta_half_read"])):
        k = _t(np.stack([key] * 3))[None, None]
        reads, _ = la.delta_prefill(k, _t(vals)[None, None], torch.full((1, 1, 3), beta, device="cuda"))
        np.testing.assert_allclose(f64(reads)[0, 0, 2], want, atol=1e-6)
    for item in g["crosstalk"]:
        rho = item["rho"]
        k2 = np.array([rho, np.sqrt(1 - rho ** 2)])
        k = _t(np.stack([key, k2, key]))[None, None]
        reads, _ = la.delta_prefill(k, _t(vals)[None, None], torch.ones((1, 1, 3), device="cuda"))
        np.testing.assert_allclose(f64(reads)[0, 0, 2], item["old_key_read"], atol=1e-6)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_exact_recall_basis_keys(la, dtype):
    # basis keys are exact in bf16: beta = 1 writes, then re-reads return the
    # stored values exactly (to fp32 rounding of v - read)
    d, dv = 128, 128
    keys = torch.eye(d, dtype=dtype)
    g = torch.Generator().manual_seed(41)
    vals = torch.randn((d, dv), generator=g).to(dtype)
    k = torch.cat([keys, keys])[None, None].cuda()
    v = torch.cat([vals, torch.zeros_like(vals)])[None, None].cuda()
    beta = torch.cat([torch.ones(d), torch.zeros(d)])[None, None].cuda()
    reads, S = la.delta_prefill(k, v, beta)
    assert torch.equal(reads[0, 0, d:].cpu(), vals.float())
    assert torch.equal(S[0, 0].cpu(), vals.float())
    # over an arbitrary old memory the fp32 path overwrites exactly up to the
    # fp32 rounding of old + (new - old)
    S0 = (torch.randn((1, 1, d, dv), generator=g) * 5).cuda()
    reads, S = la.delta_prefill(k, v, beta, S0=S0)
    if dtype == torch.float32:
        assert relmax(f64(reads[0, 0, d:]), f64(vals)) < 1e-6
        assert relmax(f64(S[0, 0]), f64(vals)) < 1e-6
        return
    # the bf16 path gives the tensor cores a bf16 copy of the state: the write
    # is S0 + bf16(v - bf16(S0)), off from v by at most 2^-9 (|S0| + |v - S0|),
    # and the read rounds that state to bf16 once more, so the error is
    # bounded by 2^-8 (max|S0| + max|v|) -- here the old memory is five times
    # the values, so that bound exceeds 2% of the values' range
    bound = 2.0 ** -8 * (S0.abs().max().item() + vals.float().abs().max().item())
    assert np.abs(f64(reads[0, 0, d:]) - f64(vals)).max() <= bound
    assert np.abs(f64(S[0, 0]) - f64(vals)).max() <= bound


SMALL = [(1, 1, 1, 1, 1), (2, 3, 37, 5, 3), (1, 2, 100, 64, 64), (2, 1, 300, 128, 128),
         (1, 1, 77, 33, 128), (1, 2, 50, 128, 7), (1, 1, 65, 100, 100)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("shape", SMALL, ids=[str(s) for s in SMALL])
@pytest.mark.parametrize("with_state", [False, True], ids=["zero", "state"])
def test_delta_small(la, orc, dtype, shape, with_state):
    from fixed_state_recurrent_gb300 import inputs
    B, H, N, dk, dv = shape
    k, v, beta = inputs.delta_inputs(B, H, N, dk, dv, dtype, seed=40 + N)
    S0 = None
    if with_state:
        g = torch.Generator().manual_seed(42)
        S0 = torch.randn((B, H, dk, dv), generator=g)
    reads, S = la.delta_prefill(k.cuda(), v.cuda(), beta.cuda(),
                                S0=None if S0 is None else S0.cuda())
    rr, rS = orc.delta(f64(k), f64(v), f64(beta), S0=None if S0 is None else f64(S0))
    tol = tol_for(dtype)
    assert relmax(f64(reads), rr) <= tol
    assert relmax(f64(S), rS) <= tol


CHUNKED_N = [1, 63, 64, 65, 127, 128, 129, 200, 256, 385, 1000]


@pytest.mark.parametrize("N", CHUNKED_N)
def test_delta_chunked_ragged(la, orc, N):
    # bf16 at dk = dv = 128 runs chunkwise (64-token chunks, processed in
    # pairs): lengths that end inside a chunk, on a chunk edge and inside the
    # second chunk of a pair, with a nonzero initial state
    from fixed_state_recurrent_gb300 import inputs
    k, v, beta = inputs.delta_inputs(1, 3, N, 128, 128, torch.bfloat16, seed=500 + N)
    g = torch.Generator().manual_seed(N)
    S0 = torch.randn((1, 3, 128, 128), generator=g) * 0.5
    reads, S = la.delta_prefill(k.cuda(), v.cuda(), beta.cuda(), S0=S0.cuda())
    rr, rS = orc.delta(f64(k), f64(v), f64(beta), S0=f64(S0))
    assert relmax(f64(reads), rr) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16


@pytest.mark.parametrize("gated", [False, True], ids=["plain", "gated"])
@pytest.mark.parametrize("N", [1, 65, 129, 385, 1000])
@pytest.mark.parametrize("d", [64, 96])
def test_delta_chunked_narrow(la, orc, d, N, gated):
    # bf16 at dk = dv = 64 and 96 runs the chunkwise kernel with the columns
    # past d zero: the reads and the state match the oracle, with S_N written
    # over S0
    from fixed_state_recurrent_gb300 import inputs
    k, v, beta = inputs.delta_inputs(2, 3, N, d, d, torch.bfloat16, seed=520 + N + d)
    g = torch.Generator().manual_seed(N + d)
    S0 = torch.randn((2, 3, d, d), generator=g) * 0.5
    alpha = (0.8 + 0.2 * torch.rand((2, 3, N), generator=g)) if gated else None
    Sd = S0.cuda()
    la.delta_read_device_status()
    reads, S = la.gated_delta_prefill(k.cuda(), v.cuda(), beta.cuda(),
                                      None if alpha is None else alpha.cuda(), S0=Sd, S_N=Sd)
    rr, rS = orc.gated_delta(f64(k), f64(v), f64(beta), None if alpha is None else f64(alpha),
                             S0=f64(S0))
    assert S.data_ptr() == Sd.data_ptr()
    assert relmax(f64(reads), rr) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert la.delta_read_device_status() == 0


def test_delta_chunked_repeatable(la, orc):
    # A few blocks (three heads) leave the SMs lightly loaded, which is where
    # an ordering hole between the kernel's roles shows up; the kernel has no
    # atomics on its data path, so every run must be bitwise identical, and
    # match the oracle.
    from fixed_state_recurrent_gb300 import inputs
    N = 1000
    k, v, beta = inputs.delta_inputs(1, 3, N, 128, 128, torch.bfloat16, seed=77)
    g = torch.Generator().manual_seed(78)
    S0 = torch.randn((1, 3, 128, 128), generator=g) * 0.5
    kd, vd, bd, Sd = k.cuda(), v.cuda(), beta.cuda(), S0.cuda()
    first = la.delta_prefill(kd, vd, bd, S0=Sd)
    for _ in range(24):
        again = la.delta_prefill(kd, vd, bd, S0=Sd)
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
    rr, rS = orc.delta(f64(k), f64(v), f64(beta), S0=f64(S0))
    assert relmax(f64(first[0]), rr) <= TOL_BF16
    assert relmax(f64(first[1]), rS) <= TOL_BF16
    assert la.delta_read_device_status() == 0  # LA_OK: no wait gave up


def test_delta_bounded_wait_reports_timeout(la, orc, monkeypatch):
    # A test hook makes the chunked kernel's MMA thread wait on an mbarrier
    # that nothing completes, with a 2 ms limit: the wait gives up, every role
    # drains what it started and the launch finishes, the status word says
    # LA_ERR_TIMEOUT (reading clears it), and the context stays usable.
    from fixed_state_recurrent_gb300 import inputs
    k, v, beta = inputs.delta_inputs(1, 2, 700, 128, 128, torch.bfloat16, seed=26)
    kd, vd, bd = k.cuda(), v.cuda(), beta.cuda()
    la.delta_read_device_status()
    monkeypatch.setenv("LA_TEST_FORCE_WAIT", "1")
    monkeypatch.setenv("LA_MBAR_TIMEOUT_NS", "2000000")
    la.delta_prefill(kd, vd, bd)
    assert la.delta_read_device_status() == 4  # LA_ERR_TIMEOUT
    assert la.delta_read_device_status() == 0  # reading clears it
    monkeypatch.delenv("LA_TEST_FORCE_WAIT")
    monkeypatch.delenv("LA_MBAR_TIMEOUT_NS")
    reads, S = la.delta_prefill(kd, vd, bd)
    assert la.delta_read_device_status() == 0
    rr, rS = orc.delta(f64(k), f64(v), f64(beta))
    assert relmax(f64(reads), rr) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16


def test_delta_in_place_alias_and_zero_length(la, orc):
    from fixed_state_recurrent_gb300 import inputs
    k, v, beta = inputs.delta_inputs(1, 2, 60, 64, 64, torch.bfloat16, seed=43)
    g = torch.Generator().manual_seed(44)
    S0 = torch.randn((1, 2, 64, 64), generator=g)
    Sd = S0.clone().cuda()
    reads, S = la.delta_prefill(k.cuda(), v.cuda(), beta.cuda(), S0=Sd, S_N=Sd)
    rr, rS = orc.delta(f64(k), f64(v), f64(beta), S0=f64(S0))
    assert relmax(f64(Sd), rS) <= TOL_BF16 and relmax(f64(reads), rr) <= TOL_BF16
    e = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device="cuda")
    reads, S = la.delta_prefill(e, e, torch.empty((1, 2, 0), device="cuda"), S0=S0.cuda())
    assert torch.equal(S.cpu(), S0)


def test_delta_config_full(la, orc):
    # B=8 H=16 N=8192 dk=dv=128: every head, every read and the whole final
    # memory against the oracle (threaded over the heads)
    from fixed_state_recurrent_gb300 import inputs
    w = inputs.WORKLOADS["delta"]
    k, v, beta = inputs.workload_inputs(w)
    reads, S = la.delta_prefill(k.cuda(), v.cuda(), beta.cuda())
    torch.cuda.synchronize()
    rr, rS = orc.delta(f64(k), f64(v), f64(beta))
    er, eS = relmax(f64(reads), rr), relmax(f64(S), rS)
    assert er <= TOL_BF16 and eS <= TOL_BF16, (er, eS)
