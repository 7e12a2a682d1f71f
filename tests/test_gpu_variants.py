"""GPU parity of gated_delta_prefill and la_prefill_variant against the fp64
oracle, through the C ABI: the pages' gated-memory values, every read order
with and without decay, both input dtypes, ragged and odd sizes."""
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


# --------------------------------------------------------------------------
# gated delta

def test_p1_gated_delta_on_gpu(la):
    g = golden("p1_gated_delta.json")
    S0 = torch.tensor(g["state"], dtype=torch.float32)[None, None].cuda()
    k = torch.tensor([g["key"], g["orthogonal_key"]], dtype=torch.float32)[None, None].cuda()
    v = torch.tensor([g["value"], [0.0, 0.0]], dtype=torch.float32)[None, None].cuda()
    beta = torch.tensor([[[g["beta"], 0.0]]], dtype=torch.float32).cuda()
    for a, want in ((g["gated_alpha"], g["gated_unrelated_key_read"]),
                    (1.0, g["no_forgetting_unrelated_key_read"])):
        alpha = torch.tensor([[[a, 1.0]]], dtype=torch.float32).cuda()
        reads, S = la.gated_delta_prefill(k, v, beta, alpha, S0=S0)
        np.testing.assert_allclose(f64(reads)[0, 0, 1], want, atol=1e-7)


GD_SHAPES = [(1, 1, 1, 4, 3), (2, 3, 37, 5, 3), (1, 2, 100, 64, 64), (2, 1, 300, 128, 128),
             (1, 1, 77, 33, 128), (1, 2, 65, 100, 100)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("shape", GD_SHAPES, ids=[str(s) for s in GD_SHAPES])
def test_gated_delta_matches_oracle(la, orc, dtype, shape):
    from fixed_state_recurrent_gb300 import inputs
    B, H, N, dk, dv = shape
    k, v, beta = inputs.delta_inputs(B, H, N, dk, dv, dtype, seed=90 + N)
    g = torch.Generator().manual_seed(91 + N)
    alpha = 0.5 + 0.5 * torch.rand((B, H, N), generator=g)
    S0 = torch.randn((B, H, dk, dv), generator=g)
    reads, S = la.gated_delta_prefill(k.cuda(), v.cuda(), beta.cuda(), alpha.cuda(), S0=S0.cuda())
    rr, rS = orc.gated_delta(f64(k), f64(v), f64(beta), f64(alpha), S0=f64(S0))
    assert relmax(f64(reads), rr) <= tol_for(dtype)
    assert relmax(f64(S), rS) <= tol_for(dtype)


def test_gated_delta_without_alpha_is_delta_prefill(la):
    from fixed_state_recurrent_gb300 import inputs
    for dtype, d in ((torch.float32, 64), (torch.bfloat16, 128)):
        k, v, beta = inputs.delta_inputs(1, 2, 200, d, d, dtype, seed=93)
        a = la.gated_delta_prefill(k.cuda(), v.cuda(), beta.cuda())
        b = la.delta_prefill(k.cuda(), v.cuda(), beta.cuda())
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# --------------------------------------------------------------------------
# decayed / read-before-write / non-causal prefill

VAR_SHAPES = [(1, 1, 1, 4, 3), (2, 3, 37, 5, 3), (1, 2, 100, 64, 64), (1, 2, 129, 128, 128),
              (1, 1, 77, 33, 7)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("mode,decay", [(0, True), (1, False), (1, True), (2, False)],
                         ids=["causal_decay", "rbw", "rbw_decay", "noncausal"])
@pytest.mark.parametrize("shape", VAR_SHAPES, ids=[str(s) for s in VAR_SHAPES])
@pytest.mark.parametrize("ws", [None, False], ids=["chunks", "whole_heads"])
def test_prefill_variant_matches_oracle(la, orc, dtype, mode, decay, shape, ws):
    # with a workspace (the binding's cached scratch) the CUDA-core path runs
    # each head in parallel chunks; without one, one block walks each head
    from fixed_state_recurrent_gb300 import inputs
    B, H, N, dk, dv = shape
    q, k, v = inputs.la_inputs(B, H, N, dk, dv, dtype, seed=100 + N)
    g = torch.Generator().manual_seed(101 + N)
    alpha = (0.8 + 0.2 * torch.rand((B, H, N), generator=g)) if decay else None
    S0 = torch.rand((B, H, dk, dv), generator=g)
    z0 = torch.rand((B, H, dk), generator=g) + 0.5
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(),
                                 None if alpha is None else alpha.cuda(), mode,
                                 S0=S0.cuda(), z0=z0.cuda(), ws=ws)
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), None if alpha is None else f64(alpha),
                                mode, S0=f64(S0), z0=f64(z0))
    tol = tol_for(dtype)
    assert relmax(f64(o), ro) <= tol
    assert relmax(f64(S), rS) <= tol
    assert relmax(f64(z), rz) <= tol


def test_prefill_variant_causal_without_decay_is_la_prefill(la):
    # the fp32 path of la_prefill and the variant run the same arithmetic
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(2, 2, 90, 64, 32, torch.float32, seed=110)
    a = la.prefill_variant(q.cuda(), k.cuda(), v.cuda())
    ws = la.workspace(2, 2, 90, 64, 32, torch.float32, 0, torch.device("cuda"))
    b = la.prefill(q.cuda(), k.cuda(), v.cuda(), ws=ws)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_read_before_write_first_read_is_zero_on_gpu(la):
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(1, 3, 20, 16, 8, torch.float32, seed=111)
    o, _, _ = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), None, la.LA_MODE_READ_BEFORE_WRITE)
    assert torch.count_nonzero(o[:, :, 0]) == 0


# read before write on the tensor cores (bf16, dk = dv = 64, no decay, with a
# workspace): la_prefill's two launches with a strict mask inside each chunk;
# chunk edges, runs that cross heads and several pieces per head
RBW_SHAPES = [(1, 3, 1), (1, 3, 127), (1, 3, 128), (1, 3, 129), (1, 3, 300), (2, 5, 3000),
              (3, 40, 333), (1, 2, 20000)]


@pytest.mark.parametrize("shape", RBW_SHAPES, ids=[str(s) for s in RBW_SHAPES])
def test_read_before_write_tc_matches_oracle(la, orc, shape):
    from fixed_state_recurrent_gb300 import inputs
    B, H, N = shape
    q, k, v = inputs.la_inputs(B, H, N, 64, 64, torch.bfloat16, seed=160 + N % 89)
    g = torch.Generator().manual_seed(161 + N)
    S0 = torch.randn((B, H, 64, 64), generator=g) * 0.5
    z0 = torch.rand((B, H, 64), generator=g) * 4 + 0.5
    la.delta_read_device_status()
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), None, la.LA_MODE_READ_BEFORE_WRITE,
                                 S0=S0.cuda(), z0=z0.cuda())
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), None, 1, S0=f64(S0), z0=f64(z0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16
    assert la.delta_read_device_status() == 0


def test_read_before_write_tc_first_read_is_zero(la):
    # from a zero state the first token of each head reads nothing: exactly 0
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(2, 3, 300, 64, 64, torch.bfloat16, seed=162)
    o, _, _ = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), None, la.LA_MODE_READ_BEFORE_WRITE)
    assert torch.count_nonzero(o[:, :, 0]) == 0
    assert torch.count_nonzero(o[:, :, 1]) > 0


# non-causal on the tensor cores (bf16, dk = dv = 64, with a workspace): the
# piece totals, then every query reads its head's final state
NC_SHAPES = [(1, 3, 1), (1, 3, 129), (1, 3, 1000), (2, 5, 3000), (3, 40, 333), (1, 2, 20000)]


@pytest.mark.parametrize("shape", NC_SHAPES, ids=[str(s) for s in NC_SHAPES])
def test_noncausal_tc_matches_oracle(la, orc, shape):
    from fixed_state_recurrent_gb300 import inputs
    B, H, N = shape
    q, k, v = inputs.la_inputs(B, H, N, 64, 64, torch.bfloat16, seed=170 + N % 83)
    g = torch.Generator().manual_seed(171 + N)
    S0 = torch.randn((B, H, 64, 64), generator=g) * 0.5
    z0 = torch.rand((B, H, 64), generator=g) * 4 + 0.5
    la.delta_read_device_status()
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), None, la.LA_MODE_NONCAUSAL,
                                 S0=S0.cuda(), z0=z0.cuda())
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), None, 2, S0=f64(S0), z0=f64(z0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16
    assert la.delta_read_device_status() == 0


# the other tensor-core forms of the two read orders: d = 128 (the three-launch
# prefill with a strict mask; the aggregate launch, then the reads of the final
# state), and d = 64 past 2048 chunks (the same at d = 64)
WIDE_SHAPES = [(128, 1, 3, 1), (128, 1, 3, 129), (128, 1, 3, 300), (128, 2, 5, 3000),
               (128, 3, 40, 333), (128, 1, 2, 20000), (64, 1, 4, 70000)]


@pytest.mark.parametrize("mode", [1, 2], ids=["rbw", "nc"])
@pytest.mark.parametrize("shape", WIDE_SHAPES, ids=[str(s) for s in WIDE_SHAPES])
def test_read_orders_tc_wide_match_oracle(la, orc, shape, mode):
    from fixed_state_recurrent_gb300 import inputs
    d, B, H, N = shape
    q, k, v = inputs.la_inputs(B, H, N, d, d, torch.bfloat16, seed=180 + N % 79 + mode)
    g = torch.Generator().manual_seed(181 + N + d)
    S0 = torch.randn((B, H, d, d), generator=g) * 0.5
    z0 = torch.rand((B, H, d), generator=g) * 4 + 0.5
    la.delta_read_device_status()
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), None, mode, S0=S0.cuda(), z0=z0.cuda())
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), None, mode, S0=f64(S0), z0=f64(z0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16
    assert la.delta_read_device_status() == 0


@pytest.mark.parametrize("mode", [1, 2], ids=["rbw", "nc"])
@pytest.mark.parametrize("d,N", [(128, 3000), (64, 70000)], ids=["d128", "d64_long"])
def test_read_orders_tc_wide_state_in_place(la, orc, d, N, mode):
    # S_N, z_N written over S0, z0: every block of a head reads S0 while one of
    # them writes S_N
    from fixed_state_recurrent_gb300 import inputs
    B, H = 1, 4
    q, k, v = inputs.la_inputs(B, H, N, d, d, torch.bfloat16, seed=185 + mode)
    g = torch.Generator().manual_seed(186 + d)
    S0 = torch.randn((B, H, d, d), generator=g) * 0.5
    z0 = torch.rand((B, H, d), generator=g) * 4 + 0.5
    Sd, zd = S0.cuda(), z0.cuda()
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), None, mode, S0=Sd, z0=zd,
                                 S_N=Sd, z_N=zd)
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), None, mode, S0=f64(S0), z0=f64(z0))
    assert S.data_ptr() == Sd.data_ptr() and z.data_ptr() == zd.data_ptr()
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16


@pytest.mark.parametrize("d,N", [(64, 1000), (128, 1000)], ids=["d64", "d128"])
def test_noncausal_tc_bounded_wait_reports_timeout(la, orc, monkeypatch, d, N):
    # the test hook makes the reads' first product wait on an mbarrier that
    # nothing completes (2 ms limit): the launch finishes, the library status
    # word says LA_ERR_TIMEOUT, reading clears it, and the next call is right
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(1, 2, N, d, d, torch.bfloat16, seed=188)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    la.delta_read_device_status()
    monkeypatch.setenv("LA_TEST_FORCE_WAIT", "1")
    monkeypatch.setenv("LA_MBAR_TIMEOUT_NS", "2000000")
    la.prefill_variant(qd, kd, vd, None, la.LA_MODE_NONCAUSAL)
    assert la.delta_read_device_status() == 4  # LA_ERR_TIMEOUT
    assert la.delta_read_device_status() == 0
    monkeypatch.delenv("LA_TEST_FORCE_WAIT")
    monkeypatch.delenv("LA_MBAR_TIMEOUT_NS")
    o, S, z = la.prefill_variant(qd, kd, vd, None, la.LA_MODE_NONCAUSAL)
    assert la.delta_read_device_status() == 0
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), None, 2)
    assert relmax(f64(o), ro) <= TOL_BF16


def test_read_before_write_tc_wide_first_read_is_zero(la):
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(2, 3, 300, 128, 128, torch.bfloat16, seed=187)
    o, _, _ = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), None, la.LA_MODE_READ_BEFORE_WRITE)
    assert torch.count_nonzero(o[:, :, 0]) == 0
    assert torch.count_nonzero(o[:, :, 1]) > 0


def test_noncausal_tc_queries_read_one_state(la):
    # every query of a head reads the same state: two equal queries far apart in
    # the sequence (other chunks, other blocks) give the same output
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(1, 2, 700, 64, 64, torch.bfloat16, seed=172)
    q[:, :, 650] = q[:, :, 3]
    o, _, _ = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), None, la.LA_MODE_NONCAUSAL)
    a, b = o[:, :, 650], o[:, :, 3]
    assert (a - b).abs().max().item() <= 1e-6 * b.abs().max().item()


def test_prefill_variant_zero_length_copies_state(la):
    e = torch.empty((1, 2, 0, 8), device="cuda")
    S0 = torch.rand((1, 2, 8, 8), device="cuda")
    z0 = torch.rand((1, 2, 8), device="cuda")
    o, S, z = la.prefill_variant(e, e, e, torch.empty((1, 2, 0), device="cuda"), 0, S0=S0, z0=z0)
    assert torch.equal(S, S0) and torch.equal(z, z0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mode,decay", [(0, True), (1, False), (1, True), (2, False)],
                         ids=["causal_decay", "rbw", "rbw_decay", "nc"])
def test_prefill_variant_tc_zero_length_copies_state(la, d, mode, decay):
    # bf16 at the tensor-core widths, every order: no tokens, the state passes through
    e = torch.empty((1, 2, 0, d), dtype=torch.bfloat16, device="cuda")
    S0 = torch.rand((1, 2, d, d), device="cuda")
    z0 = torch.rand((1, 2, d), device="cuda")
    alpha = torch.empty((1, 2, 0), device="cuda") if decay else None
    o, S, z = la.prefill_variant(e, e, e, alpha, mode, S0=S0, z0=z0)
    assert torch.equal(S, S0) and torch.equal(z, z0)


# gated delta on the tensor cores (bf16, dk = dv = 128): chunkwise with decay factors
GATED_N = [1, 64, 65, 129, 300, 1000]


@pytest.mark.parametrize("N", GATED_N)
@pytest.mark.parametrize("arange", [(0.9, 1.0), (0.3, 1.0), (0.02, 0.5)], ids=["mild", "strong", "severe"])
def test_gated_delta_chunked_matches_oracle(la, orc, N, arange):
    from fixed_state_recurrent_gb300 import inputs
    k, v, beta = inputs.delta_inputs(1, 3, N, 128, 128, torch.bfloat16, seed=120 + N)
    g = torch.Generator().manual_seed(121 + N)
    lo, hi = arange
    alpha = lo + (hi - lo) * torch.rand((1, 3, N), generator=g)
    S0 = torch.randn((1, 3, 128, 128), generator=g) * 0.5
    reads, S = la.gated_delta_prefill(k.cuda(), v.cuda(), beta.cuda(), alpha.cuda(), S0=S0.cuda())
    rr, rS = orc.gated_delta(f64(k), f64(v), f64(beta), f64(alpha), S0=f64(S0))
    assert relmax(f64(reads), rr) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert la.delta_read_device_status() == 0


def test_gated_delta_chunked_zero_alpha_erases(la, orc):
    # alpha = 0 at some tokens (clamped to 1e-30 inside the chunk factors):
    # the memory before them is forgotten
    from fixed_state_recurrent_gb300 import inputs
    N = 400
    k, v, beta = inputs.delta_inputs(1, 2, N, 128, 128, torch.bfloat16, seed=130)
    alpha = torch.full((1, 2, N), 0.97)
    alpha[:, :, [5, 64, 100, 255, 256, 399]] = 0.0
    S0 = torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(131))
    reads, S = la.gated_delta_prefill(k.cuda(), v.cuda(), beta.cuda(), alpha.cuda(), S0=S0.cuda())
    rr, rS = orc.gated_delta(f64(k), f64(v), f64(beta), f64(alpha), S0=f64(S0))
    assert relmax(f64(reads), rr) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16


def test_gated_delta_chunked_alpha_one_is_delta(la):
    # the gated kernel with alpha = 1 against the plain chunked kernel: the same
    # products, the factors all exactly 1
    from fixed_state_recurrent_gb300 import inputs
    k, v, beta = inputs.delta_inputs(1, 2, 333, 128, 128, torch.bfloat16, seed=132)
    kd, vd, bd = k.cuda(), v.cuda(), beta.cuda()
    a = la.gated_delta_prefill(kd, vd, bd, torch.ones((1, 2, 333), device="cuda"))
    b = la.delta_prefill(kd, vd, bd)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_gated_delta_chunked_repeatable(la):
    from fixed_state_recurrent_gb300 import inputs
    k, v, beta = inputs.delta_inputs(1, 3, 777, 128, 128, torch.bfloat16, seed=133)
    alpha = 0.5 + 0.5 * torch.rand((1, 3, 777), generator=torch.Generator().manual_seed(134))
    kd, vd, bd, ad = k.cuda(), v.cuda(), beta.cuda(), alpha.cuda()
    first = la.gated_delta_prefill(kd, vd, bd, ad)
    for _ in range(12):
        again = la.gated_delta_prefill(kd, vd, bd, ad)
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])


# decayed write-then-read prefill on the tensor cores (bf16, dk = dv = 64):
# one block per head, 128-token chunks with decay factors inside each chunk
DECAY_N = [1, 127, 128, 129, 300, 1000]


@pytest.mark.parametrize("N", DECAY_N)
@pytest.mark.parametrize("arange", [(0.9, 1.0), (0.3, 1.0), (0.02, 0.5)], ids=["mild", "strong", "severe"])
def test_decay_prefill_tc_matches_oracle(la, orc, N, arange):
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(1, 3, N, 64, 64, torch.bfloat16, seed=140 + N)
    g = torch.Generator().manual_seed(141 + N)
    lo, hi = arange
    alpha = lo + (hi - lo) * torch.rand((1, 3, N), generator=g)
    S0 = torch.randn((1, 3, 64, 64), generator=g) * 0.5
    z0 = torch.rand((1, 3, 64), generator=g) * 4 + 0.5
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), alpha.cuda(), 0,
                                 S0=S0.cuda(), z0=z0.cuda())
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha), 0, S0=f64(S0), z0=f64(z0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16
    assert la.delta_read_device_status() == 0


# the decayed forms over pieces: runs that cross heads, heads over many blocks
# (entry states folded from earlier totals and decays); the last shape has
# more than 2048 chunks, so it runs the three-launch form
DECAY_SHAPES = [(2, 5, 3000), (3, 40, 333), (1, 2, 20000), (1, 4, 70000)]


@pytest.mark.parametrize("shape", DECAY_SHAPES, ids=[str(s) for s in DECAY_SHAPES])
@pytest.mark.parametrize("arange", [(0.9, 1.0), (0.02, 0.5)], ids=["mild", "severe"])
def test_decay_prefill_tc_pieces_match_oracle(la, orc, shape, arange):
    from fixed_state_recurrent_gb300 import inputs
    B, H, N = shape
    q, k, v = inputs.la_inputs(B, H, N, 64, 64, torch.bfloat16, seed=145 + N % 61)
    g = torch.Generator().manual_seed(146 + N)
    lo, hi = arange
    alpha = lo + (hi - lo) * torch.rand((B, H, N), generator=g)
    S0 = torch.randn((B, H, 64, 64), generator=g) * 0.5
    z0 = torch.rand((B, H, 64), generator=g) * 4 + 0.5
    la.delta_read_device_status()
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), alpha.cuda(), 0,
                                 S0=S0.cuda(), z0=z0.cuda())
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha), 0, S0=f64(S0), z0=f64(z0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16
    assert la.delta_read_device_status() == 0


# the decayed form at d = 128 (three launches with decay weights; a workspace)
DECAY128_SHAPES = [(1, 3, 1), (1, 3, 129), (1, 3, 300), (2, 5, 3000), (3, 40, 333), (1, 2, 20000)]


@pytest.mark.parametrize("shape", DECAY128_SHAPES, ids=[str(s) for s in DECAY128_SHAPES])
@pytest.mark.parametrize("arange", [(0.9, 1.0), (0.3, 1.0), (0.02, 0.5)], ids=["mild", "strong", "severe"])
def test_decay_prefill_tc_d128_matches_oracle(la, orc, shape, arange):
    from fixed_state_recurrent_gb300 import inputs
    B, H, N = shape
    q, k, v = inputs.la_inputs(B, H, N, 128, 128, torch.bfloat16, seed=195 + N % 67)
    g = torch.Generator().manual_seed(196 + N)
    lo, hi = arange
    alpha = lo + (hi - lo) * torch.rand((B, H, N), generator=g)
    S0 = torch.randn((B, H, 128, 128), generator=g) * 0.5
    z0 = torch.rand((B, H, 128), generator=g) * 4 + 0.5
    la.delta_read_device_status()
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), alpha.cuda(), 0,
                                 S0=S0.cuda(), z0=z0.cuda())
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha), 0, S0=f64(S0), z0=f64(z0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16
    assert la.delta_read_device_status() == 0


def test_decay_prefill_tc_d128_zero_alpha_and_alpha_one(la, orc):
    # alpha = 0 at chunk edges forgets the state before them; alpha = 1 is
    # la_prefill's recurrence (through other kernels: within the tolerance)
    from fixed_state_recurrent_gb300 import inputs
    N = 520
    q, k, v = inputs.la_inputs(2, 2, N, 128, 128, torch.bfloat16, seed=197)
    alpha = torch.full((2, 2, N), 0.97)
    alpha[:, :, [0, 5, 127, 128, 255, 300, 519]] = 0.0
    S0 = torch.randn((2, 2, 128, 128), generator=torch.Generator().manual_seed(198))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, S, z = la.prefill_variant(qd, kd, vd, alpha.cuda(), 0, S0=S0.cuda())
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha), 0, S0=f64(S0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16
    a = la.prefill_variant(qd, kd, vd, torch.ones((2, 2, N), device="cuda"), 0)
    b = la.prefill(qd, kd, vd)
    for x, y in zip(a, b):
        assert relmax(f64(x), f64(y)) <= TOL_BF16


def test_decay_prefill_tc_d128_bounded_wait_reports_timeout(la, orc, monkeypatch):
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(1, 2, 600, 128, 128, torch.bfloat16, seed=199)
    alpha = torch.full((1, 2, 600), 0.99, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    la.delta_read_device_status()
    monkeypatch.setenv("LA_TEST_FORCE_WAIT", "1")
    monkeypatch.setenv("LA_MBAR_TIMEOUT_NS", "2000000")
    la.prefill_variant(qd, kd, vd, alpha, 0)
    assert la.delta_read_device_status() == 4  # LA_ERR_TIMEOUT
    assert la.delta_read_device_status() == 0
    monkeypatch.delenv("LA_TEST_FORCE_WAIT")
    monkeypatch.delenv("LA_MBAR_TIMEOUT_NS")
    o, S, z = la.prefill_variant(qd, kd, vd, alpha, 0)
    assert la.delta_read_device_status() == 0
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha.cpu()), 0)
    assert relmax(f64(o), ro) <= TOL_BF16


# read before write with a decay on the tensor cores: the three-launch forms
# with a strict mask and the query side decayed to the token before (and, at
# d = 64 without a workspace, one block per head)
RBW_DECAY_SHAPES = [(64, 1, 3, 1), (64, 1, 3, 300), (64, 2, 5, 3000), (64, 3, 40, 333),
                    (128, 1, 3, 129), (128, 2, 5, 3000), (128, 3, 40, 333)]


@pytest.mark.parametrize("shape", RBW_DECAY_SHAPES, ids=[str(s) for s in RBW_DECAY_SHAPES])
@pytest.mark.parametrize("arange", [(0.9, 1.0), (0.02, 0.5)], ids=["mild", "severe"])
@pytest.mark.parametrize("ws", [None, False], ids=["ws", "nows"])
def test_decay_read_before_write_tc_matches_oracle(la, orc, shape, arange, ws):
    from fixed_state_recurrent_gb300 import inputs
    d, B, H, N = shape
    if ws is False and d == 128:
        pytest.skip("d = 128 without a workspace runs on the CUDA cores")
    q, k, v = inputs.la_inputs(B, H, N, d, d, torch.bfloat16, seed=205 + N % 53)
    g = torch.Generator().manual_seed(206 + N + d)
    lo, hi = arange
    alpha = lo + (hi - lo) * torch.rand((B, H, N), generator=g)
    alpha[:, :, ::97] = 0.0  # some tokens forget everything before them
    S0 = torch.randn((B, H, d, d), generator=g) * 0.5
    z0 = torch.rand((B, H, d), generator=g) * 4 + 0.5
    la.delta_read_device_status()
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), alpha.cuda(), la.LA_MODE_READ_BEFORE_WRITE,
                                 S0=S0.cuda(), z0=z0.cuda(), ws=ws)
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha), 1, S0=f64(S0), z0=f64(z0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16
    assert la.delta_read_device_status() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_decay_read_before_write_tc_large_eps(la, orc, d):
    # with a large eps a stray alpha_t on the read would show: token t reads
    # S_{t-1} (decayed only up to token t - 1), numerator and denominator alike
    from fixed_state_recurrent_gb300 import inputs
    B, H, N = 1, 3, 700
    q, k, v = inputs.la_inputs(B, H, N, d, d, torch.bfloat16, seed=215 + d)
    g = torch.Generator().manual_seed(216 + d)
    alpha = 0.2 + 0.8 * torch.rand((B, H, N), generator=g)
    S0 = torch.randn((B, H, d, d), generator=g) * 0.5
    z0 = torch.rand((B, H, d), generator=g) * 4 + 0.5
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), alpha.cuda(), la.LA_MODE_READ_BEFORE_WRITE,
                                 eps=0.5, S0=S0.cuda(), z0=z0.cuda())
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha), 1, eps=0.5, S0=f64(S0), z0=f64(z0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16


def test_decay_prefill_tc_zero_alpha_forgets(la, orc):
    # alpha = 0 at some tokens (taken as 1e-30 in the chunk factors): the state
    # before them is forgotten, including right at chunk edges
    from fixed_state_recurrent_gb300 import inputs
    N = 520
    q, k, v = inputs.la_inputs(2, 2, N, 64, 64, torch.bfloat16, seed=150)
    alpha = torch.full((2, 2, N), 0.97)
    alpha[:, :, [0, 5, 127, 128, 255, 300, 519]] = 0.0
    S0 = torch.randn((2, 2, 64, 64), generator=torch.Generator().manual_seed(151))
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), alpha.cuda(), 0, S0=S0.cuda())
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha), 0, S0=f64(S0))
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16


def test_decay_prefill_tc_alpha_one_is_prefill(la):
    # alpha = 1: the decayed kernel computes la_prefill's recurrence (through
    # other kernels, so within the bf16 tolerance rather than bit for bit)
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(1, 4, 700, 64, 64, torch.bfloat16, seed=152)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    a = la.prefill_variant(qd, kd, vd, torch.ones((1, 4, 700), device="cuda"), 0)
    ws = la.workspace(1, 4, 700, 64, 64, torch.bfloat16, 0, torch.device("cuda"))
    b = la.prefill(qd, kd, vd, ws=ws)
    for x, y in zip(a, b):
        assert relmax(f64(x), f64(y)) <= TOL_BF16


def test_decay_prefill_tc_state_in_place_and_repeatable(la, orc):
    # S_N over S0 and z_N over z0 (the allowed aliasing); runs are bitwise equal
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(1, 3, 777, 64, 64, torch.bfloat16, seed=153)
    g = torch.Generator().manual_seed(154)
    alpha = 0.6 + 0.4 * torch.rand((1, 3, 777), generator=g)
    S0 = torch.randn((1, 3, 64, 64), generator=g)
    z0 = torch.rand((1, 3, 64), generator=g) + 1.0
    qd, kd, vd, ad = q.cuda(), k.cuda(), v.cuda(), alpha.cuda()
    first = la.prefill_variant(qd, kd, vd, ad, 0, S0=S0.cuda(), z0=z0.cuda())
    for _ in range(8):
        again = la.prefill_variant(qd, kd, vd, ad, 0, S0=S0.cuda(), z0=z0.cuda())
        assert all(torch.equal(x, y) for x, y in zip(first, again))
    Sd, zd = S0.clone().cuda(), z0.clone().cuda()
    o, S, z = la.prefill_variant(qd, kd, vd, ad, 0, S0=Sd, z0=zd, S_N=Sd, z_N=zd)
    assert torch.equal(o, first[0]) and torch.equal(Sd, first[1]) and torch.equal(zd, first[2])
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha), 0, S0=f64(S0), z0=f64(z0))
    assert relmax(f64(first[0]), ro) <= TOL_BF16 and relmax(f64(Sd), rS) <= TOL_BF16


def test_decay_prefill_tc_bounded_wait_reports_timeout(la, orc, monkeypatch):
    # the test hook makes the kernel's MMA thread wait on an mbarrier that
    # nothing completes (2 ms limit): the launch finishes, the library status
    # word says LA_ERR_TIMEOUT, reading clears it, and the next call is right
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(1, 2, 600, 64, 64, torch.bfloat16, seed=155)
    alpha = torch.full((1, 2, 600), 0.99, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    la.delta_read_device_status()
    monkeypatch.setenv("LA_TEST_FORCE_WAIT", "1")
    monkeypatch.setenv("LA_MBAR_TIMEOUT_NS", "2000000")
    la.prefill_variant(qd, kd, vd, alpha, 0)
    assert la.delta_read_device_status() == 4  # LA_ERR_TIMEOUT
    assert la.delta_read_device_status() == 0
    monkeypatch.delenv("LA_TEST_FORCE_WAIT")
    monkeypatch.delenv("LA_MBAR_TIMEOUT_NS")
    o, S, z = la.prefill_variant(qd, kd, vd, alpha, 0)
    assert la.delta_read_device_status() == 0
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha.cpu()), 0)
    assert relmax(f64(o), ro) <= TOL_BF16


@pytest.mark.parametrize("shape", [(1, 3, 700), (2, 8, 2000), (1, 5, 4096)],
                         ids=["3x700", "16x2000", "5x4096"])
def test_decay_prefill_tc_split_and_per_head_agree(la, orc, shape):
    # with a workspace the heads are cut into pieces over every SM (pieces
    # start and end inside heads, and one piece spans two heads), chained by
    # the scan E' = Gamma E + R; without one, one block per head.  Both match
    # the oracle, on heads that carry an entry state.
    from fixed_state_recurrent_gb300 import inputs
    B, H, N = shape
    q, k, v = inputs.la_inputs(B, H, N, 64, 64, torch.bfloat16, seed=190 + N)
    g = torch.Generator().manual_seed(191 + N)
    alpha = 0.85 + 0.15 * torch.rand((B, H, N), generator=g)
    S0 = torch.randn((B, H, 64, 64), generator=g) * 0.5
    z0 = torch.rand((B, H, 64), generator=g) + 0.5
    args = (q.cuda(), k.cuda(), v.cuda(), alpha.cuda(), 0)
    split = la.prefill_variant(*args, S0=S0.cuda(), z0=z0.cuda())
    whole = la.prefill_variant(*args, S0=S0.cuda(), z0=z0.cuda(), ws=False)
    assert la.delta_read_device_status() == 0
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), f64(alpha), 0, S0=f64(S0), z0=f64(z0))
    for got in (split, whole):
        assert relmax(f64(got[0]), ro) <= TOL_BF16
        assert relmax(f64(got[1]), rS) <= TOL_BF16
        assert relmax(f64(got[2]), rz) <= TOL_BF16


# The variant workloads the bench times, at full size (B=4 H=8 N=4096, bf16,
# the bench's seeds and alpha ~ U(0.9, 1)): every head against the oracle, in
# the launch configuration the bench uses (a workspace from the binding).
@pytest.mark.parametrize("wname", ["prefill", "prefill128"])
@pytest.mark.parametrize("mode,decay", [(0, True), (1, False), (2, False)], ids=["decay", "rbw", "nc"])
def test_variant_bench_workloads_full(la, orc, wname, mode, decay):
    from fixed_state_recurrent_gb300 import inputs
    w = inputs.WORKLOADS[wname]
    q, k, v = inputs.la_inputs(w.B, w.H, w.N, w.dk, w.dv, w.dtype, w.seed)
    alpha = None
    if decay:
        g = torch.Generator().manual_seed(6)
        alpha = 0.9 + 0.1 * torch.rand((w.B, w.H, w.N), generator=g)
    la.delta_read_device_status()
    o, S, z = la.prefill_variant(q.cuda(), k.cuda(), v.cuda(), None if alpha is None else alpha.cuda(), mode)
    ro, rS, rz = orc.la_variant(f64(q), f64(k), f64(v), None if alpha is None else f64(alpha), mode)
    assert relmax(f64(o), ro) <= TOL_BF16
    assert relmax(f64(S), rS) <= TOL_BF16
    assert relmax(f64(z), rz) <= TOL_BF16
    assert la.delta_read_device_status() == 0
