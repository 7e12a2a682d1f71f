"""la_prefill_noalloc: the prefill entry point for callers that cannot
allocate device memory (graph-capturing code, server plugins that only get
input and output buffers, processes whose device memory another allocator
owns).  It must give what la_prefill gives, call after call, from the
library's own fixed scratch.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It also passes alone in a
fresh process (the first call does the one-time scratch set-up)."""
import ctypes

import pytest
import torch

from helpers import f64, relmax, TOL_BF16, TOL_F32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrent_gb300 import build, api
    build.build()
    api.load()
    return api


def _inputs(B, H, N, d, dtype, seed):
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(B, H, N, d, d, dtype, seed)
    return q.cuda(), k.cuda(), v.cuda()


@pytest.mark.parametrize("case", [(2, 4, 4096, 64, torch.bfloat16),   # tensor-core path
                                  (2, 3, 1000, 128, torch.bfloat16),  # tensor-core, d = 128
                                  (1, 2, 300, 64, torch.float32)],    # CUDA-core path
                         ids=["bf16_d64", "bf16_d128", "f32"])
def test_noalloc_matches_prefill_two_calls_in_a_row(la, case):
    B, H, N, d, dtype = case
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    g = torch.Generator().manual_seed(77)
    S0 = (torch.randn((B, H, d, d), generator=g) * 2).cuda()
    z0 = (torch.rand((B, H, d), generator=g) * 10 + 1).cuda()
    for call in range(2):  # two calls in a row on fresh inputs: the scratch is reused
        q, k, v = _inputs(B, H, N, d, dtype, seed=300 + call)
        o_ref, S_ref, z_ref = la.prefill(q, k, v, S0=S0, z0=z0)
        o, S, z = la.prefill_noalloc(q, k, v, S0=S0, z0=z0)
        torch.cuda.synchronize()
        assert relmax(f64(o), f64(o_ref)) <= tol
        assert relmax(f64(S), f64(S_ref)) <= tol
        assert relmax(f64(z), f64(z_ref)) <= tol


def test_noalloc_rejects_requests_beyond_its_scratch(la):
    # 64 heads x 65536 tokens at d = 64 needs far more than the 16 MiB scratch
    need = la.prefill_workspace_bytes(1, 64, 65536, 64, 64)
    assert need > (16 << 20)
    q = torch.empty((1, 64, 65536, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(la.LAError) as err:
        la.prefill_noalloc(q, q, q)
    assert err.value.status == 1  # LA_ERR_INVALID_ARG
