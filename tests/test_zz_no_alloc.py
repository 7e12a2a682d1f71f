"""la_prefill_noalloc: the prefill entry point for callers that cannot
allocate device memory (graph-capturing code, server plugins that only get
input and output buffers, processes whose device memory another allocator
owns).  It must give exactly what la_prefill gives, call after call, from the
library's own fixed scratch: both run the same kernels on the same inputs, so
the results are compared bit for bit, and once against the oracle.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It also passes alone in a
fresh process (the first call does the one-time set-up), and one case makes
that first call in a fresh child process on a non-default stream."""
import os
import subprocess
import sys

import pytest
import torch

from helpers import f64, relmax, tol_for

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
    return inputs.la_inputs(B, H, N, d, d, dtype, seed)


@pytest.mark.parametrize("case", [(2, 4, 4096, 64, torch.bfloat16),   # tensor-core path
                                  (1, 4, 70000, 64, torch.bfloat16),  # d = 64, past 2048 chunks
                                  (2, 3, 1000, 128, torch.bfloat16),  # tensor-core, d = 128
                                  (1, 2, 300, 64, torch.float32)],    # CUDA-core path
                         ids=["bf16_d64", "bf16_d64_long", "bf16_d128", "f32"])
def test_noalloc_matches_prefill_two_calls_in_a_row(la, orc, case):
    B, H, N, d, dtype = case
    g = torch.Generator().manual_seed(77)
    S0 = torch.randn((B, H, d, d), generator=g) * 2
    z0 = torch.rand((B, H, d), generator=g) * 10 + 1
    S0d, z0d = S0.cuda(), z0.cuda()
    la.delta_read_device_status()  # start from a clear library status word
    for call in range(2):  # two calls in a row on fresh inputs: the scratch is reused
        q, k, v = _inputs(B, H, N, d, dtype, seed=300 + call)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        o_ref, S_ref, z_ref = la.prefill(qd, kd, vd, S0=S0d, z0=z0d)
        o, S, z = la.prefill_noalloc(qd, kd, vd, S0=S0d, z0=z0d)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(S, S_ref) and torch.equal(z, z_ref)
        if call == 1:  # and against the oracle, within the parity tolerance
            ro, rS, rz = orc.la_recurrent(f64(q), f64(k), f64(v), S0=f64(S0), z0=f64(z0))
            tol = tol_for(dtype)
            assert relmax(f64(o), ro) <= tol
            assert relmax(f64(S), rS) <= tol and relmax(f64(z), rz) <= tol
    assert la.delta_read_device_status() == 0  # LA_OK: no wait gave up


_CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from fixed_state_recurrent_gb300 import api, inputs
api.load()
q, k, v = (t.cuda() for t in inputs.la_inputs(2, 4, 2000, 64, 64, torch.bfloat16, 41))
side = torch.cuda.Stream()
with torch.cuda.stream(side):
    first = api.prefill_noalloc(q, k, v)          # the very first call, on a side stream
    ref = api.prefill(q, k, v)
side.synchronize()
assert all(torch.equal(a, b) for a, b in zip(first, ref)), "first call differs"
print("noalloc-child-ok")
"""


def test_noalloc_first_call_on_a_side_stream_in_a_fresh_process(la):
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "noalloc-child-ok" in r.stdout, r.stdout + r.stderr


def test_noalloc_bounded_wait_reports_timeout(la, orc, monkeypatch):
    # The test hook makes one wait of the output kernel wait on a barrier that
    # nothing completes, with a 2 ms limit: the call finishes, the library
    # status word says LA_ERR_TIMEOUT, reading clears it, and the next call is
    # correct again.
    q, k, v = _inputs(1, 2, 1024, 64, torch.bfloat16, seed=25)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    la.delta_read_device_status()  # start from a clear library status word
    monkeypatch.setenv("LA_TEST_FORCE_WAIT", "1")
    monkeypatch.setenv("LA_MBAR_TIMEOUT_NS", "2000000")
    la.prefill_noalloc(qd, kd, vd)
    assert la.delta_read_device_status() == 4  # LA_ERR_TIMEOUT
    assert la.delta_read_device_status() == 0  # reading clears it
    monkeypatch.delenv("LA_TEST_FORCE_WAIT")
    monkeypatch.delenv("LA_MBAR_TIMEOUT_NS")
    o, S, z = la.prefill_noalloc(qd, kd, vd)
    assert la.delta_read_device_status() == 0
    ro, rS, rz = orc.la_recurrent(f64(q), f64(k), f64(v))
    assert relmax(f64(o), ro) <= tol_for(q.dtype)


def test_noalloc_rejects_requests_beyond_its_scratch(la):
    # 64 heads x 4096 tokens at d = 64 (2048 chunks, the two-launch form, which
    # keeps a bf16 copy of phi(K)) needs more than the 16 MiB scratch
    need = la.prefill_workspace_bytes(1, 64, 4096, 64, 64)
    assert need > (16 << 20)
    q = torch.empty((1, 64, 4096, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(la.LAError) as err:
        la.prefill_noalloc(q, q, q)
    assert err.value.status == 1  # LA_ERR_INVALID_ARG
