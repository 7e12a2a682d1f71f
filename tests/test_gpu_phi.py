"""The ELU+1 feature map of the tensor-core prefill, over every finite bf16
input, through the C ABI.

The tensor-core kernels need phi only as a bf16 MMA operand; they form
exp(u) as 2^(u log2 e) with the hardware base-2 exponential and round the
result to bf16.  The claim checked here: for every finite bf16 u, the value
the kernels use is within one bf16 rounding (relative 2^-8) of the fp64
oracle's phi(u) (page "AIGC 基本功|线性、循环与记忆架构-LinearMem", section 03:
u + 1 for u > 0, exp(u) otherwise), except that results below 2^-126 may be
flushed to zero.  The kernels' phi values are read out exactly:

* phi(K): with v_t = e_t (one-hot values) and S0 = 0, the final state is
  S_N[i][j] = phi(k_j)_i, one bf16 product per entry, exact in fp32;
* phi(Q): with k_t very negative (phi(k) flushed to 0), v = 0, S0 = I and
  z0 = e_0, the output is o_t[j] = phi(q_t)_j / (phi(q_t)_0 + eps), and
  q_t[0] = 0 makes the denominator 1 + eps.
"""
import numpy as np
import pytest
import torch

from helpers import f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrent_gb300 import build, api
    build.build()
    api.load()
    return api


def _finite_bf16():
    """Every finite bf16 value, in bit-pattern order (65280 values)."""
    bits = np.arange(65536, dtype=np.uint32)
    exp_all_ones = (bits & 0x7F80) == 0x7F80
    f32 = (bits[~exp_all_ones] << 16).view(np.float32)
    return torch.from_numpy(f32.copy()).to(torch.bfloat16)


def _check_phi(orc, got, u):
    ref = orc.phi(f64(u))
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    tiny = ref < 2.0 ** -126  # may flush to zero
    ok = (err <= 2.0 ** -8 * ref) | (tiny & (got <= 2.0 ** -126))
    bad = np.flatnonzero(~ok)
    assert bad.size == 0, [(float(f64(u)[i]), got[i], ref[i]) for i in bad[:8]]
    # most values are the correctly rounded bf16 of phi
    rounded = f64(torch.from_numpy(ref).to(torch.bfloat16))
    assert np.mean(got == rounded) > 0.99


@pytest.mark.parametrize("d", [64, 128])
def test_phi_of_k_every_finite_bf16(la, orc, d):
    u = _finite_bf16()
    heads = (u.numel() + d * d - 1) // (d * d)
    k = torch.zeros(heads * d * d, dtype=torch.bfloat16)
    k[:u.numel()] = u
    k = k.view(1, heads, d, d)                       # token j of a head holds d inputs
    v = torch.eye(d, dtype=torch.bfloat16).expand(1, heads, d, d).contiguous()
    q = torch.zeros_like(k)
    _, S, _ = la.prefill(q.cuda(), k.cuda(), v.cuda())
    S = S.cpu()
    phik = S.transpose(-1, -2).reshape(-1)[:u.numel()]  # S_N[i][j] = phi(k_j)_i
    _check_phi(orc, f64(phik), u)


@pytest.mark.parametrize("d", [64, 128])
def test_phi_of_q_every_finite_bf16(la, orc, d):
    u = _finite_bf16()
    per = d - 1                                      # feature 0 of every token is 0
    N = (u.numel() + per - 1) // per
    q = torch.zeros((N * per,), dtype=torch.bfloat16)
    q[:u.numel()] = u
    q = torch.cat([torch.zeros((N, 1), dtype=torch.bfloat16), q.view(N, per)], dim=1)
    q = q.view(1, 1, N, d).contiguous()
    k = torch.full_like(q, -100.0)                   # phi(k) = e^-100: below 2^-126
    v = torch.zeros_like(q)
    S0 = torch.eye(d, dtype=torch.float32).view(1, 1, d, d).contiguous()
    z0 = torch.zeros((1, 1, d), dtype=torch.float32)
    z0[0, 0, 0] = 1.0
    eps = 1e-6
    o, _, _ = la.prefill(q.cuda(), k.cuda(), v.cuda(), eps=eps, S0=S0.cuda(), z0=z0.cuda())
    o = f64(o.cpu())[0, 0]
    phiq = (o[:, 1:] * (1.0 + eps)).reshape(-1)[:u.numel()]
    # o carries the fp32 rounding of 1 / (1 + eps) and of one product, far
    # below a bf16 step: rounding to bf16 gives back the operand the MMA used
    phiq = f64(torch.from_numpy(phiq).to(torch.bfloat16))
    _check_phi(orc, phiq, u)
