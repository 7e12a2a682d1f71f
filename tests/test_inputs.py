"""The seeded input generators: deterministic, right shapes, dtypes and
distributions.  They hold no arithmetic of the method."""
import torch

from fixed_state_recurrent_gb300 import inputs


def test_la_inputs_deterministic_and_rounded():
    a = inputs.la_inputs(2, 3, 17, 8, 5, torch.bfloat16, seed=5)
    b = inputs.la_inputs(2, 3, 17, 8, 5, torch.bfloat16, seed=5)
    c = inputs.la_inputs(2, 3, 17, 8, 5, torch.bfloat16, seed=6)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])
    q, k, v = a
    assert q.shape == (2, 3, 17, 8) and k.shape == (2, 3, 17, 8) and v.shape == (2, 3, 17, 5)
    assert q.dtype == torch.bfloat16 and q.is_contiguous()
    # round-to-nearest-even of the same fp32 draw
    g = torch.Generator().manual_seed(5)
    q32 = torch.randn((2, 3, 17, 8), generator=g)
    assert torch.equal(q, q32.to(torch.bfloat16))


def test_scale_applied_before_rounding():
    q, _, _ = inputs.la_inputs(1, 1, 64, 4, 4, torch.bfloat16, seed=2, scale=0.5)
    g = torch.Generator().manual_seed(2)
    q32 = torch.randn((1, 1, 64, 4), generator=g) * 0.5
    assert torch.equal(q, q32.to(torch.bfloat16))


def test_delta_inputs_unit_keys_and_beta_range():
    k, v, beta = inputs.delta_inputs(2, 2, 50, 16, 8, torch.bfloat16, seed=4)
    n = k.float().norm(dim=-1)
    assert torch.all((n - 1).abs() < 2e-2)  # unit up to bf16 rounding
    assert beta.dtype == torch.float32 and beta.shape == (2, 2, 50)
    assert torch.all((beta > 0) & (beta < 1))
    assert v.dtype == torch.bfloat16 and v.shape == (2, 2, 50, 8)


def test_named_workloads():
    w = inputs.WORKLOADS
    assert (w["prefill"].B, w["prefill"].H, w["prefill"].N, w["prefill"].dk) == (4, 8, 4096, 64)
    assert w["prefill"].tokens == 131072
    assert w["long"].scale == 0.5 and w["long"].tokens == 1048576
    assert (w["decode"].B, w["decode"].H, w["decode"].dk, w["decode"].steps) == (256, 32, 128, 100)
    assert (w["delta"].B, w["delta"].H, w["delta"].N, w["delta"].dk) == (8, 16, 8192, 128)
    assert w["pr1"].dtype == torch.float32
