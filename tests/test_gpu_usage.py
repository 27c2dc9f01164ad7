"""The README's usage example at a small size: every call runs and returns
finite values of the documented shapes, and the forward agrees with the
sequential unroll within the method error of K = 3."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_usage_example_runs():
    import nonlinear_rnn_gb300 as nr
    torch.manual_seed(0)
    B, T, d = 2, 256, 64
    x = torch.randn(B, T, d, device="cuda", dtype=torch.bfloat16)
    W_x = (torch.randn(3 * d, d, device="cuda") / d ** 0.5).to(torch.bfloat16)
    params = torch.rand(6, d) * 2 - 1
    P = nr.input_projection(x, W_x)
    assert P.shape == (B, T, 3 * d) and P.dtype == torch.bfloat16
    H, rho = nr.newton_forward(P, params, K=3)
    assert H.shape == (B, T, d) and torch.isfinite(H.float()).all() and rho.item() < 1.0
    gP, gparams = nr.newton_backward(P, params, H, torch.ones_like(H))
    assert gP.shape == P.shape and gparams.shape == (6, d)
    assert torch.isfinite(gP.float()).all() and torch.isfinite(gparams).all()
    h = nr.decode_step(params, h=H[:, -1], x=x[:, -1], W_x=W_x)
    assert h.shape == (B, d) and torch.isfinite(h.float()).all()
    Hs = nr.sequential_forward(P, params)
    assert (H.float() - Hs.float()).abs().max().item() < 0.1
