"""The two exponential routines of the softmax against 2^x in fp64: the MUFU
ex2 and the FMA-pipe polynomial that takes part of each row's exponentials
(range reduction to [-1/2, 1/2], degree-3 minimax fit, 1.0e-4 relative)."""
import math

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import sequence_attn_fwd_gb300 as sa

    return sa


def run(sa, x, poly):
    y = torch.full_like(x, float("nan"))
    st = torch.cuda.current_stream().cuda_stream
    assert sa.lib.attn_debug_exp2(x.data_ptr(), y.data_ptr(), x.numel(), poly, st) == 0
    torch.cuda.synchronize()
    return y


def inputs():
    special = torch.tensor([-math.inf, -1000.0, -127.0, -126.75, -126.5, -126.0, -125.0, -0.5, 0.5, 0.0,
                            -0.0, 1e-30, -1e-30, 7.999, 8.0, 0.49999997, -0.49999997])
    grid = torch.linspace(-130.0, 9.0, 400_001, dtype=torch.float64).float()
    return torch.cat([special, grid, torch.tensor([3.0])]).cuda()  # odd length: last pairs with itself


@pytest.mark.parametrize("poly,bound", [(1, 1.02e-4), (0, 4e-6)])
def test_exp2_relative_error_in_normal_range(sa, poly, bound):
    x = inputs()
    y = run(sa, x, poly).double()
    ref = torch.exp2(x.double())
    normal = x >= -125.0
    rel = (y[normal] / ref[normal] - 1).abs()
    assert rel.max().item() < bound, rel.max().item()
    assert torch.isfinite(y).all() and (y >= 0).all()


def test_poly_exp2_underflow_and_minus_inf_give_exact_zero(sa):
    x = inputs()
    y = run(sa, x, 1)
    assert (y[x <= -127.0] == 0).all()  # includes -inf: masked scores must add nothing
    low = (x > -127.0) & (x < -125.0)
    assert (y[low] >= 0).all() and (y[low] <= 2.0 ** -124).all()
    assert y[(x == 0)].eq(1.0).all()  # p(0) = 1 exactly


def test_poly_and_mufu_agree(sa):
    x = inputs()
    a, b = run(sa, x, 1).double(), run(sa, x, 0).double()
    m = x >= -125.0
    assert ((a[m] / b[m]) - 1).abs().max().item() < 1.1e-4
