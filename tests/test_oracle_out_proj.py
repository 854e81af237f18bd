"""Pins of the oracle's output projection with the residual add,
y = x + a Wo^T with Wo stored [out][in] ("ModernBERT-base Architecture
Teardown", "How Does ModernBERT Make Q, K and V?"; "ModernBertModel",
"Implementing it").  Each pin fixes the result by something other than the
oracle's own formula: a hand-worked example, special weights whose result is
known exactly, or a factorisation computed in a different order.
"""
import numpy as np
import torch

import oracle

D = 768


def bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).double().numpy()


def rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def test_hand_worked_example():
    # d = 3, worked by hand: y[t][o] = x[t][o] + sum_c a[t][c] wo[o][c]
    a = torch.tensor([[1.0, 2.0, 0.5], [-1.0, 0.0, 4.0]])
    wo = torch.tensor([[1.0, 0.0, 2.0], [0.0, -1.0, 0.25], [3.0, 1.0, 0.0]])
    x = torch.tensor([[0.5, -2.0, 1.0], [0.0, 0.0, 0.0]])
    y = oracle.out_proj(bits(a), bits(wo), bits(x))
    expected = np.array([[2.5, -3.875, 6.0], [7.0, 1.0, -3.0]])
    assert np.array_equal(y, expected)


def test_permutation_weight_permutes_columns():
    # wo[o][c] = 1 iff c = perm[o]: y = x + a[:, perm], exactly
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(D, generator=g)
    wo = torch.zeros(D, D)
    wo[torch.arange(D), perm] = 1.0
    a, x = rand((16, D), 6), rand((16, D), 7)
    y = oracle.out_proj(bits(a), bits(wo), bits(x))
    assert np.array_equal(y, f64(x) + f64(a)[:, perm.numpy()])


def test_zero_weight_returns_the_residual():
    a, x = rand((9, D), 8), rand((9, D), 9)
    y = oracle.out_proj(bits(a), bits(torch.zeros(D, D)), bits(x))
    assert np.array_equal(y, f64(x))


def test_power_of_two_diagonal():
    # wo = diag(2^k): each output column scales one input column, exactly
    k = torch.arange(D) % 7 - 3
    wo = torch.diag(torch.pow(2.0, k.double()).float())
    a, x = rand((5, D), 10), rand((5, D), 11)
    y = oracle.out_proj(bits(a), bits(wo), bits(x))
    assert np.array_equal(y, f64(x) + f64(a) * np.power(2.0, k.numpy().astype(np.float64)))


def test_rank_one_weight_factorises():
    # wo = u v^T: a wo^T = (a v) u^T, the contraction taken first
    u, v = rand((D,), 12), rand((D,), 13, 0.05)
    wo = torch.outer(u.float(), v.float()).to(torch.bfloat16)
    a, x = rand((8, D), 14), rand((8, D), 15)
    # wo's entries are u_o v_c rounded to bf16; use them as the oracle sees them
    y = oracle.out_proj(bits(a), bits(wo), bits(x))
    w = f64(wo)
    # row t: x_t + sum_c a_tc w_oc, with w taken column block by column block
    ref = f64(x).copy()
    A = f64(a)
    for c0 in range(0, D, 96):
        ref += A[:, c0:c0 + 96] @ w[:, c0:c0 + 96].T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # and the exact factorisation where the weights factor exactly
    u2 = torch.pow(2.0, (torch.arange(D) % 5 - 2).double()).float()
    v2 = torch.pow(2.0, (torch.arange(D) % 3 - 1).double()).float()
    wo2 = torch.outer(u2, v2)
    y2 = oracle.out_proj(bits(a), bits(wo2), bits(x))
    av = f64(a) @ v2.double().numpy()
    assert np.allclose(y2, f64(x) + np.outer(av, u2.double().numpy()), rtol=1e-13, atol=1e-12)


def test_sampled_rows_equal_full_rows():
    a, x, wo = rand((40, D), 16), rand((40, D), 17), rand((D, D), 18, 0.04)
    full = oracle.out_proj(bits(a), bits(wo), bits(x))
    rows = np.array([0, 3, 17, 39], dtype=np.int64)
    part = oracle.out_proj(bits(a), bits(wo), bits(x), rows=rows)
    assert np.array_equal(part, full[rows])
