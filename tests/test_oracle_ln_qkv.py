"""Pins of the oracle's pre-attention LayerNorm and fused Wqkv projection:
h = LayerNorm(x) (bias-free, population variance, eps 1e-5 under the square
root, times the weight; the identity on layer 0), qkv = h Wqkv^T with Wqkv
stored [out][in] = [2304][768] ("ModernBERT-base Architecture Teardown",
"What Does LayerNorm Do?" and "How Does ModernBERT Make Q, K and V?";
"ModernBERT" (candding), "The pre-norm layer and the final norm";
"ModernBertModel" (safebydesign), "Implementing it").

Each pin fixes the result by something other than the oracle's own formula:
the page's worked example, closed forms, exact invariances, or an
independent library routine.
"""
import os

import numpy as np
import pytest
import torch

import oracle

D = 768
N_OUT = 3 * D
HERE = os.path.dirname(os.path.abspath(__file__))


def bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).double().numpy()


def rand(shape, seed, scale=1.0, shift=0.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale + shift).to(torch.bfloat16)


def read_fixture():
    rec = {}
    with open(os.path.join(HERE, "golden", "layernorm_worked_example.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *vals = line.split()
            rec[k] = [float(v) for v in vals]
    return rec


def test_page_worked_example():
    # the page divides by the plain standard deviation (no eps) in its hand
    # computation, then notes the eps of the real LayerNorm
    rec = read_fixture()
    x = torch.tensor([rec["input"]])
    ones = bits(torch.ones(4))
    h0 = oracle.layernorm(bits(x), ones, eps=0.0)[0]
    assert np.array_equal(np.round(h0, 4), np.array(rec["normalised"]))
    v = np.array(rec["input"])
    mean, std = rec["mean"][0], rec["std"][0]
    assert np.allclose(mean + std * h0, v, atol=2e-4)      # the printed mean and spread
    h = oracle.layernorm(bits(x), ones)[0]                 # eps = 1e-5: var 2.297 barely moves
    assert np.allclose(h, h0, rtol=3e-6, atol=0) and not np.array_equal(h, h0)


def test_mean_zero_and_spread_closed_form():
    # sum_c h_c = 0 and sum_c h_c^2 / d = var / (var + eps) for weight 1
    x = rand((16, D), 1, scale=3.0, shift=0.7)
    h = oracle.layernorm(bits(x), bits(torch.ones(D)))
    xv = f64(x)
    var = xv.var(axis=1)                       # population variance (numpy's default)
    assert np.allclose(h.sum(axis=1), 0.0, atol=1e-10)
    assert np.allclose((h ** 2).mean(axis=1), var / (var + oracle.NORM_EPS), rtol=1e-12)


def test_constant_row_gives_zero():
    x = torch.full((3, D), 2.5)
    h = oracle.layernorm(bits(x), bits(rand((D,), 2)))
    assert np.array_equal(h, np.zeros((3, D)))


def test_scale_invariance_without_eps():
    # with eps = 0, scaling a row by a power of two changes nothing, bit for bit
    x = rand((8, D), 3)
    w = bits(rand((D,), 4))
    h1 = oracle.layernorm(bits(x), w, eps=0.0)
    h2 = oracle.layernorm(bits(x.float() * 4.0), w, eps=0.0)
    assert np.array_equal(h1, h2)


def test_shift_invariance_on_integers():
    # rows of small integers that sum to zero, shifted by an integer: the
    # means are exactly 0 and 37, so the deviations, hence the outputs, are
    # the same bit for bit
    g = torch.Generator().manual_seed(5)
    a = torch.randint(-20, 21, (6, D // 2), generator=g).float()
    x = torch.cat([a, -a], dim=1)
    w = bits(rand((D,), 6))
    h1 = oracle.layernorm(bits(x), w)
    h2 = oracle.layernorm(bits(x + 37.0), w)
    assert np.array_equal(h1, h2)


def test_weight_scales_positions():
    # LayerNorm(x; w) = LayerNorm(x; 1) * w position by position
    x = rand((8, D), 7)
    w = rand((D,), 8)
    h1 = oracle.layernorm(bits(x), bits(torch.ones(D)))
    hw = oracle.layernorm(bits(x), bits(w))
    assert np.allclose(hw, h1 * f64(w)[None, :], rtol=1e-15, atol=1e-15)


def test_matches_torch_layer_norm():
    # an independent implementation: torch's layer_norm in fp64, no bias
    x = rand((32, D), 9, scale=2.0, shift=-1.0)
    w = rand((D,), 10)
    h = oracle.layernorm(bits(x), bits(w))
    ref = torch.nn.functional.layer_norm(torch.from_numpy(f64(x)), (D,),
                                         weight=torch.from_numpy(f64(w)), bias=None,
                                         eps=oracle.NORM_EPS).numpy()
    assert np.allclose(h, ref, rtol=0, atol=1e-12)


def test_ln_qkv_equals_library_matmul():
    # qkv = LayerNorm(x) Wqkv^T: torch layer_norm then a numpy matmul
    x = rand((24, D), 11)
    w = rand((D,), 12)
    wq = rand((N_OUT, D), 13, scale=D ** -0.5)
    got = oracle.ln_qkv(bits(x), bits(w), bits(wq))
    h = torch.nn.functional.layer_norm(torch.from_numpy(f64(x)), (D,),
                                       weight=torch.from_numpy(f64(w)), eps=oracle.NORM_EPS)
    ref = h.numpy() @ f64(wq).T
    assert got.shape == (24, N_OUT)
    assert np.allclose(got, ref, rtol=0, atol=1e-11)


def test_identity_norm_of_layer_zero():
    # no norm before layer 0's attention: qkv = x Wqkv^T
    x = rand((20, D), 14)
    wq = rand((N_OUT, D), 15, scale=D ** -0.5)
    got = oracle.ln_qkv(bits(x), None, bits(wq))
    assert np.allclose(got, f64(x) @ f64(wq).T, rtol=0, atol=1e-11)
    assert np.array_equal(oracle.layernorm(bits(x), None), f64(x))


def test_three_way_split_with_selection_weights():
    # Wqkv = [I; 2I; -I]: q = h, k = 2h, v = -h, exactly, in the order the
    # model cuts the 2304 outputs
    x = rand((5, D), 16)
    w = rand((D,), 17)
    eye = torch.eye(D)
    wq = torch.cat([eye, 2 * eye, -eye])
    got = oracle.ln_qkv(bits(x), bits(w), bits(wq))
    h = oracle.layernorm(bits(x), bits(w))
    assert np.array_equal(got[:, :D], h)
    assert np.array_equal(got[:, D:2 * D], 2 * h)
    assert np.array_equal(got[:, 2 * D:], -h)


def test_linear_in_the_weight():
    x = rand((6, D), 18)
    w = bits(rand((D,), 19))
    w1 = rand((N_OUT, D), 20, scale=0.03)
    w2 = rand((N_OUT, D), 21, scale=0.03)
    # bf16 sums of bf16 values need not be exact: use exactly representable halves
    y1 = oracle.ln_qkv(bits(x), w, bits(w1))
    y2 = oracle.ln_qkv(bits(x), w, bits(w2))
    w12 = bits(w1.float() * 0.5) , bits(w2.float() * 0.5)
    y12 = oracle.ln_qkv(bits(x), w, w12[0]) + oracle.ln_qkv(bits(x), w, w12[1])
    assert np.allclose(y12, 0.5 * (y1 + y2), rtol=0, atol=1e-12)


@pytest.mark.parametrize("fn", ["layernorm", "ln_qkv"])
def test_sampled_rows_equal_full_rows(fn):
    x = rand((50, D), 22)
    w = bits(rand((D,), 23))
    rows = np.array([0, 7, 31, 49])
    if fn == "layernorm":
        full = oracle.layernorm(bits(x), w)
        part = oracle.layernorm(bits(x), w, rows=rows)
    else:
        wq = bits(rand((N_OUT, D), 24, scale=D ** -0.5))
        full = oracle.ln_qkv(bits(x), w, wq)
        part = oracle.ln_qkv(bits(x), w, wq, rows=rows)
    assert np.array_equal(part, full[rows])
