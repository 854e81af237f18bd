"""Pins of the oracle's GeGLU MLP block: y = x + (GELU(g) * u) Wo^T with
g, u the first and second halves of LayerNorm(x; mlp_norm) Wi^T, GELU in its
exact erf form, Wi [2304][768] and Wo [768][1152] stored [out][in]
("ModernBERT-base Architecture Teardown", "What Does the GeGLU MLP Do?";
"ModernBERT" (candding), "The feed-forward halves"; "modernbert-base"
(nest.franknoh), "The fused projections" and "Why the GELU matters";
"ModernBertModel" (safebydesign), "Implementing it").

Each pin fixes the result by something other than the oracle's own formula:
the printed GELU values, exact special weights, and independent library
routines.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

D = 768
INNER = 1152
HERE = os.path.dirname(os.path.abspath(__file__))


def bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).double().numpy()


def rand(shape, seed, scale=1.0, shift=0.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale + shift).to(torch.bfloat16)


def weights(seed):
    w = rand((D,), seed, 0.1, 1.0)
    wi = rand((2 * INNER, D), seed + 1, D ** -0.5)
    wo = rand((D, INNER), seed + 2, INNER ** -0.5)
    return w, wi, wo


def read_gelu_fixture():
    out = []
    with open(os.path.join(HERE, "golden", "gelu_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            tag, z, v = line.split()
            out.append((tag, float(z), float(v)))
    return out


def test_gelu_printed_values():
    rec = read_gelu_fixture()
    for tag, z, v in rec:
        got = oracle.gelu(np.array([z]))[0]
        if tag == "teardown":
            assert round(got, 4) == v, (z, got, v)
        elif tag == "erf_form":
            # the reference computes in fp32: within one fp32 ulp of the exact value
            assert abs(got - v) <= np.spacing(np.float32(v)), (z, got, v)
        else:                                    # the tanh form is not the model's
            assert abs(got - v) > 1e-4, (z, got, v)


def test_gelu_matches_torch_exact_form():
    z = np.linspace(-8, 8, 2001)
    ref = torch.nn.functional.gelu(torch.from_numpy(z), approximate="none").numpy()
    assert np.allclose(oracle.gelu(z), ref, rtol=0, atol=2e-15)


def test_gelu_is_x_times_normal_cdf():
    z = np.array([-3.5, -1.0, -0.25, 0.5, 1.5, 4.0])
    phi = np.array([0.5 * math.erfc(-v / math.sqrt(2.0)) for v in z])  # normal CDF, another route
    assert np.allclose(oracle.gelu(z), z * phi, rtol=1e-14, atol=1e-16)


def test_zero_down_projection_returns_the_residual():
    x = rand((9, D), 1)
    w, wi, _ = weights(2)
    y = oracle.mlp(bits(x), bits(w), bits(wi), bits(torch.zeros(D, INNER)))
    assert np.array_equal(y, f64(x))


def test_selection_weights_give_gelu_times_gate():
    # Wi = [I_1152 x 768 block; 2 I block], Wo = [I; 0] (768 x 1152):
    # y = x + GELU(h) * 2h on the first 768 positions (h = LayerNorm(x)).
    # Reading the halves the other way round would give GELU(2h) * h.
    x = rand((7, D), 3)
    w = rand((D,), 4, 0.1, 1.0)
    eye_in = torch.zeros(INNER, D)
    eye_in[:D, :] = torch.eye(D)
    wi = torch.cat([eye_in, 2 * eye_in])
    wo = torch.zeros(D, INNER)
    wo[:, :D] = torch.eye(D)
    y = oracle.mlp(bits(x), bits(w), bits(wi), bits(wo))
    h = oracle.layernorm(bits(x), bits(w))
    expected = f64(x) + torch.nn.functional.gelu(torch.from_numpy(h)).numpy() * 2 * h
    assert np.allclose(y, expected, rtol=0, atol=1e-14)


def test_matches_library_composition():
    # torch: layer_norm, linear, chunk, exact gelu, linear, all in fp64
    x = rand((16, D), 5, 2.0, 0.3)
    w, wi, wo = weights(6)
    y = oracle.mlp(bits(x), bits(w), bits(wi), bits(wo))
    xt = torch.from_numpy(f64(x))
    h = torch.nn.functional.layer_norm(xt, (D,), weight=torch.from_numpy(f64(w)), eps=oracle.NORM_EPS)
    a, b = torch.nn.functional.linear(h, torch.from_numpy(f64(wi))).chunk(2, dim=-1)
    ref = xt + torch.nn.functional.linear(torch.nn.functional.gelu(a) * b, torch.from_numpy(f64(wo)))
    assert np.allclose(y, ref.numpy(), rtol=0, atol=1e-11)


def test_sampled_rows_equal_full_rows():
    x = rand((40, D), 7)
    w, wi, wo = weights(8)
    rows = np.array([0, 3, 39])
    full = oracle.mlp(bits(x), bits(w), bits(wi), bits(wo))
    part = oracle.mlp(bits(x), bits(w), bits(wi), bits(wo), rows=rows)
    assert np.array_equal(part, full[rows])
