"""GPU parity of the output projection with the residual add, y = x + a Wo^T,
through the C ABI, against the fp64 oracle on the same seeded inputs.

Tolerance as for the attention block: max |err| <= 2e-2 and mean |err| <=
2e-3 over every compared element (bf16 inputs, fp32 accumulation, bf16 y).
"""
import numpy as np
import pytest
import torch

import oracle
from encoder_only_transformer_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu

D = 768
MAX_ERR = 2e-2
MEAN_ERR = 2e-3


@pytest.fixture(scope="module")
def attn():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    h = binding.Attention(0)
    yield h
    assert h.get_error() == 0
    h.close()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def inputs(T, seed):
    g = torch.Generator().manual_seed(seed)
    a = (torch.randn(T, D, generator=g) * 0.5).to(torch.bfloat16)
    wo = (torch.randn(D, D, generator=g) * (1.0 / D ** 0.5)).to(torch.bfloat16)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16)
    return a, wo, x


def compare(y_gpu, ref, what):
    got = y_gpu.cpu().double().numpy()
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert err.max() <= MAX_ERR and err.mean() <= MEAN_ERR, \
        f"{what}: max|err| {err.max():.3e} mean|err| {err.mean():.3e}"


@pytest.mark.parametrize("T", [1, 127, 128, 129, 300, 1000])
def test_parity_full(attn, T):
    a, wo, x = inputs(T, 100 + T)
    y = attn.out_proj(a.cuda(), wo.cuda(), x.cuda())
    torch.cuda.synchronize()
    assert attn.get_error() == 0
    compare(y, oracle.out_proj(bits(a), bits(wo), bits(x)), f"T={T}")


def test_in_place_equals_out_of_place(attn):
    a, wo, x = inputs(777, 5)
    ad, wd, xd = a.cuda(), wo.cuda(), x.cuda()
    y = attn.out_proj(ad, wd, xd)
    attn.out_proj(ad, wd, xd, out=xd)
    torch.cuda.synchronize()
    assert torch.equal(xd, y)


def test_permutation_weight(attn):
    g = torch.Generator().manual_seed(9)
    perm = torch.randperm(D, generator=g)
    wo = torch.zeros(D, D)
    wo[torch.arange(D), perm] = 1.0
    a, _, x = inputs(260, 10)
    y = attn.out_proj(a.cuda(), wo.to(torch.bfloat16).cuda(), x.cuda())
    torch.cuda.synchronize()
    # one exact product per output plus x, rounded once to bf16
    exp = (x.double() + a.double()[:, perm]).to(torch.bfloat16)
    assert torch.equal(y.cpu(), exp)


@pytest.mark.parametrize("cfg", [3, 4])
def test_full_size_sampled(attn, cfg):
    T = W.config(cfg).T
    a, wo, x = inputs(T, 200 + cfg)
    y = attn.out_proj(a.cuda(), wo.cuda(), x.cuda())
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, T, 97), [0, T - 1]])).astype(np.int64)
    ref = oracle.out_proj(bits(a), bits(wo), bits(x), rows=rows)
    compare(y.cpu()[torch.from_numpy(rows)], ref, f"config{cfg} sampled")


def test_after_attention(attn):
    """The attention block then the projection (config 2, a local layer),
    against the oracle's attention output rounded to bf16 and projected."""
    wl = W.config(2)
    g = torch.Generator().manual_seed(77)
    wo = (torch.randn(D, D, generator=g) * (1.0 / D ** 0.5)).to(torch.bfloat16)
    x = torch.randn(wl.T, D, generator=g).to(torch.bfloat16)
    out = attn.forward(wl.qkv.cuda(), wl.cu_seqlens.cuda(), "local")
    y = attn.out_proj(out, wo.cuda(), x.cuda())
    torch.cuda.synchronize()
    ref_a, _ = oracle.attention_kind(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), "local")
    a_bf16 = torch.from_numpy(ref_a).to(torch.bfloat16)
    compare(y, oracle.out_proj(bits(a_bf16), bits(wo), bits(x)), "attention then projection")


def test_rejects_bad_buffers(attn):
    a, wo, x = inputs(64, 3)
    ad, wd, xd = a.cuda(), wo.cuda(), x.cuda()
    lib = binding.load_library()
    st = torch.cuda.current_stream().cuda_stream
    # y overlapping a, and a misaligned y
    assert lib.mbert_attn_out_proj(attn._h, ad.data_ptr(), wd.data_ptr(), xd.data_ptr(), 64,
                                   ad.data_ptr(), st) == -1
    buf = torch.empty(64 * D + 8, dtype=torch.bfloat16, device="cuda")
    assert lib.mbert_attn_out_proj(attn._h, ad.data_ptr(), wd.data_ptr(), xd.data_ptr(), 64,
                                   buf.data_ptr() + 2, st) == -1
    assert lib.mbert_attn_out_proj(attn._h, ad.data_ptr(), wd.data_ptr(), xd.data_ptr(), 0,
                                   buf.data_ptr(), st) == 0
