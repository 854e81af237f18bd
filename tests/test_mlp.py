"""GPU parity of the GeGLU MLP block, y = x + (GELU(g) * u) Wo^T with g, u
the halves of LayerNorm(x) Wi^T, and of a whole encoder layer built from the
library's calls, through the C ABI, against the fp64 oracle.

Tolerance as for the other GEMM steps: with e = |err| / max(1, |ref|),
e <= 2e-2 for every element and mean(e) <= 2e-3 (bf16 rounding of the norm's
output, of GELU(g) * u and of y is relative to the size of each value).
"""
import numpy as np
import pytest
import torch

import oracle
from encoder_only_transformer_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu

D = 768
INNER = 1152
REL_ERR = 2e-2
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
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def mlp_weights(seed):
    g = torch.Generator().manual_seed(seed)
    w = (1.0 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    wi = (torch.randn(2 * INNER, D, generator=g) * D ** -0.5).to(torch.bfloat16)
    wo = (torch.randn(D, INNER, generator=g) * INNER ** -0.5).to(torch.bfloat16)
    return w, wi, wo


def rows_x(T, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(T, D, generator=g) * 2.0 + 0.5).to(torch.bfloat16)


def compare(got_t, ref, what):
    got = got_t.cpu().double().numpy()
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    e = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    assert e.max() <= REL_ERR and e.mean() <= MEAN_ERR, \
        f"{what}: max e {e.max():.3e} mean e {e.mean():.3e} (e = |err| / max(1, |ref|))"


@pytest.mark.parametrize("T", [1, 127, 128, 129, 300, 1000])
def test_parity_full(attn, T):
    x = rows_x(T, 300 + T)
    w, wi, wo = mlp_weights(31)
    y = attn.mlp(x.cuda(), w.cuda(), wi.cuda(), wo.cuda())
    torch.cuda.synchronize()
    compare(y, oracle.mlp(bits(x), bits(w), bits(wi), bits(wo)), f"T={T}")


def test_in_place_equals_out_of_place(attn):
    T = 777
    x = rows_x(T, 32).cuda()
    w, wi, wo = [t.cuda() for t in mlp_weights(33)]
    y = attn.mlp(x, w, wi, wo)
    x2 = x.clone()
    attn.mlp(x2, w, wi, wo, out=x2)
    torch.cuda.synchronize()
    assert torch.equal(x2, y)


@pytest.mark.parametrize("cfg", [3, 4])
def test_full_size_sampled(attn, cfg):
    T = W.config(cfg).T
    x = rows_x(T, 400 + cfg)
    w, wi, wo = mlp_weights(34)
    y = attn.mlp(x.cuda(), w.cuda(), wi.cuda(), wo.cuda())
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, T, 97), [0, T - 1]])).astype(np.int64)
    ref = oracle.mlp(bits(x), bits(w), bits(wi), bits(wo), rows=rows)
    compare(y.cpu()[torch.from_numpy(rows)], ref, f"config{cfg} sampled")


@pytest.mark.parametrize("kind", ["global", "local"])
def test_whole_encoder_layer(attn, kind):
    """x -> qkv = LN(x) Wqkv^T -> attention -> x1 = x + a Wo^T -> y = x1 +
    MLP(x1), on config 2's pack (8 sequences).  Each step is checked against
    the oracle applied to the GPU's own input to that step, at that step's
    bound; the result is also checked against the oracle's steps chained
    independently, at the sum of the four steps' bounds (each step passes an
    earlier error on with a gain of about 1: the norms rescale to unit
    spread, attention averages, the weights keep the scale)."""
    wl = W.config(2)
    T = wl.T
    g = torch.Generator().manual_seed(35)
    x = rows_x(T, 36)
    wn = (1.0 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    wqkv = (torch.randn(3 * D, D, generator=g) * D ** -0.5).to(torch.bfloat16)
    wo_a = (torch.randn(D, D, generator=g) * D ** -0.5).to(torch.bfloat16)
    mw, wi, wo = mlp_weights(37)
    cu = wl.cu_seqlens.cuda()
    xg = x.cuda()
    qkv = attn.ln_qkv(xg, wn.cuda(), wqkv.cuda())
    a = attn.forward(qkv, cu, kind)
    x1 = attn.out_proj(a, wo_a.cuda(), xg)
    y = attn.mlp(x1, mw.cuda(), wi.cuda(), wo.cuda())
    torch.cuda.synchronize()
    qkv, a, x1 = qkv.cpu(), a.cpu(), x1.cpu()
    cu_np = wl.cu_seqlens.numpy()

    # step by step, each on the GPU's own input
    compare(qkv, oracle.ln_qkv(bits(x), bits(wn), bits(wqkv)), f"{kind}: ln_qkv")
    a_ref, _ = oracle.attention_kind(bits(qkv), cu_np, kind)
    err = np.abs(a.double().numpy() - a_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, f"{kind}: attention {err.max():.3e} {err.mean():.3e}"
    compare(x1, oracle.out_proj(bits(a), bits(wo_a), bits(x)), f"{kind}: out_proj")
    compare(y, oracle.mlp(bits(x1), bits(mw), bits(wi), bits(wo)), f"{kind}: mlp")

    # end to end against the independent chain
    def bf(v):
        return torch.from_numpy(v).to(torch.bfloat16)
    qkv_r = bf(oracle.ln_qkv(bits(x), bits(wn), bits(wqkv)))
    a_r, _ = oracle.attention_kind(bits(qkv_r), cu_np, kind)
    x1_r = bf(oracle.out_proj(bits(bf(a_r)), bits(wo_a), bits(x)))
    y_r = oracle.mlp(bits(x1_r), bits(mw), bits(wi), bits(wo))
    got = y.cpu().double().numpy()
    e = np.abs(got - y_r) / np.maximum(1.0, np.abs(y_r))
    assert e.max() <= 4 * REL_ERR and e.mean() <= 4 * MEAN_ERR, \
        f"{kind} layer end to end: max e {e.max():.3e} mean e {e.mean():.3e}"


def test_rejects_bad_buffers(attn):
    lib = binding.load_library()
    T = 256
    x = rows_x(T, 38).cuda()
    w, wi, wo = [t.cuda() for t in mlp_weights(39)]
    y = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
    st = binding._stream_ptr(x.device)
    h = attn._h
    call = lambda xp, wp, yp, eps=1e-5: lib.mbert_attn_mlp(h, xp, wp, wi.data_ptr(), wo.data_ptr(),
                                                          T, eps, yp, st)
    assert call(x.data_ptr(), w.data_ptr(), y.data_ptr()) == 0
    assert call(x.data_ptr(), None, y.data_ptr()) == -1                  # the MLP norm is not optional
    assert call(x.data_ptr(), w.data_ptr(), x.data_ptr() + 2 * D) == -1  # y partly over x
    assert call(x.data_ptr(), w.data_ptr(), wi.data_ptr()) == -1         # y over a weight
    assert call(x.data_ptr(), w.data_ptr(), y.data_ptr() + 2) == -1      # misaligned
    assert call(x.data_ptr(), w.data_ptr(), y.data_ptr(), -1.0) == -1
    torch.cuda.synchronize()
