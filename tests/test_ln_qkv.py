"""GPU parity of the pre-attention LayerNorm and fused Wqkv projection,
qkv = LayerNorm(x) Wqkv^T, through the C ABI, against the fp64 oracle on the
same seeded inputs.

Tolerance, derived from the arithmetic: the GPU rounds the norm's output to
bf16 (the GEMM operand, relative error <= 2^-9 per element), accumulates in
fp32 and rounds qkv to bf16 (relative 2^-9), so an element's error scales
with its size: with e = |err| / max(1, |ref|), e <= 2e-2 for every element
and mean(e) <= 2e-3, the attention block's bounds applied relative to the
size of the result.
"""
import numpy as np
import pytest
import torch

import oracle
from encoder_only_transformer_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu

D = 768
N_OUT = 3 * D
REL_ERR = 2e-2
MEAN_ERR = 2e-3
ATT_MAX, ATT_MEAN = 2e-2, 2e-3


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
    """x ~ 2 N(0, 1) + 0.5 (a non-zero mean for the norm to remove), a norm
    weight near 1 (1 + 0.1 N(0, 1)), Wqkv ~ N(0, 1/768)."""
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(T, D, generator=g) * 2.0 + 0.5).to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    wq = (torch.randn(N_OUT, D, generator=g) * D ** -0.5).to(torch.bfloat16)
    return x, w, wq


def compare(got_t, ref, what):
    got = got_t.cpu().double().numpy()
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    e = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    assert e.max() <= REL_ERR and e.mean() <= MEAN_ERR, \
        f"{what}: max e {e.max():.3e} mean e {e.mean():.3e} (e = |err| / max(1, |ref|))"


@pytest.mark.parametrize("T", [1, 127, 128, 129, 300, 1000])
def test_parity_full(attn, T):
    x, w, wq = inputs(T, 100 + T)
    qkv = attn.ln_qkv(x.cuda(), w.cuda(), wq.cuda())
    torch.cuda.synchronize()
    compare(qkv, oracle.ln_qkv(bits(x), bits(w), bits(wq)), f"T={T}")


@pytest.mark.parametrize("T", [1, 300])
def test_identity_norm_of_layer_zero(attn, T):
    x, _, wq = inputs(T, 7)
    qkv = attn.ln_qkv(x.cuda(), None, wq.cuda())
    torch.cuda.synchronize()
    compare(qkv, oracle.ln_qkv(bits(x), None, bits(wq)), f"identity T={T}")


def test_selection_weights_reproduce_the_norm(attn):
    # Wqkv = [I; 2I; -I]: q = bf16(h), k = 2 bf16(h), v = -bf16(h) exactly,
    # h the GPU's normalised rows; h itself within bf16 of the oracle
    T = 257
    x, w, _ = inputs(T, 8)
    eye = torch.eye(D)
    wq = torch.cat([eye, 2 * eye, -eye]).to(torch.bfloat16)
    qkv = attn.ln_qkv(x.cuda(), w.cuda(), wq.cuda()).cpu()
    q, k, v = qkv[:, :D], qkv[:, D:2 * D], qkv[:, 2 * D:]
    assert torch.equal(k.float(), 2 * q.float()) and torch.equal(v.float(), -q.float())
    compare(q, oracle.layernorm(bits(x), bits(w)), "normalised rows")


@pytest.mark.parametrize("cfg", [3, 4])
def test_full_size_sampled(attn, cfg):
    T = W.config(cfg).T
    x, w, wq = inputs(T, 200 + cfg)
    qkv = attn.ln_qkv(x.cuda(), w.cuda(), wq.cuda())
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, T, 97), [0, T - 1]])).astype(np.int64)
    ref = oracle.ln_qkv(bits(x), bits(w), bits(wq), rows=rows)
    compare(qkv.cpu()[torch.from_numpy(rows)], ref, f"config{cfg} sampled")


def test_then_attention(attn):
    """The norm and projection, then the attention block (config 2's pack, a
    local layer), against the oracle's qkv rounded to bf16 then its
    attention."""
    wl = W.config(2)
    x, w, wq = inputs(wl.T, 9)
    qkv = attn.ln_qkv(x.cuda(), w.cuda(), wq.cuda())
    out = attn.forward(qkv, wl.cu_seqlens.cuda(), "local")
    torch.cuda.synchronize()
    qkv_ref = torch.from_numpy(oracle.ln_qkv(bits(x), bits(w), bits(wq))).to(torch.bfloat16)
    ref, _ = oracle.attention_kind(bits(qkv_ref), wl.cu_seqlens.numpy(), "local")
    err = np.abs(out.cpu().double().numpy() - ref)
    assert err.max() <= ATT_MAX and err.mean() <= ATT_MEAN, \
        f"max|err| {err.max():.3e} mean|err| {err.mean():.3e}"


def test_rejects_bad_buffers(attn):
    lib = binding.load_library()
    T = 256
    x, w, wq = [t.cuda() for t in inputs(T, 10)]
    qkv = torch.empty(T, N_OUT, dtype=torch.bfloat16, device="cuda")
    st = binding._stream_ptr(x.device)
    h = attn._h
    assert lib.mbert_attn_ln_qkv(h, x.data_ptr(), w.data_ptr(), wq.data_ptr(), 0, 1e-5,
                                 qkv.data_ptr(), st) == 0
    big = torch.empty(T, N_OUT + D, dtype=torch.bfloat16, device="cuda")
    # qkv overlapping x
    assert lib.mbert_attn_ln_qkv(h, big.data_ptr(), w.data_ptr(), wq.data_ptr(), T, 1e-5,
                                 big.data_ptr() + 2 * D, st) == -1
    # misaligned output
    assert lib.mbert_attn_ln_qkv(h, x.data_ptr(), w.data_ptr(), wq.data_ptr(), T, 1e-5,
                                 qkv.data_ptr() + 2, st) == -1
    # bad eps
    assert lib.mbert_attn_ln_qkv(h, x.data_ptr(), w.data_ptr(), wq.data_ptr(), T, -1.0,
                                 qkv.data_ptr(), st) == -1
    assert lib.mbert_attn_ln_qkv(h, x.data_ptr(), w.data_ptr(), wq.data_ptr(), T, float("nan"),
                                 qkv.data_ptr(), st) == -1
    torch.cuda.synchronize()
