"""The library's calls inside a CUDA graph: after warm-up calls have sized
the handle's buffers, a captured sequence of calls (the prologue, both
attention kinds, the projection and the MLP) replays on new inputs with
results equal bit for bit to the same calls run eagerly."""
import pytest
import torch

from encoder_only_transformer_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu

D = 768


@pytest.fixture(scope="module")
def attn():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    h = binding.Attention(0)
    yield h
    assert h.get_error() == 0
    h.close()


def test_captured_layer_replays_bit_equal(attn):
    wl = W.config(2)
    T = wl.T
    g = torch.Generator().manual_seed(51)
    mk = lambda *s, sc=1.0: (torch.randn(*s, generator=g) * sc).to(torch.bfloat16).cuda()
    nw, mw = mk(D, sc=0.1) + 1, mk(D, sc=0.1) + 1
    wqkv, wo = mk(3 * D, D, sc=D ** -0.5), mk(D, D, sc=D ** -0.5)
    wi, wo2 = mk(2 * 1152, D, sc=D ** -0.5), mk(D, 1152, sc=1152 ** -0.5)
    cu = wl.cu_seqlens.cuda()
    x = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
    qkv = torch.empty(T, 3 * D, dtype=torch.bfloat16, device="cuda")
    a_g = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
    a_l = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
    x1 = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")

    def layer():
        attn.ln_qkv(x, nw, wqkv, out=qkv)
        attn.forward(qkv, cu, "global", out=a_g)
        attn.forward(qkv, cu, "local", out=a_l)
        attn.out_proj(a_g, wo, x, out=x1)
        attn.mlp(x1, mw, wi, wo2, out=y)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        x.copy_(mk(T, D))
        layer()                                   # warm-up: sizes every buffer
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer()
    for trial in range(2):
        x.copy_(mk(T, D))
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (qkv, a_g, a_l, x1, y)]
        layer()
        torch.cuda.synchronize()
        for name, a, b in zip(("qkv", "global", "local", "x1", "y"), got, (qkv, a_g, a_l, x1, y)):
            assert torch.equal(a, b), f"replay {trial}: {name} differs from the eager call"
    assert attn.get_error() == 0
