"""The allocation-free entry point, mbert_attn_forward_noalloc.

Callers that cannot call cudaMalloc (a plugin inside a framework that owns
the device memory pool, a service whose memory is fixed at start-up, a loop
that cannot afford the synchronisation an allocation may cause) use it
instead of a handle; its scratch lives in a static device array.  These
tests call it through the C ABI, twice in a row, and compare its output with
the handle-based mbert_attn_forward within the parity tolerance used
everywhere else (max |err| <= 2e-2, mean |err| <= 2e-3).  The file is named
to be collected last, and it builds what it needs, so it passes both alone
in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

from encoder_only_transformer_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu

MAX_ERR = 2e-2
MEAN_ERR = 2e-3
LIMIT = 8192   # MBERT_NOALLOC_MAX_TOKENS


@pytest.fixture(scope="module")
def ref():
    import __graft_entry__
    __graft_entry__.build()
    h = binding.Attention(0)
    yield h
    h.close()


def _noalloc(qkv, cu, kind, out, status, n_seqs=None, T=None, max_seqlen=0):
    lib = binding.load_library()
    return lib.mbert_attn_forward_noalloc(
        qkv.data_ptr(), cu.data_ptr(), cu.numel() - 1 if n_seqs is None else n_seqs,
        qkv.shape[0] if T is None else T, max_seqlen, binding._kind(kind), out.data_ptr(),
        status.data_ptr() if status is not None else None,
        torch.cuda.current_stream().cuda_stream)


def _close(a, b):
    d = (a.double() - b.double()).abs()
    return d.max().item() <= MAX_ERR and d.mean().item() <= MEAN_ERR


@pytest.mark.parametrize("kind", ["global", "local"])
def test_noalloc_matches_forward_two_calls(ref, kind):
    for wl in (W.config(2), W.custom([300, 1, 129, 4000, 77], seed=404)):
        qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
        expect = ref.forward(qkv, cu, kind)
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        for _ in range(2):                         # two calls in a row
            out = torch.full_like(expect, float("nan"))
            status.fill_(-1)
            assert _noalloc(qkv, cu, kind, out, status) == 0
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert _close(out, expect), f"{wl.name} {kind}"
        assert ref.get_error() == 0


def test_noalloc_reports_device_errors_per_call(ref):
    wl = W.custom([100], seed=3)
    qkv = wl.qkv.cuda()
    out = torch.empty(100, 768, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([0, 60, 50, 100], dtype=torch.int32, device="cuda")
    assert _noalloc(qkv, bad, "local", out, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    good = wl.cu_seqlens.cuda()
    assert _noalloc(qkv, good, "local", out, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert _close(out, ref.forward(qkv, good, "local"))


def test_noalloc_rejects_sizes_beyond_limit(ref):
    wl = W.custom([LIMIT + 1], seed=8)
    qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
    out = torch.empty(LIMIT + 1, 768, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(qkv, cu, "global", out, None) == -1
    many = torch.zeros(LIMIT + 2, dtype=torch.int32, device="cuda")
    assert _noalloc(qkv, many, "global", out, None, n_seqs=LIMIT + 1, T=0) == -1
    assert _noalloc(qkv, cu, "global", out, None, T=LIMIT, max_seqlen=LIMIT + 1) == -3
    # at the limit it runs
    wl = W.custom([LIMIT], seed=9)
    qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
    out = torch.empty(LIMIT, 768, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(qkv, cu, "local", out, None) == 0
    assert _close(out, ref.forward(qkv, cu, "local"))
