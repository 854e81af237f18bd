"""The allocation-free entry point, mbert_attn_forward_noalloc.

Callers that cannot call cudaMalloc (a plugin inside a framework that owns
the device memory pool, a service whose memory is fixed at start-up, a loop
that cannot afford the synchronisation an allocation may cause) use it
instead of a handle; its scratch lives in a static device array.  These
tests call it through the C ABI, twice in a row, and compare its output with
the fp64 oracle and with the handle-based mbert_attn_forward, each within the
parity tolerance used everywhere else (max |err| <= 2e-2, mean |err| <=
2e-3).  The file is named to be collected last, and it builds what it needs,
so it passes both alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
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


def _oracle_close(got, wl, kind, rows=None):
    exp, _ = oracle.attention_kind(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), kind, rows=rows)
    g = got.cpu().double().numpy()
    if rows is not None:
        g = g[rows]
    err = np.abs(g - exp)
    return err.max() <= MAX_ERR and err.mean() <= MEAN_ERR, (err.max(), err.mean())


@pytest.mark.parametrize("kind", ["global", "local"])
def test_noalloc_matches_oracle_and_forward_two_calls(ref, kind):
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
            ok, errs = _oracle_close(out, wl, kind)
            assert ok, f"{wl.name} {kind} against the oracle: {errs}"
            assert _close(out, expect), f"{wl.name} {kind} against forward"
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
    ok, errs = _oracle_close(out, wl, "local")
    assert ok, errs


def test_noalloc_reports_a_sequence_longer_than_max_seqlen(ref):
    """max_seqlen below a real length: the call is accepted on the host, the
    device check sets bit 2 in the status and nothing is written."""
    wl = W.custom([300, 40], seed=6)
    qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
    for kind in ("global", "local"):
        out = torch.full((wl.T, 768), 7.0, dtype=torch.bfloat16, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(qkv, cu, kind, out, status, max_seqlen=200) == 0
        torch.cuda.synchronize()
        assert int(status.item()) & 2
        assert torch.all(out == 7.0)


def test_noalloc_rejects_sizes_beyond_limit(ref):
    wl = W.custom([LIMIT + 1], seed=8)
    qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
    out = torch.empty(LIMIT + 1, 768, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(qkv, cu, "global", out, None) == -1
    many = torch.zeros(LIMIT + 2, dtype=torch.int32, device="cuda")
    assert _noalloc(qkv, many, "global", out, None, n_seqs=LIMIT + 1, T=0) == -1
    assert _noalloc(qkv, cu, "global", out, None, T=LIMIT, max_seqlen=LIMIT + 1) == -3


@pytest.mark.parametrize("kind", ["global", "local"])
def test_noalloc_at_the_limit(ref, kind):
    """One sequence of exactly MBERT_NOALLOC_MAX_TOKENS tokens: status 0 and
    the oracle's values (every row on a local layer, a seeded sample of 512
    rows on a global layer)."""
    wl = W.custom([LIMIT], seed=9)
    qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
    out = torch.full((LIMIT, 768), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    assert _noalloc(qkv, cu, kind, out, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = None if kind == "local" else W.sample_rows(wl.cu_seqlens, 512, seed=10)
    ok, errs = _oracle_close(out, wl, kind, rows=rows)
    assert ok, f"{kind} at {LIMIT} tokens: {errs}"
    assert _close(out, ref.forward(qkv, cu, kind))
