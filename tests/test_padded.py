"""GPU parity of the padded-batch attention call (B rows of S tokens with a
0/1 attention mask) through the C ABI, against the oracle's masked form.

Same tolerance as the packed call: max |err| <= 2e-2 and mean |err| <= 2e-3
over every compared element; pad rows of the output are exactly zero.
"""
import numpy as np
import pytest
import torch

import oracle
from encoder_only_transformer_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu

WIDTH = 2304
MAX_ERR, MEAN_ERR = 2e-2, 2e-3


@pytest.fixture(scope="module")
def attn():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    h = binding.Attention(0)
    yield h
    assert h.get_error() == 0
    h.close()


def batch(B, S, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, S, WIDTH, generator=g).to(torch.bfloat16)


def masks(B, S, seed):
    """Right-padded rows of random length, a left-padded row, a row with
    holes, an all-pad row and a full row (as many as B allows)."""
    rng = np.random.default_rng(seed)
    m = np.zeros((B, S), dtype=np.int32)
    for b in range(B):
        kind = b % 5
        if kind == 0:
            m[b, :rng.integers(1, S + 1)] = 1
        elif kind == 1:
            m[b, S - rng.integers(1, S + 1):] = 1
        elif kind == 2:
            m[b] = rng.random(S) < 0.8
        elif kind == 3:
            pass                                   # all pads
        else:
            m[b] = 1
    return m


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("kind", ["global", "local"])
@pytest.mark.parametrize("B,S", [(5, 64), (5, 200), (3, 513)])
def test_parity(attn, kind, B, S):
    qkv = batch(B, S, 10 * B + S)
    m = masks(B, S, S)
    out = attn.forward_padded(qkv.cuda(), torch.from_numpy(m).cuda(), kind).cpu()
    p = oracle.KINDS[kind]
    ref = oracle.attention_padded(bits(qkv), m, p["theta"], p["half_window"])
    got = out.double().numpy()
    assert np.array_equal(got[m == 0], np.zeros_like(got[m == 0])), "pad rows must be zero"
    err = np.abs(got - ref)[m == 1]
    assert err.max() <= MAX_ERR and err.mean() <= MEAN_ERR, f"{err.max():.3e} {err.mean():.3e}"


@pytest.mark.parametrize("kind", ["global", "local"])
def test_right_padded_equals_packed_call(attn, kind):
    lengths, S = [300, 1, 129, 300], 300
    qkv = batch(len(lengths), S, 7)
    m = np.array([[1] * L + [0] * (S - L) for L in lengths], dtype=np.int32)
    out = attn.forward_padded(qkv.cuda(), torch.from_numpy(m).cuda(), kind).cpu()
    packed = torch.cat([qkv[b, :L] for b, L in enumerate(lengths)]).cuda()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32).cuda()
    ref = attn.forward(packed, cu, kind).cpu()
    o = 0
    for b, L in enumerate(lengths):
        assert torch.equal(out[b, :L], ref[o:o + L])
        o += L


def test_full_size_rows_sampled(attn):
    """Two rows of 8192 with 8192 and 3000 real tokens, a global layer, on
    sampled rows against the packed oracle (equal to the masked form by the
    oracle's pins)."""
    lengths, S = [8192, 3000], 8192
    qkv = batch(2, S, 8)
    m = np.array([[1] * L + [0] * (S - L) for L in lengths], dtype=np.int32)
    out = attn.forward_padded(qkv.cuda(), torch.from_numpy(m).cuda(), "global").cpu()
    packed = torch.cat([qkv[b, :L] for b, L in enumerate(lengths)])
    cu = np.array([0, 8192, 11192], dtype=np.int32)
    rows = np.unique(np.concatenate([np.arange(0, 11192, 211), [0, 8191, 8192, 11191]])).astype(np.int64)
    ref, _ = oracle.attention(bits(packed), cu, oracle.GLOBAL["theta"], -1, rows=rows)
    got = torch.cat([out[0, :8192], out[1, :3000]]).double().numpy()[rows]
    err = np.abs(got - ref)
    assert err.max() <= MAX_ERR and err.mean() <= MEAN_ERR, f"{err.max():.3e} {err.mean():.3e}"
    assert torch.count_nonzero(out[1, 3000:]) == 0


def test_rejects_bad_arguments(attn):
    lib = binding.load_library()
    st = binding._stream_ptr(torch.device("cuda"))
    qkv = batch(2, 16, 9).cuda()
    m = torch.ones(2, 16, dtype=torch.int32, device="cuda")
    out = torch.empty(2, 16, 768, dtype=torch.bfloat16, device="cuda")
    h = attn._h
    assert lib.mbert_attn_forward_padded(h, qkv.data_ptr(), m.data_ptr(), 2, 16, 0, out.data_ptr(), st) == 0
    assert lib.mbert_attn_forward_padded(h, qkv.data_ptr(), m.data_ptr() + 2, 2, 16, 0, out.data_ptr(), st) == -1
    assert lib.mbert_attn_forward_padded(h, qkv.data_ptr(), m.data_ptr(), 2, 16, 0, qkv.data_ptr(), st) == -1
    assert lib.mbert_attn_forward_padded(h, qkv.data_ptr(), m.data_ptr(), 1, 9000, 0, out.data_ptr(), st) == -3
    assert lib.mbert_attn_forward_padded(h, qkv.data_ptr(), m.data_ptr(), 2, 16, 7, out.data_ptr(), st) == -1
    assert lib.mbert_attn_forward_padded(h, qkv.data_ptr(), m.data_ptr(), 0, 16, 0, out.data_ptr(), st) == 0
    torch.cuda.synchronize()


def test_buffers_survive_workspace_growth():
    """The handle's buffers of the norm, the MLP and the padded call stay
    valid when a later call grows another of its workspaces (here the
    rotated-Q/K scratch, by a global layer longer than any before)."""
    h = binding.Attention(0)
    try:
        D = 768
        g = torch.Generator().manual_seed(21)
        x = torch.randn(300, D, generator=g).to(torch.bfloat16).cuda()
        nw = torch.ones(D, dtype=torch.bfloat16, device="cuda")
        wq = (torch.randn(3 * D, D, generator=g) / D ** 0.5).to(torch.bfloat16).cuda()
        wi = (torch.randn(2 * 1152, D, generator=g) / D ** 0.5).to(torch.bfloat16).cuda()
        wo = (torch.randn(D, 1152, generator=g) / 1152 ** 0.5).to(torch.bfloat16).cuda()
        qkv_p = batch(2, 40, 22).cuda()
        m = torch.ones(2, 40, dtype=torch.int32, device="cuda")
        before = (h.ln_qkv(x, nw, wq).cpu(), h.mlp(x, nw, wi, wo).cpu(),
                  h.forward_padded(qkv_p, m, "local").cpu())
        big = W.custom([8192, 8192, 4000], seed=23)          # 20384 rows: the scratch grows
        h.forward(big.qkv.cuda(), big.cu_seqlens.cuda(), "global")
        after = (h.ln_qkv(x, nw, wq).cpu(), h.mlp(x, nw, wi, wo).cpu(),
                 h.forward_padded(qkv_p, m, "local").cpu())
        torch.cuda.synchronize()
        assert h.get_error() == 0
        for a, b in zip(before, after):
            assert torch.equal(a, b)
    finally:
        h.close()
