"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.

Tolerance (floating point): max |err| <= 2e-2 and mean |err| <= 2e-3 over
every compared element, with the bf16 GPU output widened to fp64 and the
oracle left unrounded.  Integer work (admitted-key counts of the tile
schedule and mask) is compared bit-exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from encoder_only_transformer_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu

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


def _run(attn, wl, kind):
    qkv = wl.qkv.cuda()
    cu = wl.cu_seqlens.cuda()
    out = attn.forward(qkv, cu, kind)
    torch.cuda.synchronize()
    assert attn.get_error() == 0
    return out.cpu()


def _compare(got_bf16, ref, what):
    got = got_bf16.double().numpy()
    assert got.shape == ref.shape
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert err.max() <= MAX_ERR and err.mean() <= MEAN_ERR, \
        f"{what}: max|err| {err.max():.3e} mean|err| {err.mean():.3e}"
    return err


def _full_check(attn, wl, kind):
    out = _run(attn, wl, kind)
    ref, counts = oracle.attention_kind(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), kind)
    _compare(out, ref, f"{wl.name} {kind}")
    gc = attn.key_counts(wl.cu_seqlens.cuda(), wl.T, kind).cpu().numpy()
    np.testing.assert_array_equal(gc, counts)
    return out


def _sampled_check(attn, wl, kind, per_seq, seed):
    out = _run(attn, wl, kind)
    rows = W.sample_rows(wl.cu_seqlens, per_seq, seed)
    ref, counts = oracle.attention_kind(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), kind, rows=rows)
    _compare(out[torch.from_numpy(rows)], ref, f"{wl.name} {kind} sampled")
    gc = attn.key_counts(wl.cu_seqlens.cuda(), wl.T, kind).cpu().numpy()
    np.testing.assert_array_equal(gc, oracle.key_counts(wl.cu_seqlens.numpy(),
                                                        oracle.KINDS[kind]["half_window"]))
    return out


# ---------------------------------------------------------------------------
# small workloads: every row against the oracle
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", [1, 2])
@pytest.mark.parametrize("kind", ["global", "local"])
def test_small_configs_full(attn, cfg, kind):
    _full_check(attn, W.config(cfg), kind)


EDGE_PACKS = {
    "len1": [1],
    "tile_edges": [127, 128, 129],
    "two_tiles_ragged": [255, 256, 257],
    "window_edges": [64, 65, 66, 193, 194],
    "empties": [0, 5, 0, 300, 0],
    "long_ragged": [1000, 3, 777],
}


@pytest.mark.parametrize("name", list(EDGE_PACKS))
@pytest.mark.parametrize("kind", ["global", "local"])
def test_edge_packs(attn, name, kind):
    _full_check(attn, W.custom(EDGE_PACKS[name], seed=len(name) * 7 + 3), kind)


@pytest.mark.parametrize("kind", ["global", "local"])
def test_many_tiny_sequences(attn, kind):
    g = torch.Generator().manual_seed(77)
    lengths = torch.randint(1, 21, (300,), generator=g).tolist()
    _full_check(attn, W.custom(lengths, seed=78), kind)


@pytest.mark.parametrize("seed", range(12))
def test_global_split_schedules(attn, seed):
    """Seeded packs of 2-60 sequences of 1-3000 tokens: the global kernel's
    split of iterations among CTAs cuts units at every kind of place
    (segments of one or two tiles, a CTA ending a unit's first tile, many
    segment ends in a row), where its waits between the softmax groups
    and the issuers must all complete: no device error, and sampled rows
    against the oracle."""
    g = torch.Generator().manual_seed(900 + seed)
    n = int(torch.randint(2, 61, (1,), generator=g))
    hi = [20, 300, 3000][seed % 3]
    lengths = torch.randint(1, hi + 1, (n,), generator=g).tolist()
    _sampled_check(attn, W.custom(lengths, seed=950 + seed), "global", per_seq=8, seed=seed)


@pytest.mark.parametrize("lengths", [[1024], [1025], [1280], [1025, 3, 257, 640]])
def test_global_split_weighting_edge(attn, lengths):
    """The global kernel splits its iterations into ranges of equal cost,
    counting each unit start inside a range as extra iterations, but only
    where every range stays non-empty.  On 152 CTAs a single sequence of 1024
    tokens (4 query blocks) falls back to ranges of equal iterations and one
    of 1025 (5 blocks) is the first to be weighted; 1280 and the mixed pack
    put range starts between units, including at entry boundaries.  Sampled
    rows against the oracle on both sides."""
    _sampled_check(attn, W.custom(lengths, seed=960 + sum(lengths)), "global", per_seq=96, seed=7)


@pytest.mark.parametrize("kind", ["global", "local"])
def test_length_one_returns_value_exactly(attn, kind):
    wl = W.custom([1, 1, 3, 1], seed=5)
    out = _run(attn, wl, kind)
    v = wl.qkv[:, 1536:]
    for r in (0, 1, 5):
        assert torch.equal(out[r], v[r])


# ---------------------------------------------------------------------------
# the full-size workloads (sampled rows where the oracle would take long)
# ---------------------------------------------------------------------------

def test_config3_local_full(attn):
    _full_check(attn, W.config(3), "local")


def test_config3_global_sampled(attn):
    _sampled_check(attn, W.config(3), "global", per_seq=384, seed=31)


@pytest.mark.parametrize("kind", ["global", "local"])
def test_config4_sampled(attn, kind):
    _sampled_check(attn, W.config(4), kind, per_seq=24, seed=41)


@pytest.mark.parametrize("layer", [0, 1])
def test_config5_layer_sampled(attn, layer):
    wl = W.config(5, layer=layer)
    _sampled_check(attn, wl, W.layer_kind(layer), per_seq=8, seed=50 + layer)


# ---------------------------------------------------------------------------
# properties that hold at any size
# ---------------------------------------------------------------------------

def _same(a, b, kind):
    """Local layers process each sequence on its own: bit-identical.  The
    global kernel splits the whole batch's work evenly among the SMs, so
    where a sequence's work is cut (and partial results merged) depends on
    the rest of the pack: equal up to rounding."""
    if kind == "local":
        assert torch.equal(a, b)
    else:
        d = (a.double() - b.double()).abs()
        assert d.max().item() <= 1e-2 and d.mean().item() <= 1e-4


@pytest.mark.parametrize("kind", ["global", "local"])
def test_pad_sequence_leaves_real_rows_unchanged(attn, kind):
    """A padded token packed as its own sequence does not change the real
    outputs (gap 0)."""
    real = W.custom([300, 41], seed=9)
    padded = W.custom([300, 41, 5], seed=9)
    a = _run(attn, real, kind)
    b = _run(attn, padded, kind)
    _same(a, b[:341], kind)


@pytest.mark.parametrize("kind", ["global", "local"])
def test_offset_in_pack_does_not_matter(attn, kind):
    a = W.custom([333], seed=91)
    b = W.custom([150], seed=92)
    pack = W.Workload("pack", 0, 1.0, [150, 333], [kind], torch.cat([b.qkv, a.qkv]),
                      W.cu_from_lengths([150, 333]))
    alone = _run(attn, a, kind)
    packed = _run(attn, pack, kind)
    _same(alone, packed[150:], kind)


@pytest.mark.parametrize("kind", ["global", "local"])
def test_deterministic(attn, kind):
    wl = W.config(2)
    assert torch.equal(_run(attn, wl, kind), _run(attn, wl, kind))


def test_global_equals_wide_band(attn):
    """A handle whose band covers every sequence gives the global result on
    its local layers when both use the same base.  Global and local layers
    run different kernels (different fp32 summation orders), so the two are
    compared within the parity tolerance, and each against the oracle."""
    wide = binding.Attention(0, half_window=128, theta_local=160000.0)
    try:
        wl = W.custom([100, 129, 7], seed=13)   # every |i - j| <= 128
        g = _run(attn, wl, "global")
        qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
        w = wide.forward(qkv, cu, "local").cpu()
        assert wide.get_error() == 0
        _compare(w, g.double().numpy(), "wide band vs global")
        ref, _ = oracle.attention(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), 160000.0, -1)
        _compare(g, ref, "global")
        _compare(w, ref, "wide band")
        gc = wide.key_counts(cu, wl.T, "local").cpu().numpy()
        np.testing.assert_array_equal(gc, oracle.key_counts(wl.cu_seqlens.numpy(), -1))
    finally:
        wide.close()


def test_no_write_outside_output(attn):
    """Every output row is written and nothing past the end of out is."""
    wl = W.custom([200, 1, 300], seed=17)
    qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
    buf = torch.full((wl.T + 64, 768), float("nan"), dtype=torch.bfloat16, device="cuda")
    for kind in ("global", "local"):
        buf.fill_(float("nan"))
        attn.forward(qkv, cu, kind, out=buf[:wl.T])
        torch.cuda.synchronize()
        assert torch.isfinite(buf[:wl.T].float()).all()
        assert torch.isnan(buf[wl.T:].float()).all()


def test_runs_on_a_side_stream(attn):
    wl = W.config(1)
    qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
    ref = attn.forward(qkv, cu, "global").cpu()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = attn.forward(qkv, cu, "global")
    s.synchronize()
    assert torch.equal(out.cpu(), ref)


def test_module_level_function(attn):
    wl = W.config(1)
    out = binding.attention(wl.qkv.cuda(), wl.cu_seqlens.cuda(), "local")
    torch.cuda.synchronize()
    ref, _ = oracle.attention_kind(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), "local")
    _compare(out.cpu(), ref, "module attention")


@pytest.mark.parametrize("thetas", [(150000.0, 160000.0), (80000.0, 10000.0)])
def test_sibling_checkpoint_bases(thetas):
    """Checkpoints of the same shape whose RoPE bases differ ("ModernBertModel"
    (safebydesign), "Implementing it": one lists 150000 global / 160000 local,
    another 80000 / 10000) run through the same kernels with the bases in the
    handle's configuration."""
    tg, tl = thetas
    h = binding.Attention(0, theta_global=tg, theta_local=tl)
    try:
        wl = W.config(2)
        qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
        for kind, theta in (("global", tg), ("local", tl)):
            got = h.forward(qkv, cu, kind).cpu()
            ref, _ = oracle.attention(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), theta,
                                      oracle.KINDS[kind]["half_window"])
            _compare(got, ref, f"{kind} theta {theta}")
        assert h.get_error() == 0
    finally:
        h.close()
