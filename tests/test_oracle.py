"""Pins of the fp64 oracle against what the pages and mathematics fix.

Each test names the passage it follows.  None of them compares the oracle
with itself: the expected values are the pages' printed numbers, closed
forms, invariants of the definition, or independent brute-force formulations
(numpy dense scores with an explicit mask and complex-number RoPE; torch
float64 scaled_dot_product_attention with a boolean mask).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from encoder_only_transformer_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------------------
# independent brute-force formulations (used on tiny inputs only)
# ---------------------------------------------------------------------------

def _heads_view(qkv_bf16):
    """(3, 12, 64) view of every row, as the teardown's "How Does ModernBERT
    Make Q, K and V?" cuts the Wqkv output: view(..., 3, 12, 64).unbind."""
    x = qkv_bf16.double().view(-1, 3, 12, 64)
    q, k, v = x.unbind(dim=1)
    return q.numpy(), k.numpy(), v.numpy()


def _rope_complex(x, pos, theta):
    """RoPE written as complex multiplication: pair m = x[m] + i x[m+32] is
    multiplied by exp(i * pos * theta^(-2m/64))."""
    m = np.arange(32, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta ** (-2.0 * m / 64.0)[None, :]
    z = (x[:, :32] + 1j * x[:, 32:]) * np.exp(1j * ang)
    return np.concatenate([z.real, z.imag], axis=1)


def _band_mask(L, half_window):
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    if half_window < 0:
        return np.ones((L, L), dtype=bool)
    return np.abs(i - j) <= half_window


def _brute_numpy(wl, theta, half_window):
    q, k, v = _heads_view(wl.qkv)
    out = np.zeros((wl.T, 768))
    cu = wl.cu_seqlens.tolist()
    for s in range(len(cu) - 1):
        b, e = cu[s], cu[s + 1]
        L = e - b
        if L == 0:
            continue
        pos = np.arange(L)
        mask = _band_mask(L, half_window)
        for h in range(12):
            qr = _rope_complex(q[b:e, h], pos, theta)
            kr = _rope_complex(k[b:e, h], pos, theta)
            sc = qr @ kr.T / 8.0
            sc = np.where(mask, sc, -np.inf)
            sc = sc - sc.max(axis=1, keepdims=True)
            p = np.exp(sc)
            p /= p.sum(axis=1, keepdims=True)
            out[b:e, h * 64:(h + 1) * 64] = p @ v[b:e, h]
    return out


def _brute_torch_sdpa(wl, theta, half_window):
    q, k, v = _heads_view(wl.qkv)
    out = torch.zeros(wl.T, 768, dtype=torch.float64)
    cu = wl.cu_seqlens.tolist()
    for s in range(len(cu) - 1):
        b, e = cu[s], cu[s + 1]
        L = e - b
        if L == 0:
            continue
        pos = np.arange(L)
        mask = torch.from_numpy(_band_mask(L, half_window))
        qs = torch.stack([torch.from_numpy(_rope_complex(q[b:e, h], pos, theta)) for h in range(12)])
        ks = torch.stack([torch.from_numpy(_rope_complex(k[b:e, h], pos, theta)) for h in range(12)])
        vs = torch.stack([torch.from_numpy(np.ascontiguousarray(v[b:e, h])) for h in range(12)])
        o = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask)
        out[b:e] = o.permute(1, 0, 2).reshape(L, 768)
    return out.numpy()


# ---------------------------------------------------------------------------
# scale, softmax axis and blend: the teardown's worked example
# ---------------------------------------------------------------------------

def test_worked_example_weights_match_page():
    """Teardown, "How Does Self-Attention Work?": the seed-0 4-token example.
    The oracle's dense core must print the page's 4x4 weights to 4 decimals
    and agree with torch's scaled_dot_product_attention (fp64)."""
    printed = np.array([[float(x) for x in r] for r in _read_table("worked_example_weights.txt")])
    torch.manual_seed(0)
    X = torch.randn(4, 8)
    Wq = torch.randn(8, 4) / 8 ** 0.5
    Wk = torch.randn(8, 4) / 8 ** 0.5
    Wv = torch.randn(8, 4) / 8 ** 0.5
    Xd = X.double().numpy()
    Q, K, V = Xd @ Wq.double().numpy(), Xd @ Wk.double().numpy(), Xd @ Wv.double().numpy()
    w, o = oracle.sdpa_dense(Q, K, V, scale=1.0 / np.sqrt(4.0))
    assert np.array_equal(np.round(w, 4), printed)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V)).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    # the first token weighs the last one (no causal mask): 0.3224 on the page
    assert w[0, 3] > 0.3


def test_dense_rows_sum_to_one_and_mask_zeroes():
    """Rows of weights sum to 1 (teardown, "How Does Self-Attention Work?");
    masked keys get weight exactly 0 (rayaq, padding mask)."""
    rng = np.random.default_rng(7)
    Q, K, V = rng.normal(size=(9, 16)), rng.normal(size=(11, 16)), rng.normal(size=(11, 5))
    mask = rng.random((9, 11)) < 0.6
    mask[:, 0] = True
    w, o = oracle.sdpa_dense(Q, K, V, 0.25, mask)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(w[~mask] == 0.0)
    np.testing.assert_allclose(o, w @ V, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def test_inv_freq_matches_printed_values():
    """Teardown, "How Does RoPE Work With Two Bases?": inv_freq[-1] is
    9.088847036764491e-06 (base 160000) and 1.333521504420787e-04 (base
    10000).  The page prints HF's fp32 values, within one fp32 ulp of fp64."""
    t = {r[0]: float(r[1]) for r in _read_table("rope_inv_freq.txt")}
    g = oracle.inv_freq(oracle.GLOBAL["theta"])
    l = oracle.inv_freq(oracle.LOCAL["theta"])
    assert g.shape == (32,) and l.shape == (32,)
    assert abs(g[31] / t["global_inv_freq_31"] - 1) < 1e-7
    assert abs(l[31] / t["local_inv_freq_31"] - 1) < 1e-7
    assert g[0] == 1.0 and l[0] == 1.0
    assert np.all(np.diff(g) < 0) and np.all(np.diff(l) < 0)
    # "about 15 times faster"
    assert 14.5 < l[31] / g[31] < 15.0
    assert round(8191 * g[31], 4) == t["global_turn_8191"]


def test_rope_matches_complex_multiplication():
    """Rotate-half RoPE (candding, "The two rope tables") equals multiplying
    pair (x[m], x[m+32]) as a complex number by exp(i*pos*inv_freq[m])."""
    rng = np.random.default_rng(3)
    x = rng.normal(size=(6, 64))
    pos = [0, 1, 7, 300, 4097, 8191]
    for theta in (160000.0, 10000.0):
        ref = _rope_complex(x, pos, theta)
        for r, p in enumerate(pos):
            np.testing.assert_allclose(oracle.rope(x[r], p, theta), ref[r], rtol=0, atol=1e-12)


def test_rope_rows_equal_row_by_row():
    """The many-rows form rotates each row exactly as the one-row form."""
    g = np.random.default_rng(8)
    x = g.standard_normal((50, 64))
    pos = g.integers(0, 8192, 50)
    y = oracle.rope_rows(x, pos, 160000.0)
    for r in range(50):
        np.testing.assert_array_equal(y[r], oracle.rope(x[r], int(pos[r]), 160000.0))


def test_rope_relative_position_and_norm():
    """Teardown: after RoPE the score depends on how far apart the two
    tokens are.  q(m).k(n) == q(m+t).k(n+t); each pair keeps its length;
    position 0 is the identity."""
    rng = np.random.default_rng(4)
    q, k = rng.normal(size=64), rng.normal(size=64)
    for theta in (160000.0, 10000.0):
        for m, n, t in [(0, 5, 17), (100, 36, 4000), (8000, 3, 191)]:
            a = oracle.rope(q, m, theta) @ oracle.rope(k, n, theta)
            b = oracle.rope(q, m + t, theta) @ oracle.rope(k, n + t, theta)
            assert abs(a - b) < 1e-10
        y = oracle.rope(q, 1234, theta)
        np.testing.assert_allclose(y[:32] ** 2 + y[32:] ** 2, q[:32] ** 2 + q[32:] ** 2,
                                   rtol=1e-12, atol=1e-12)
        assert np.array_equal(oracle.rope(q, 0, theta), q)


# ---------------------------------------------------------------------------
# the band and the admitted-key counts
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("row", _read_table("key_counts.txt"), ids=lambda r: r[0])
def test_key_counts_match_pages(row):
    """The printed key counts (candding, "The alternating attention";
    teardown, "What Are Local and Global Attention?")."""
    name, kind, L, where, expected = row
    L, expected = int(L), int(expected)
    hw = oracle.KINDS[kind]["half_window"]
    counts = oracle.key_counts([0, L], hw)
    if where == "sum":
        assert int(counts.astype(np.int64).sum()) == expected
    else:
        assert int(counts[int(where)]) == expected
        # the attention itself reports the same size of the admitted set
        wl = W.custom([L], seed=11)
        _, c = oracle.attention_kind(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), kind,
                                     rows=np.array([int(where)]))
        assert int(c[0]) == expected


def test_key_counts_closed_form():
    """Sum over rows of |A_i|: 129 L - 4160 for L >= 65 on a local layer
    (129 in the interior, 65..128 at each end), L^2 on a global layer."""
    for L in (1, 2, 64, 65, 66, 127, 128, 129, 300, 1000):
        loc = int(oracle.key_counts([0, L], 64).astype(np.int64).sum())
        glo = int(oracle.key_counts([0, L], -1).astype(np.int64).sum())
        assert glo == L * L
        assert loc == (129 * L - 4160 if L >= 65 else L * L)


def test_key_counts_never_cross_sequences():
    lengths = [5, 0, 200, 1, 70]
    cu = W.cu_from_lengths(lengths).numpy()
    c = oracle.key_counts(cu, 64)
    for s, L in enumerate(lengths):
        np.testing.assert_array_equal(c[cu[s]:cu[s + 1]], oracle.key_counts([0, L], 64))


# ---------------------------------------------------------------------------
# the whole block against brute force on tiny inputs
# ---------------------------------------------------------------------------

TINY_PACKS = [[1], [5, 64, 65], [130, 7, 200], [0, 129, 0, 33]]


@pytest.mark.parametrize("lengths", TINY_PACKS, ids=str)
@pytest.mark.parametrize("kind", ["global", "local"])
def test_attention_matches_bruteforce(lengths, kind):
    """Dense fp64 scores with an explicit -inf band mask (rayaq's padding
    mask idea; teardown's band), complex-number RoPE, and torch fp64
    scaled_dot_product_attention with a boolean mask (nest.franknoh,
    "The sliding window": a boolean [Q, K] band passed to SDPA)."""
    wl = W.custom(lengths, seed=sum(lengths) + 5)
    p = oracle.KINDS[kind]
    out, counts = oracle.attention(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), p["theta"],
                                   p["half_window"])
    ref_np = _brute_numpy(wl, p["theta"], p["half_window"])
    ref_t = _brute_torch_sdpa(wl, p["theta"], p["half_window"])
    np.testing.assert_allclose(out, ref_np, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, ref_t, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(counts, oracle.key_counts(wl.cu_seqlens.numpy(), p["half_window"]))


# ---------------------------------------------------------------------------
# the rotated operands rounded to bf16 (what a bf16 tensor-core path
# multiplies): the rounding itself and the block computed on rounded operands
# ---------------------------------------------------------------------------

def _round_bf16_bits(x):
    """Round fp64 values to 8 significant bits, ties to even, by bit
    manipulation of the binary64 encoding: keep the top 7 of the 52 stored
    fraction bits, then add one unit of the kept last place when the dropped
    part is above half of it, or exactly half with an odd kept part."""
    x = np.asarray(x, dtype=np.float64)
    u = x.view(np.uint64).copy()
    drop = np.uint64(45)
    low = u & ((np.uint64(1) << drop) - np.uint64(1))
    half = np.uint64(1) << (drop - np.uint64(1))
    kept = u & ~((np.uint64(1) << drop) - np.uint64(1))
    odd = (kept >> drop) & np.uint64(1)
    up = (low > half) | ((low == half) & (odd == np.uint64(1)))
    kept = kept + np.where(up, np.uint64(1) << drop, np.uint64(0)).astype(np.uint64)
    out = kept.view(np.float64)
    return np.where(x == 0, x, out)


def test_round_bf16_matches_torch_and_bit_rounding():
    """oracle.round_bf16 against torch's fp32 -> bf16 conversion on values
    that fp32 holds exactly, against the bit-level rounding on arbitrary fp64
    values, and on exact midpoints (ties go to the even neighbour)."""
    g = np.random.default_rng(5)
    x32 = (g.standard_normal(20000) * np.exp(g.uniform(-20, 20, 20000))).astype(np.float32)
    x = x32.astype(np.float64)
    ref = torch.from_numpy(x32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), ref)
    y = g.standard_normal(20000) * np.exp(g.uniform(-20, 20, 20000))
    np.testing.assert_array_equal(oracle.round_bf16(y), _round_bf16_bits(y))
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3 * 2.0 ** -9 + 2.0 ** -17])
    np.testing.assert_array_equal(oracle.round_bf16(ties)[:3], [1.0, 1 + 2.0 ** -6, -1.0])
    assert oracle.round_bf16(ties)[3] == _round_bf16_bits(ties)[3]


@pytest.mark.parametrize("lengths", [[5, 64, 65], [130, 7, 200]], ids=str)
@pytest.mark.parametrize("kind", ["global", "local"])
def test_rounded_operands_match_bruteforce(lengths, kind):
    """The block on rounded operands: complex-number RoPE in numpy, the
    bit-level rounding above on the rotated q and k, dense scores / 8 with an
    explicit band mask, softmax and blend.  Inputs of spread 4 (scores of
    spread ~16) make the rounding matter: the result differs from the
    unrounded block, yet equals the brute force to 1e-12."""
    wl = W.custom(lengths, seed=sum(lengths) + 17, sigma=4.0)
    p = oracle.KINDS[kind]
    out, _ = oracle.attention(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), p["theta"],
                              p["half_window"], round_operands=True)
    q, k, v = _heads_view(wl.qkv)
    ref = np.zeros((wl.T, 768))
    cu = wl.cu_seqlens.tolist()
    for s in range(len(cu) - 1):
        b, e = cu[s], cu[s + 1]
        pos = np.arange(e - b)
        mask = _band_mask(e - b, p["half_window"])
        for h in range(12):
            qr = _round_bf16_bits(_rope_complex(q[b:e, h], pos, p["theta"]))
            kr = _round_bf16_bits(_rope_complex(k[b:e, h], pos, p["theta"]))
            sc = np.where(mask, qr @ kr.T / 8.0, -np.inf)
            w = np.exp(sc - sc.max(axis=1, keepdims=True))
            w /= w.sum(axis=1, keepdims=True)
            ref[b:e, h * 64:(h + 1) * 64] = w @ v[b:e, h]
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    plain, _ = oracle.attention(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), p["theta"],
                                p["half_window"])
    assert np.abs(plain - out).max() > 1e-3


def test_rounded_operands_at_position_zero_are_exact():
    """At position 0 RoPE turns nothing, so the rotated rows are the bf16
    inputs themselves and rounding them changes nothing: a pack of length-1
    sequences gives bit-identical results with and without the rounding."""
    wl = W.custom([1, 1, 1, 1, 1], seed=23, sigma=4.0)
    for kind in ("global", "local"):
        a, _ = oracle.attention_kind(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), kind)
        b, _ = oracle.attention_kind(W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy(), kind,
                                     round_operands=True)
        np.testing.assert_array_equal(a, b)


def test_wrong_theta_or_window_is_detected():
    """The brute force separates the two layer kinds: swapping the bases or
    widening the band changes the outputs well beyond rounding."""
    wl = W.custom([300], seed=12)
    bits, cu = W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy()
    ref = _brute_numpy(wl, 10000.0, 64)
    swapped, _ = oracle.attention(bits, cu, 160000.0, 64)
    wider, _ = oracle.attention(bits, cu, 10000.0, 65)
    assert np.abs(swapped - ref).max() > 1e-3
    assert np.abs(wider - ref).max() > 1e-6


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

def test_global_equals_band_covering_sequence():
    """A global layer is a band whose window covers the sequence
    (nest.franknoh, "The sliding window"), with the same base."""
    wl = W.custom([150, 1, 97], seed=21)
    bits, cu = W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy()
    g, _ = oracle.attention(bits, cu, 160000.0, -1)
    b, _ = oracle.attention(bits, cu, 160000.0, 149)
    assert np.array_equal(g, b)


def test_masked_pad_gap_is_zero():
    """rayaq, padding mask: a masked pad leaves the real outputs unchanged
    (gap 0).  Packing a pad as its own sequence after the real one, and
    masking its key in the dense core, both give bit-identical rows."""
    real = W.custom([37], seed=31)
    padded = W.custom([37, 3], seed=31)  # same generator: first 37 rows equal
    assert torch.equal(padded.qkv[:37], real.qkv)
    for kind in ("global", "local"):
        a, _ = oracle.attention_kind(W.bf16_bits(real.qkv), real.cu_seqlens.numpy(), kind)
        b, _ = oracle.attention_kind(W.bf16_bits(padded.qkv), padded.cu_seqlens.numpy(), kind)
        assert np.array_equal(a, b[:37])
    # key-padding mask form: one extra key that every query masks out
    rng = np.random.default_rng(5)
    Q, K, V = rng.normal(size=(6, 8)), rng.normal(size=(7, 8)), rng.normal(size=(7, 8))
    mask = np.ones((6, 7), dtype=bool)
    mask[:, 6] = False
    w1, o1 = oracle.sdpa_dense(Q, K[:6], V[:6], 0.3)
    w2, o2 = oracle.sdpa_dense(Q, K, V, 0.3, mask)
    assert np.array_equal(o1, o2) and np.array_equal(w1, w2[:, :6])


def test_offset_in_pack_does_not_matter():
    """Positions restart in every sequence (candding, "The two rope
    tables"): moving a sequence within the pack leaves its rows unchanged."""
    a = W.custom([90], seed=41)
    b = W.custom([90], seed=42)
    pack = torch.cat([b.qkv, a.qkv])
    cu = np.array([0, 90, 180], dtype=np.int32)
    for kind in ("global", "local"):
        alone, _ = oracle.attention_kind(W.bf16_bits(a.qkv), a.cu_seqlens.numpy(), kind)
        packed, _ = oracle.attention_kind(W.bf16_bits(pack), cu, kind)
        assert np.array_equal(alone, packed[90:])


def test_length_one_sequence_returns_its_value():
    """A sequence of one token attends only to itself: out = v exactly."""
    wl = W.custom([1, 4, 1], seed=51)
    bits, cu = W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy()
    v = wl.qkv.double()[:, 1536:].numpy()
    for kind in ("global", "local"):
        out, counts = oracle.attention_kind(bits, cu, kind)
        assert np.array_equal(out[0], v[0]) and np.array_equal(out[5], v[5])
        assert counts[0] == 1 and counts[5] == 1


def test_unit_values_give_unit_outputs():
    """Rows of weights sum to 1: with every value row equal to 1 the output
    is 1 to rounding, on both layer kinds."""
    wl = W.custom([260, 3], seed=61)
    q = wl.qkv.clone()
    q[:, 1536:] = 1.0
    for kind in ("global", "local"):
        out, _ = oracle.attention_kind(W.bf16_bits(q), wl.cu_seqlens.numpy(), kind)
        np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-12)


def test_sampled_rows_equal_full_rows():
    wl = W.config(2)
    bits, cu = W.bf16_bits(wl.qkv), wl.cu_seqlens.numpy()
    rows = W.sample_rows(cu, 16, seed=9)
    for kind in ("global", "local"):
        full, cf = oracle.attention_kind(bits, cu, kind)
        part, cp = oracle.attention_kind(bits, cu, kind, rows=rows)
        assert np.array_equal(full[rows], part)
        assert np.array_equal(cf[rows], cp)


def test_bad_cu_seqlens_rejected():
    wl = W.custom([10], seed=1)
    bits = W.bf16_bits(wl.qkv)
    for cu in ([1, 10], [0, 11], [0, 6, 4, 10]):
        with pytest.raises(ValueError):
            oracle.attention(bits, np.array(cu, dtype=np.int32), 1e4, 64)


def test_workload_recipes():
    """The synthetic workloads have the shapes their recipes state."""
    c1 = W.config(1)
    assert c1.lengths == [300] and tuple(c1.qkv.shape) == (300, 2304)
    c2 = W.config(2)
    assert len(c2.lengths) == 8 and all(64 <= L <= 512 for L in c2.lengths)
    assert c2.T == sum(c2.lengths)
    assert W.config(2).lengths == c2.lengths and torch.equal(W.config(2).qkv, c2.qkv)
    g = torch.Generator().manual_seed(4)
    lens = W._fill_lengths(g, 65536, 128, 8192)
    assert sum(lens) == 65536 and all(L <= 8192 for L in lens[:-1])
    assert all(L >= 128 for L in lens[:-1])
    assert [W.layer_kind(i) for i in range(22)].count("global") == 8
