"""Pins of the oracle's padded-batch attention (the masked form over
[B, S] with a 0/1 attention mask): pads are masked keys, a real token's
position is its rank among its row's real tokens, pad rows of the output are
0 ("ModernBERT-base Architecture Teardown", the tokenizer with padding=True
and its attention mask; "Encoder-only models", "Padding and the key padding
mask").  Each pin fixes the result by something other than the padded
oracle's own formula: the packed oracle on the unpadded sequences, or exact
invariances the pages state.
"""
import numpy as np
import pytest
import torch

import oracle

HEADS, HD = 12, 64
WIDTH = 3 * HEADS * HD


def rand_qkv(B, S, seed):
    g = torch.Generator().manual_seed(seed)
    t = torch.randn(B, S, WIDTH, generator=g).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def right_mask(lengths, S):
    return np.array([[1] * L + [0] * (S - L) for L in lengths], dtype=np.int32)


@pytest.mark.parametrize("kind", ["global", "local"])
def test_masked_rows_equal_the_sequences_alone(kind):
    # the page's check: with the pads masked, the real outputs equal those of
    # each sequence run alone (here the packed oracle on the unpadded rows)
    p = oracle.KINDS[kind]
    lengths, S = [100, 37, 1], 100
    qkv = rand_qkv(3, S, 1)
    got = oracle.attention_padded(qkv, right_mask(lengths, S), p["theta"], p["half_window"])
    packed = np.concatenate([qkv[b, :L] for b, L in enumerate(lengths)])
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    ref, _ = oracle.attention(packed, cu, p["theta"], p["half_window"])
    for b, L in enumerate(lengths):
        assert np.allclose(got[b, :L], ref[cu[b]:cu[b] + L], rtol=0, atol=1e-12)


def test_pad_contents_do_not_matter_and_pad_rows_are_zero():
    lengths, S = [20, 33], 40
    mask = right_mask(lengths, S)
    a = rand_qkv(2, S, 2)
    b = a.copy()
    noise = rand_qkv(2, S, 3)
    b[mask == 0] = noise[mask == 0]
    for kind in ("global", "local"):
        p = oracle.KINDS[kind]
        oa = oracle.attention_padded(a, mask, p["theta"], p["half_window"])
        ob = oracle.attention_padded(b, mask, p["theta"], p["half_window"])
        assert np.array_equal(oa[mask == 1], ob[mask == 1])
        assert np.array_equal(oa[mask == 0], np.zeros_like(oa[mask == 0]))


def test_forgetting_the_mask_changes_real_outputs():
    # the page: without the mask the pads take attention weight and the real
    # outputs move
    lengths, S = [10], 14
    qkv = rand_qkv(1, S, 4)
    p = oracle.GLOBAL
    masked = oracle.attention_padded(qkv, right_mask(lengths, S), p["theta"], -1)
    unmasked = oracle.attention_padded(qkv, np.ones((1, S), np.int32), p["theta"], -1)
    assert np.abs(masked[0, :10] - unmasked[0, :10]).max() > 1e-3


def test_left_padding_equals_right_padding():
    # positions count the real tokens, so where the pads sit does not matter
    S, L = 60, 45
    right = rand_qkv(1, S, 5)
    left = np.zeros_like(right)
    left[0, S - L:] = right[0, :L]
    mr = right_mask([L], S)
    ml = np.array([[0] * (S - L) + [1] * L], dtype=np.int32)
    for kind in ("global", "local"):
        p = oracle.KINDS[kind]
        orr = oracle.attention_padded(right, mr, p["theta"], p["half_window"])
        oll = oracle.attention_padded(left, ml, p["theta"], p["half_window"])
        assert np.array_equal(orr[0, :L], oll[0, S - L:])


def test_all_pad_row_is_zero():
    qkv = rand_qkv(2, 16, 6)
    mask = np.array([[0] * 16, [1] * 16], dtype=np.int32)
    out = oracle.attention_padded(qkv, mask, 160000.0, -1)
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.abs(out[1]).max() > 0
