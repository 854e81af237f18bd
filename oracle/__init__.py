"""fp64 CPU oracle for the ModernBERT-base attention block (ctypes binding).

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline / reference legs may import this package.  The CUDA library never
does, and this package imports nothing from it.

What it computes is stated in mbert_attn_oracle.c with the passages it follows.
Layer constants are restated here from the pages, independently of the CUDA
path:

* "ModernBERT-base Architecture Teardown", "How Does RoPE Work With Two
  Bases?": base 160000 on global layers, 10000 on local layers.
* same page, "What Are Local and Global Attention?" and "ModernBERT"
  (candding), "The alternating attention": local layers keep |i - j| <= 64.
* teardown, "How Does ModernBERT Make Q, K and V?": 12 heads of 64.
* teardown, "What Does LayerNorm Do?": eps 1e-5 under the square root.
"""
import ctypes
import os

import numpy as np

from . import build as _build

HEADS = 12
HEAD_DIM = 64
GLOBAL = {"theta": 160000.0, "half_window": -1}
LOCAL = {"theta": 10000.0, "half_window": 64}
KINDS = {"global": GLOBAL, "local": LOCAL}
NORM_EPS = 1e-5

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        L.oracle_inv_freq.argtypes = [ctypes.c_double, ctypes.c_int, dp]
        L.oracle_inv_freq.restype = None
        L.oracle_rope_row.argtypes = [dp, ctypes.c_int64, ctypes.c_double, ctypes.c_int, dp]
        L.oracle_rope_row.restype = None
        L.oracle_key_counts.argtypes = [i32p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, i32p]
        L.oracle_key_counts.restype = ctypes.c_int
        L.oracle_sdpa_dense.argtypes = [dp, dp, dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_double, u8p, dp, dp]
        L.oracle_sdpa_dense.restype = ctypes.c_int
        L.oracle_attention.argtypes = [u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, i32p,
                                       ctypes.c_int, ctypes.c_double, ctypes.c_int, i64p,
                                       ctypes.c_int64, dp, i32p, ctypes.c_int]
        L.oracle_attention.restype = ctypes.c_int
        L.oracle_attention_rounded.argtypes = L.oracle_attention.argtypes
        L.oracle_attention_rounded.restype = ctypes.c_int
        L.oracle_round_bf16.argtypes = [ctypes.c_double]
        L.oracle_round_bf16.restype = ctypes.c_double
        L.oracle_round_bf16_n.argtypes = [dp, ctypes.c_int64, dp]
        L.oracle_round_bf16_n.restype = None
        L.oracle_rope_rows.argtypes = [dp, ctypes.c_int64, i64p, ctypes.c_double, ctypes.c_int, dp]
        L.oracle_rope_rows.restype = None
        L.oracle_out_proj.argtypes = [u16p, u16p, u16p, ctypes.c_int64, ctypes.c_int, i64p,
                                      ctypes.c_int64, dp, ctypes.c_int]
        L.oracle_out_proj.restype = ctypes.c_int
        L.oracle_layernorm.argtypes = [u16p, u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                       i64p, ctypes.c_int64, dp, ctypes.c_int]
        L.oracle_layernorm.restype = ctypes.c_int
        L.oracle_ln_qkv.argtypes = [u16p, u16p, u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_double, i64p, ctypes.c_int64, dp, ctypes.c_int]
        L.oracle_ln_qkv.restype = ctypes.c_int
        L.oracle_gelu.argtypes = [dp, ctypes.c_int64, dp]
        L.oracle_gelu.restype = None
        L.oracle_mlp.argtypes = [u16p, u16p, u16p, u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_double, i64p, ctypes.c_int64, dp, ctypes.c_int]
        L.oracle_mlp.restype = ctypes.c_int
        L.oracle_max_threads.argtypes = []
        L.oracle_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def inv_freq(theta: float, head_dim: int = HEAD_DIM) -> np.ndarray:
    out = np.empty(head_dim // 2, dtype=np.float64)
    lib().oracle_inv_freq(float(theta), int(head_dim), _ptr(out, ctypes.c_double))
    return out


def rope(x, pos: int, theta: float) -> np.ndarray:
    """Rotate one head row x[head_dim] (fp64) sitting at position `pos`."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib().oracle_rope_row(_ptr(x, ctypes.c_double), int(pos), float(theta), x.shape[0],
                          _ptr(y, ctypes.c_double))
    return y


def rope_rows(x, pos, theta: float) -> np.ndarray:
    """Rotate rows x[n, head_dim] (fp64), row r sitting at position pos[r]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    p = np.ascontiguousarray(pos, dtype=np.int64)
    assert x.ndim == 2 and p.shape == (x.shape[0],)
    y = np.empty_like(x)
    lib().oracle_rope_rows(_ptr(x, ctypes.c_double), x.shape[0], _ptr(p, ctypes.c_int64),
                           float(theta), x.shape[1], _ptr(y, ctypes.c_double))
    return y


def key_counts(cu_seqlens, half_window: int) -> np.ndarray:
    """|A_i| of every packed row, by brute force over the band predicate."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T = int(cu[-1])
    counts = np.zeros(T, dtype=np.int32)
    rc = lib().oracle_key_counts(_ptr(cu, ctypes.c_int32), len(cu) - 1, T, int(half_window),
                                 _ptr(counts, ctypes.c_int32))
    if rc:
        raise ValueError(f"oracle_key_counts: bad cu_seqlens (code {rc})")
    return counts


def sdpa_dense(Q, K, V, scale: float, mask=None):
    """softmax(scale * Q K^T, masked) V in fp64.  Returns (weights, out)."""
    Q = np.ascontiguousarray(Q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    n, d = Q.shape
    m, dv = V.shape
    assert K.shape == (m, d)
    w = np.empty((n, m), dtype=np.float64)
    o = np.empty((n, dv), dtype=np.float64)
    mp = None
    if mask is not None:
        mk = np.ascontiguousarray(mask, dtype=np.uint8)
        assert mk.shape == (n, m)
        mp = _ptr(mk, ctypes.c_uint8)
    rc = lib().oracle_sdpa_dense(_ptr(Q, ctypes.c_double), _ptr(K, ctypes.c_double),
                                 _ptr(V, ctypes.c_double), n, m, d, dv, float(scale), mp,
                                 _ptr(w, ctypes.c_double), _ptr(o, ctypes.c_double))
    if rc:
        raise ValueError(f"oracle_sdpa_dense failed ({rc})")
    return w, o


def round_bf16(x) -> np.ndarray:
    """Each value rounded to the nearest bf16 (8 significant bits, ties to
    even), as fp64."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(a)
    lib().oracle_round_bf16_n(_ptr(a, ctypes.c_double), a.size, _ptr(y, ctypes.c_double))
    return y


def attention(qkv_bits, cu_seqlens, theta: float, half_window: int, rows=None,
              threads: int = 0, heads: int = HEADS, head_dim: int = HEAD_DIM,
              round_operands: bool = False):
    """The attention block in fp64.

    qkv_bits: uint16 [T, 3*heads*head_dim], the bf16 bit patterns of the fused
    Wqkv output.  cu_seqlens: int32 [n_seqs+1].  rows: None (every row) or a
    sorted array of packed row indices.  Returns (out fp64 [n, heads*head_dim],
    counts int32 [n]).  round_operands: round the rotated q and k rows to bf16
    before forming the scores (the operands a bf16 tensor-core path
    multiplies); everything else stays fp64.
    """
    q = np.ascontiguousarray(qkv_bits)
    if q.dtype != np.uint16:
        raise TypeError("qkv_bits must be uint16 bf16 bit patterns")
    T = q.shape[0]
    assert q.shape[1] == 3 * heads * head_dim
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    if rows is None:
        n = T
        rp = None
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        n = r.shape[0]
        rp = _ptr(r, ctypes.c_int64)
    out = np.empty((n, heads * head_dim), dtype=np.float64)
    counts = np.zeros(n, dtype=np.int32)
    fn = lib().oracle_attention_rounded if round_operands else lib().oracle_attention
    rc = fn(_ptr(q, ctypes.c_uint16), T, heads, head_dim, _ptr(cu, ctypes.c_int32),
            len(cu) - 1, float(theta), int(half_window), rp, n, _ptr(out, ctypes.c_double),
            _ptr(counts, ctypes.c_int32), int(threads))
    if rc:
        raise ValueError(f"oracle_attention failed (code {rc})")
    return out, counts


def out_proj(a_bits, wo_bits, x_bits, rows=None, threads: int = 0):
    """y = x + a Wo^T in fp64 (Wo stored [out][in]).

    a_bits, x_bits: uint16 [T, d] bf16 bit patterns (joined head outputs and
    the residual stream); wo_bits: uint16 [d, d].  rows: None (every row) or
    sorted packed row indices.  Returns fp64 [n, d].
    """
    a = np.ascontiguousarray(a_bits)
    x = np.ascontiguousarray(x_bits)
    w = np.ascontiguousarray(wo_bits)
    if a.dtype != np.uint16 or x.dtype != np.uint16 or w.dtype != np.uint16:
        raise TypeError("inputs must be uint16 bf16 bit patterns")
    T, d = a.shape
    assert x.shape == (T, d) and w.shape == (d, d)
    if rows is None:
        n, rp = T, None
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        n, rp = r.shape[0], _ptr(r, ctypes.c_int64)
    y = np.empty((n, d), dtype=np.float64)
    rc = lib().oracle_out_proj(_ptr(a, ctypes.c_uint16), _ptr(w, ctypes.c_uint16),
                               _ptr(x, ctypes.c_uint16), T, d, rp, n,
                               _ptr(y, ctypes.c_double), int(threads))
    if rc:
        raise ValueError(f"oracle_out_proj failed (code {rc})")
    return y


def _rows_arg(rows, T):
    if rows is None:
        return T, None, None
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r.shape[0], r, _ptr(r, ctypes.c_int64)


def layernorm(x_bits, w_bits=None, eps: float = NORM_EPS, rows=None, threads: int = 0):
    """Bias-free LayerNorm in fp64, row by row; w_bits None is the identity
    (layer 0's attn_norm).

    x_bits: uint16 [T, d] bf16 bit patterns; w_bits: uint16 [d] or None.
    Returns fp64 [n, d] (rows: None for every row, or sorted row indices).
    """
    x = np.ascontiguousarray(x_bits)
    if x.dtype != np.uint16 or x.ndim != 2:
        raise TypeError("x must be uint16 [T, d] bf16 bit patterns")
    T, d = x.shape
    wp = None
    if w_bits is not None:
        w = np.ascontiguousarray(w_bits)
        if w.dtype != np.uint16 or w.shape != (d,):
            raise TypeError("w must be uint16 [d] bf16 bit patterns")
        wp = _ptr(w, ctypes.c_uint16)
    n, r, rp = _rows_arg(rows, T)
    h = np.empty((n, d), dtype=np.float64)
    rc = lib().oracle_layernorm(_ptr(x, ctypes.c_uint16), wp, T, d, float(eps), rp, n,
                                _ptr(h, ctypes.c_double), int(threads))
    if rc:
        raise ValueError(f"oracle_layernorm failed (code {rc})")
    return h


def ln_qkv(x_bits, w_bits, wqkv_bits, eps: float = NORM_EPS, rows=None, threads: int = 0):
    """qkv = LayerNorm(x) Wqkv^T in fp64 (Wqkv stored [out][in]); w_bits None
    is the identity norm of layer 0.

    x_bits: uint16 [T, d]; w_bits: uint16 [d] or None; wqkv_bits: uint16
    [n_out, d].  Returns fp64 [n, n_out].
    """
    x = np.ascontiguousarray(x_bits)
    wq = np.ascontiguousarray(wqkv_bits)
    if x.dtype != np.uint16 or wq.dtype != np.uint16 or x.ndim != 2 or wq.ndim != 2:
        raise TypeError("x and wqkv must be 2-D uint16 bf16 bit patterns")
    T, d = x.shape
    n_out = wq.shape[0]
    assert wq.shape == (n_out, d)
    wp = None
    if w_bits is not None:
        w = np.ascontiguousarray(w_bits)
        if w.dtype != np.uint16 or w.shape != (d,):
            raise TypeError("w must be uint16 [d] bf16 bit patterns")
        wp = _ptr(w, ctypes.c_uint16)
    n, r, rp = _rows_arg(rows, T)
    out = np.empty((n, n_out), dtype=np.float64)
    rc = lib().oracle_ln_qkv(_ptr(x, ctypes.c_uint16), wp, _ptr(wq, ctypes.c_uint16), T, d,
                             n_out, float(eps), rp, n, _ptr(out, ctypes.c_double), int(threads))
    if rc:
        raise ValueError(f"oracle_ln_qkv failed (code {rc})")
    return out


def gelu(z):
    """The exact (erf) GELU, elementwise, fp64."""
    zz = np.ascontiguousarray(z, dtype=np.float64)
    out = np.empty_like(zz)
    lib().oracle_gelu(_ptr(zz, ctypes.c_double), zz.size, _ptr(out, ctypes.c_double))
    return out


def mlp(x_bits, norm_w_bits, wi_bits, wo_bits, eps: float = NORM_EPS, rows=None, threads: int = 0):
    """y = x + (GELU(g) * u) Wo^T, g, u = halves of LayerNorm(x) Wi^T, fp64.

    x_bits: uint16 [T, d]; norm_w_bits: uint16 [d]; wi_bits: uint16
    [2 * inner, d]; wo_bits: uint16 [d, inner] (bf16 bit patterns, weights
    stored [out][in]).  Returns fp64 [n, d].
    """
    x = np.ascontiguousarray(x_bits)
    w = np.ascontiguousarray(norm_w_bits)
    wi = np.ascontiguousarray(wi_bits)
    wo = np.ascontiguousarray(wo_bits)
    for t in (x, w, wi, wo):
        if t.dtype != np.uint16:
            raise TypeError("inputs must be uint16 bf16 bit patterns")
    T, d = x.shape
    inner = wo.shape[1]
    assert w.shape == (d,) and wi.shape == (2 * inner, d) and wo.shape == (d, inner)
    n, r, rp = _rows_arg(rows, T)
    y = np.empty((n, d), dtype=np.float64)
    rc = lib().oracle_mlp(_ptr(x, ctypes.c_uint16), _ptr(w, ctypes.c_uint16),
                          _ptr(wi, ctypes.c_uint16), _ptr(wo, ctypes.c_uint16), T, d, inner,
                          float(eps), rp, n, _ptr(y, ctypes.c_double), int(threads))
    if rc:
        raise ValueError(f"oracle_mlp failed (code {rc})")
    return y


def attention_padded(qkv_bits, mask, theta: float, half_window: int,
                     heads: int = HEADS, head_dim: int = HEAD_DIM):
    """The attention block over a padded batch, in its masked form, fp64.

    qkv_bits: uint16 [B, S, 3 heads head_dim] bf16 bit patterns; mask: [B, S],
    non-zero for a real token, 0 for a pad.  Inside attention the pads are
    masked keys ("ModernBERT-base Architecture Teardown", the tokenizer with
    padding=True: the 0s of the attention mask become a mask, so no real token
    takes information from a pad; "Encoder-only models", "Padding and the key
    padding mask": -inf at the ignored keys).  A real token's position is its
    rank among the row's real tokens (its index in the row for right padding,
    the tokenizer's form).  Query i admits key j iff both are real and, on a
    local layer, |pos_i - pos_j| <= half_window.  A pad's row of the output is
    0 (nothing downstream reads it).  Pure Python over rows and heads, for
    small batches.  Returns fp64 [B, S, heads head_dim].
    """
    qkv = np.ascontiguousarray(qkv_bits)
    m = np.asarray(mask) != 0
    B, S, width = qkv.shape
    assert m.shape == (B, S) and width == 3 * heads * head_dim
    vals = (qkv.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out = np.zeros((B, S, heads * head_dim), dtype=np.float64)
    for b in range(B):
        real = np.flatnonzero(m[b])
        if real.size == 0:
            continue
        pos = np.cumsum(m[b]) - 1
        adm = m[b][:, None] & m[b][None, :]
        if half_window >= 0:
            adm &= np.abs(pos[:, None] - pos[None, :]) <= half_window
        for h in range(heads):
            q = vals[b, :, h * head_dim:(h + 1) * head_dim]
            k = vals[b, :, (heads + h) * head_dim:(heads + h + 1) * head_dim]
            v = vals[b, :, (2 * heads + h) * head_dim:(2 * heads + h + 1) * head_dim]
            Q = np.zeros((S, head_dim))
            K = np.zeros((S, head_dim))
            for t in real:
                Q[t] = rope(q[t], int(pos[t]), theta)
                K[t] = rope(k[t], int(pos[t]), theta)
            _, o = sdpa_dense(Q, K, v, 1.0 / np.sqrt(head_dim), mask=adm)
            out[b, :, h * head_dim:(h + 1) * head_dim] = o
    return out


def attention_kind(qkv_bits, cu_seqlens, kind: str, rows=None, threads: int = 0,
                   round_operands: bool = False):
    """attention() with the constants of a ModernBERT-base layer kind."""
    p = KINDS[kind]
    return attention(qkv_bits, cu_seqlens, p["theta"], p["half_window"], rows=rows,
                     threads=threads, round_operands=round_operands)
