"""Thin ctypes binding of libmbert_attn.so (argument marshalling only).

Every step of the attention block runs in the library's CUDA kernels; this
module checks torch dtypes, devices and shapes, passes raw device pointers
and the current CUDA stream, and turns status codes into exceptions.  There
is no fallback: if the library is missing, every call raises.
"""
import ctypes
import os
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libmbert_attn.so"

GLOBAL = 0
LOCAL = 1
_KINDS = {"global": GLOBAL, "local": LOCAL, GLOBAL: GLOBAL, LOCAL: LOCAL}

HEADS, HEAD_DIM = 12, 64
QKV_WIDTH, OUT_WIDTH = 3 * HEADS * HEAD_DIM, HEADS * HEAD_DIM
MLP_INNER = 1152  # the GeGLU MLP's inner width (teardown, "What Does the GeGLU MLP Do?")
NORM_EPS = 1e-5   # LayerNorm eps of ModernBERT-base (teardown, "What Does LayerNorm Do?")

# Every symbol the public header declares, with its ctypes signature.
_c_int, _c_i64, _vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p


class Config(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("half_window", ctypes.c_int), ("max_seqlen", ctypes.c_int),
                ("theta_global", ctypes.c_double), ("theta_local", ctypes.c_double)]


SIGNATURES = {
    "mbert_attn_default_config": (_c_int, [ctypes.POINTER(Config)]),
    "mbert_attn_create": (_c_int, [ctypes.POINTER(_vp), ctypes.POINTER(Config), _c_int]),
    "mbert_attn_reserve": (_c_int, [_vp, _c_i64, _c_i64]),
    "mbert_attn_forward": (_c_int, [_vp, _vp, _vp, _c_int, _c_i64, _c_int, _c_int, _vp, _vp]),
    "mbert_attn_forward_padded": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp]),
    "mbert_attn_key_counts": (_c_int, [_vp, _vp, _c_int, _c_i64, _c_int, _c_int, _vp, _vp]),
    "mbert_attn_out_proj": (_c_int, [_vp, _vp, _vp, _vp, _c_i64, _vp, _vp]),
    "mbert_attn_ln_qkv": (_c_int, [_vp, _vp, _vp, _vp, _c_i64, ctypes.c_float, _vp, _vp]),
    "mbert_attn_mlp": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_i64, ctypes.c_float, _vp, _vp]),
    "mbert_attn_get_error": (_c_int, [_vp]),
    "mbert_attn_selftest_timeout": (_c_int, [_vp, _c_i64, _vp]),
    "mbert_attn_forward_noalloc": (_c_int, [_vp, _vp, _c_int, _c_i64, _c_int, _c_int, _vp, _vp,
                                            _vp]),
    "mbert_attn_profile_enable": (_c_int, [_vp, _c_int]),
    "mbert_attn_profile_read": (_c_int, [_vp, ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_int64),
                                         ctypes.POINTER(ctypes.c_int64)]),
    "mbert_attn_destroy": (None, [_vp]),
    "mbert_attn_strerror": (ctypes.c_char_p, [_c_int]),
}

_lib = None
_lib_lock = threading.Lock()


class MbertAttnError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        msg = strerror(status) if _lib is not None else str(status)
        super().__init__(f"{what}: {msg} (status {status})" if what else f"{msg} (status {status})")


def library_path() -> str:
    return os.path.join(PKG, "_build", LIB_NAME)


def load_library(path: str = None):
    """Load the CUDA library (once).  Raises OSError if it is not built."""
    global _lib
    with _lib_lock:
        if _lib is None:
            p = path or library_path()
            if not os.path.exists(p):
                raise OSError(f"{p} is missing: build it with "
                              f"`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def strerror(status: int) -> str:
    return load_library().mbert_attn_strerror(int(status)).decode()


def _check(status, what):
    if status != 0:
        raise MbertAttnError(status, what)


def _kind(layer_kind) -> int:
    try:
        return _KINDS[layer_kind]
    except KeyError:
        raise ValueError(f"layer_kind must be 'global', 'local', 0 or 1, not {layer_kind!r}")


def _stream_ptr(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


class Attention:
    """A library handle on one CUDA device (owns the RoPE tables, the work
    list, the rotated-operand scratch and the device error word)."""

    def __init__(self, device=None, half_window: int = 64, max_seqlen: int = 8192,
                 theta_global: float = 160000.0, theta_local: float = 10000.0):
        lib = load_library()
        if device is None:
            idx = torch.cuda.current_device()
        elif isinstance(device, int):
            idx = device
        else:
            d = torch.device(device)
            idx = d.index if d.index is not None else torch.cuda.current_device()
        self.device = torch.device("cuda", idx)
        cfg = Config()
        _check(lib.mbert_attn_default_config(ctypes.byref(cfg)), "default_config")
        cfg.half_window = half_window
        cfg.max_seqlen = max_seqlen
        cfg.theta_global = theta_global
        cfg.theta_local = theta_local
        self.config = cfg
        h = _vp()
        _check(lib.mbert_attn_create(ctypes.byref(h), ctypes.byref(cfg), self.device.index), "create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            load_library().mbert_attn_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check_cu(self, cu_seqlens):
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
            raise TypeError("cu_seqlens must be a 1-D int32 tensor")
        if cu_seqlens.device != self.device:
            raise ValueError(f"cu_seqlens must be on {self.device}")
        if not cu_seqlens.is_contiguous():
            raise ValueError("cu_seqlens must be contiguous")

    def reserve(self, max_tokens: int, max_seqs: int):
        _check(load_library().mbert_attn_reserve(self._h, int(max_tokens), int(max_seqs)), "reserve")

    def forward(self, qkv: torch.Tensor, cu_seqlens: torch.Tensor, layer_kind,
                max_seqlen: int = 0, out: torch.Tensor = None) -> torch.Tensor:
        """out[T, 768] bf16 = the attention block of one layer over qkv[T, 2304]."""
        kind = _kind(layer_kind)
        if qkv.dtype != torch.bfloat16 or qkv.dim() != 2 or qkv.shape[1] != QKV_WIDTH:
            raise TypeError("qkv must be a bf16 tensor of shape [T, 2304]")
        if qkv.device != self.device:
            raise ValueError(f"qkv must be on {self.device}")
        if not qkv.is_contiguous():
            raise ValueError("qkv must be contiguous")
        self._check_cu(cu_seqlens)
        T = qkv.shape[0]
        if out is None:
            out = torch.empty(T, OUT_WIDTH, dtype=torch.bfloat16, device=self.device)
        elif (out.dtype != torch.bfloat16 or tuple(out.shape) != (T, OUT_WIDTH)
              or out.device != self.device or not out.is_contiguous()):
            raise TypeError("out must be a contiguous bf16 [T, 768] tensor on the same device")
        st = load_library().mbert_attn_forward(
            self._h, qkv.data_ptr(), cu_seqlens.data_ptr(), cu_seqlens.numel() - 1, T,
            int(max_seqlen), kind, out.data_ptr(), _stream_ptr(self.device))
        _check(st, "forward")
        return out

    def out_proj(self, a: torch.Tensor, wo: torch.Tensor, x: torch.Tensor,
                 out: torch.Tensor = None) -> torch.Tensor:
        """y[T, 768] bf16 = x + a Wo^T: the output projection (Wo [768, 768],
        stored [out, in]) with the residual add.  `out` may be `x` itself."""
        def check(t, name, shape):
            if (t.dtype != torch.bfloat16 or tuple(t.shape) != shape or t.device != self.device
                    or not t.is_contiguous()):
                raise TypeError(f"{name} must be a contiguous bf16 {list(shape)} tensor on {self.device}")
        T = a.shape[0] if a.dim() == 2 else -1
        check(a, "a", (T, OUT_WIDTH))
        check(wo, "wo", (OUT_WIDTH, OUT_WIDTH))
        check(x, "x", (T, OUT_WIDTH))
        if out is None:
            out = torch.empty(T, OUT_WIDTH, dtype=torch.bfloat16, device=self.device)
        check(out, "out", (T, OUT_WIDTH))
        st = load_library().mbert_attn_out_proj(self._h, a.data_ptr(), wo.data_ptr(), x.data_ptr(),
                                                T, out.data_ptr(), _stream_ptr(self.device))
        _check(st, "out_proj")
        return out

    def forward_padded(self, qkv: torch.Tensor, attention_mask: torch.Tensor, layer_kind,
                       out: torch.Tensor = None) -> torch.Tensor:
        """out[B, S, 768] bf16 for a padded batch: qkv [B, S, 2304] bf16 and
        attention_mask [B, S] int32 (1 = real token, 0 = pad) on this device;
        pad rows of out are zeros."""
        kind = _kind(layer_kind)
        if qkv.dim() != 3 or qkv.shape[2] != QKV_WIDTH or qkv.dtype != torch.bfloat16 \
                or qkv.device != self.device or not qkv.is_contiguous():
            raise TypeError(f"qkv must be a contiguous bf16 [B, S, {QKV_WIDTH}] tensor on {self.device}")
        B, S = qkv.shape[0], qkv.shape[1]
        if (attention_mask.dtype != torch.int32 or tuple(attention_mask.shape) != (B, S)
                or attention_mask.device != self.device or not attention_mask.is_contiguous()):
            raise TypeError(f"attention_mask must be a contiguous int32 [{B}, {S}] tensor on {self.device}")
        if out is None:
            out = torch.empty(B, S, OUT_WIDTH, dtype=torch.bfloat16, device=self.device)
        if (out.dtype != torch.bfloat16 or tuple(out.shape) != (B, S, OUT_WIDTH)
                or out.device != self.device or not out.is_contiguous()):
            raise TypeError(f"out must be a contiguous bf16 [{B}, {S}, {OUT_WIDTH}] tensor")
        st = load_library().mbert_attn_forward_padded(self._h, qkv.data_ptr(),
                                                      attention_mask.data_ptr(), B, S, kind,
                                                      out.data_ptr(), _stream_ptr(self.device))
        _check(st, "forward_padded")
        return out

    def ln_qkv(self, x: torch.Tensor, norm_w, wqkv: torch.Tensor, eps: float = NORM_EPS,
               out: torch.Tensor = None) -> torch.Tensor:
        """qkv[T, 2304] bf16 = LayerNorm(x) Wqkv^T: the bias-free pre-attention
        norm (weight norm_w [768], or None for layer 0's identity) and the
        fused Wqkv projection (Wqkv [2304, 768], stored [out, in])."""
        def check(t, name, shape):
            if (t.dtype != torch.bfloat16 or tuple(t.shape) != shape or t.device != self.device
                    or not t.is_contiguous()):
                raise TypeError(f"{name} must be a contiguous bf16 {list(shape)} tensor on {self.device}")
        T = x.shape[0] if x.dim() == 2 else -1
        check(x, "x", (T, OUT_WIDTH))
        if norm_w is not None:
            check(norm_w, "norm_w", (OUT_WIDTH,))
        check(wqkv, "wqkv", (QKV_WIDTH, OUT_WIDTH))
        if out is None:
            out = torch.empty(T, QKV_WIDTH, dtype=torch.bfloat16, device=self.device)
        check(out, "out", (T, QKV_WIDTH))
        st = load_library().mbert_attn_ln_qkv(
            self._h, x.data_ptr(), None if norm_w is None else norm_w.data_ptr(), wqkv.data_ptr(),
            T, float(eps), out.data_ptr(), _stream_ptr(self.device))
        _check(st, "ln_qkv")
        return out

    def mlp(self, x: torch.Tensor, norm_w: torch.Tensor, wi: torch.Tensor, wo: torch.Tensor,
            eps: float = NORM_EPS, out: torch.Tensor = None) -> torch.Tensor:
        """y[T, 768] bf16 = x + (GELU(g) * u) Wo^T, g and u the halves of
        LayerNorm(x) Wi^T (norm_w [768], Wi [2304, 768], Wo [768, 1152], stored
        [out, in]).  `out` may be `x` itself."""
        def check(t, name, shape):
            if (t.dtype != torch.bfloat16 or tuple(t.shape) != shape or t.device != self.device
                    or not t.is_contiguous()):
                raise TypeError(f"{name} must be a contiguous bf16 {list(shape)} tensor on {self.device}")
        T = x.shape[0] if x.dim() == 2 else -1
        check(x, "x", (T, OUT_WIDTH))
        check(norm_w, "norm_w", (OUT_WIDTH,))
        check(wi, "wi", (2 * MLP_INNER, OUT_WIDTH))
        check(wo, "wo", (OUT_WIDTH, MLP_INNER))
        if out is None:
            out = torch.empty(T, OUT_WIDTH, dtype=torch.bfloat16, device=self.device)
        check(out, "out", (T, OUT_WIDTH))
        st = load_library().mbert_attn_mlp(self._h, x.data_ptr(), norm_w.data_ptr(), wi.data_ptr(),
                                           wo.data_ptr(), T, float(eps), out.data_ptr(),
                                           _stream_ptr(self.device))
        _check(st, "mlp")
        return out

    def key_counts(self, cu_seqlens: torch.Tensor, total_tokens: int, layer_kind,
                   max_seqlen: int = 0) -> torch.Tensor:
        """int32 [T]: keys the kernels' schedule and mask admit per query row."""
        kind = _kind(layer_kind)
        self._check_cu(cu_seqlens)
        counts = torch.full((int(total_tokens),), -1, dtype=torch.int32, device=self.device)
        st = load_library().mbert_attn_key_counts(
            self._h, cu_seqlens.data_ptr(), cu_seqlens.numel() - 1, int(total_tokens),
            int(max_seqlen), kind, counts.data_ptr(), _stream_ptr(self.device))
        _check(st, "key_counts")
        return counts

    def selftest_timeout(self, limit_us: int = 20000):
        """Enqueue the bounded-wait self-test (sets the timeout status)."""
        _check(load_library().mbert_attn_selftest_timeout(self._h, int(limit_us),
                                                          _stream_ptr(self.device)),
               "selftest_timeout")

    def profile(self, enable: bool = True):
        """Record a CUDA event pair around every attention, projection and norm kernel."""
        _check(load_library().mbert_attn_profile_enable(self._h, 1 if enable else 0), "profile")

    def profile_read(self):
        """-> ({'global', 'local', 'out_proj', 'qkv_proj', 'layernorm', 'mlp_up',
        'mlp_down'} -> summed kernel ms, the same keys -> kernel count,
        total_launches); synchronises and clears the record."""
        keys = ("global", "local", "out_proj", "qkv_proj", "layernorm", "mlp_up", "mlp_down")
        ms = (ctypes.c_double * len(keys))()
        n = (ctypes.c_int64 * len(keys))()
        tot = ctypes.c_int64()
        _check(load_library().mbert_attn_profile_read(self._h, ms, n, ctypes.byref(tot)),
               "profile_read")
        return ({k: ms[i] for i, k in enumerate(keys)}, {k: n[i] for i, k in enumerate(keys)},
                int(tot.value))

    def get_error(self) -> int:
        """Synchronise and return (and clear) the device-side status."""
        return int(load_library().mbert_attn_get_error(self._h))


_handles = {}


def _default(device) -> Attention:
    idx = device.index if device.index is not None else torch.cuda.current_device()
    h = _handles.get(idx)
    if h is None:
        h = _handles[idx] = Attention(idx)
    return h


def attention(qkv: torch.Tensor, cu_seqlens: torch.Tensor, layer_kind, max_seqlen: int = 0,
              out: torch.Tensor = None) -> torch.Tensor:
    """ModernBERT-base attention for one layer: qkv[T,2304] bf16 (CUDA),
    cu_seqlens int32 [n+1] (CUDA), layer_kind 'global' | 'local' ->
    out[T,768] bf16, enqueued on the current stream."""
    if not qkv.is_cuda:
        raise ValueError("qkv must be a CUDA tensor")
    return _default(qkv.device).forward(qkv, cu_seqlens, layer_kind, max_seqlen, out)


def attention_padded(qkv: torch.Tensor, attention_mask: torch.Tensor, layer_kind,
                     out: torch.Tensor = None) -> torch.Tensor:
    """The attention block for a padded batch: qkv [B, S, 2304] bf16 and
    attention_mask [B, S] int32 (CUDA) -> out [B, S, 768], zeros at pads."""
    if not qkv.is_cuda:
        raise ValueError("qkv must be a CUDA tensor")
    return _default(qkv.device).forward_padded(qkv, attention_mask, layer_kind, out)


def ln_qkv(x: torch.Tensor, norm_w, wqkv: torch.Tensor, eps: float = NORM_EPS,
           out: torch.Tensor = None) -> torch.Tensor:
    """qkv = LayerNorm(x) Wqkv^T (bf16, CUDA tensors; norm_w None on layer 0):
    the step before the attention block."""
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    return _default(x.device).ln_qkv(x, norm_w, wqkv, eps, out)


def mlp(x: torch.Tensor, norm_w: torch.Tensor, wi: torch.Tensor, wo: torch.Tensor,
        eps: float = NORM_EPS, out: torch.Tensor = None) -> torch.Tensor:
    """y = x + (GELU(g) * u) Wo^T after the MLP's LayerNorm (bf16, CUDA tensors)."""
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    return _default(x.device).mlp(x, norm_w, wi, wo, eps, out)


def out_proj(a: torch.Tensor, wo: torch.Tensor, x: torch.Tensor, out: torch.Tensor = None) -> torch.Tensor:
    """y = x + a Wo^T (bf16, CUDA tensors): the step after the attention block."""
    if not a.is_cuda:
        raise ValueError("a must be a CUDA tensor")
    return _default(a.device).out_proj(a, wo, x, out=out)


def key_counts(cu_seqlens: torch.Tensor, total_tokens: int, layer_kind) -> torch.Tensor:
    if not cu_seqlens.is_cuda:
        raise ValueError("cu_seqlens must be a CUDA tensor")
    return _default(cu_seqlens.device).key_counts(cu_seqlens, total_tokens, layer_kind)
