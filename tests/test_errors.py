"""GPU error paths: host-side checks, device-side cu_seqlens checks and the
bounded-wait timeout status.  Nothing here faults, traps or hangs a GPU:
device checks set the error word and the kernels return."""
import ctypes

import pytest
import torch

from encoder_only_transformer_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import __graft_entry__
    __graft_entry__.build()
    h = binding.Attention(0)
    yield h
    h.get_error()
    h.close()


def _fwd_raw(attn, qkv_ptr, cu, n, T, max_seqlen, kind, out_ptr):
    return binding.load_library().mbert_attn_forward(
        attn.handle, qkv_ptr, cu.data_ptr(), n, T, max_seqlen, kind, out_ptr,
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("cu_list,expect", [
    ([0, 50, 40, 100], -4),      # decreasing
    ([3, 50, 100], -4),          # cu[0] != 0
    ([0, 50, 99], -4),           # cu[n] != T
])
def test_bad_cu_seqlens_detected_on_device(attn, cu_list, expect):
    T = 100
    wl = W.custom([T], seed=1)
    qkv = wl.qkv.cuda()
    cu = torch.tensor(cu_list, dtype=torch.int32, device="cuda")
    out = torch.full((T, 768), 7.0, dtype=torch.bfloat16, device="cuda")
    rc = _fwd_raw(attn, qkv.data_ptr(), cu, len(cu_list) - 1, T, 0, 0, out.data_ptr())
    assert rc == 0                       # host checks pass; the device finds it
    assert attn.get_error() == expect
    assert torch.all(out == 7.0)         # nothing written
    assert attn.get_error() == 0         # cleared
    # the handle keeps working afterwards
    good = attn.forward(qkv, torch.tensor([0, T], dtype=torch.int32, device="cuda"), "local")
    torch.cuda.synchronize()
    assert attn.get_error() == 0 and torch.isfinite(good.float()).all()


def test_sequence_longer_than_bound(attn):
    wl = W.custom([300], seed=2)
    qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
    out = torch.zeros(300, 768, dtype=torch.bfloat16, device="cuda")
    rc = _fwd_raw(attn, qkv.data_ptr(), cu, 1, 300, 200, 0, out.data_ptr())
    assert rc == 0
    assert attn.get_error() == -3
    assert torch.all(out == 0)


# The local kernel validates cu_seqlens itself on two of its paths: one lane
# per sequence for up to 32 sequences, a warp-wide pass for up to 256; with
# more sequences the plan kernel checks first.  Each path must report the
# defect and write nothing.
LOCAL_PATHS = {"per_lane": 3, "warp_pass": 40, "plan_kernel": 300}


@pytest.mark.parametrize("defect", ["decreasing", "first_not_zero", "last_not_total", "too_long"])
@pytest.mark.parametrize("path", list(LOCAL_PATHS))
def test_local_layer_device_checks(attn, path, defect):
    n = LOCAL_PATHS[path]
    T = 2 * n                                 # n sequences of 2 tokens
    cu_list = list(range(0, T + 1, 2))
    max_seqlen = 0
    if defect == "decreasing":
        cu_list[n // 2] = cu_list[n // 2 + 1] + 1
    elif defect == "first_not_zero":
        cu_list[0] = 1
    elif defect == "last_not_total":
        cu_list[-1] = T - 1
    else:
        max_seqlen = 1                        # every sequence is longer
    wl = W.custom([T], seed=4)
    qkv = wl.qkv.cuda()
    cu = torch.tensor(cu_list, dtype=torch.int32, device="cuda")
    out = torch.full((T, 768), 7.0, dtype=torch.bfloat16, device="cuda")
    rc = _fwd_raw(attn, qkv.data_ptr(), cu, n, T, max_seqlen, 1, out.data_ptr())
    assert rc == 0
    assert attn.get_error() == (-3 if defect == "too_long" else -4)
    assert torch.all(out == 7.0)              # nothing written
    good = attn.forward(qkv, torch.arange(0, T + 1, 2, dtype=torch.int32, device="cuda"), "local")
    torch.cuda.synchronize()
    assert attn.get_error() == 0 and torch.isfinite(good.float()).all()


def test_host_checks(attn):
    wl = W.custom([64], seed=3)
    qkv, cu = wl.qkv.cuda(), wl.cu_seqlens.cuda()
    out = torch.empty(64, 768, dtype=torch.bfloat16, device="cuda")
    lib = binding.load_library()
    # bad kind, misaligned pointers, overlap, too-long bound, null pointers
    assert _fwd_raw(attn, qkv.data_ptr(), cu, 1, 64, 0, 2, out.data_ptr()) == -1
    assert _fwd_raw(attn, qkv.data_ptr() + 2, cu, 1, 64, 0, 0, out.data_ptr()) == -1
    assert _fwd_raw(attn, qkv.data_ptr(), cu, 1, 64, 0, 0, out.data_ptr() + 8) == -1
    assert _fwd_raw(attn, qkv.data_ptr(), cu, 1, 64, 0, 0, qkv.data_ptr() + 4608) == -1
    assert _fwd_raw(attn, qkv.data_ptr(), cu, 1, 64, 9000, 0, out.data_ptr()) == -3
    assert _fwd_raw(attn, 0, cu, 1, 64, 0, 0, out.data_ptr()) == -1
    assert _fwd_raw(attn, qkv.data_ptr(), cu, 0, 64, 0, 0, out.data_ptr()) == -1
    assert _fwd_raw(attn, qkv.data_ptr(), cu, 1, -1, 0, 0, out.data_ptr()) == -1
    # T == 0 is a no-op
    empty = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.mbert_attn_forward(attn.handle, 0, empty.data_ptr(), 0, 0, 0, 0, 0, None) == 0
    with pytest.raises(TypeError):
        attn.forward(qkv.float(), cu, "global")
    with pytest.raises(ValueError):
        attn.forward(qkv, cu, "sideways")
    assert attn.get_error() == 0


def test_bounded_wait_reports_timeout(attn):
    """A barrier that nothing completes: the wait gives up after 20 ms, the
    kernel returns, and the host reads the timeout status."""
    attn.selftest_timeout(20000)
    assert attn.get_error() == -5
    assert attn.get_error() == 0
    wl = W.config(1)
    out = attn.forward(wl.qkv.cuda(), wl.cu_seqlens.cuda(), "global")
    torch.cuda.synchronize()
    assert attn.get_error() == 0 and torch.isfinite(out.float()).all()


def test_create_rejects_unsupported_shapes():
    lib = binding.load_library()
    h = ctypes.c_void_p()
    cfg = binding.Config()
    lib.mbert_attn_default_config(ctypes.byref(cfg))
    cfg.head_dim = 128
    assert lib.mbert_attn_create(ctypes.byref(h), ctypes.byref(cfg), 0) == -2
    lib.mbert_attn_default_config(ctypes.byref(cfg))
    assert lib.mbert_attn_create(ctypes.byref(h), ctypes.byref(cfg), 99) == -1
