"""CPU-side checks of the C-ABI library: it builds, loads, exports every
symbol include/mbert_attn.h declares, and its host-only logic behaves.
No GPU compute is called here."""
import ctypes
import os
import re
import subprocess

import pytest

from encoder_only_transformer_gb300 import binding, build as pkg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mbert_attn.h")


@pytest.fixture(scope="module")
def lib():
    pkg_build.build()
    return binding.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mbert_attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("mbert_attn_create", "mbert_attn_forward", "mbert_attn_destroy",
              "mbert_attn_key_counts", "mbert_attn_get_error", "mbert_attn_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"
    # the binding knows every one of them too
    assert set(names) == set(binding.SIGNATURES)
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (mbert_attn_\w+)", out))
    assert exported == set(names), exported ^ set(names)


def test_library_is_built_for_sm103a():
    """Every object carries sm_103a code (read from nvcc's own flags, not
    from the binary)."""
    assert "arch=compute_103a,code=sm_103a" in " ".join(pkg_build.ARCH)


def test_strerror_and_default_config(lib):
    assert binding.strerror(0) == "success"
    assert "cu_seqlens" in binding.strerror(-4)
    assert binding.strerror(12345) == "unknown status"
    cfg = binding.Config()
    assert lib.mbert_attn_default_config(ctypes.byref(cfg)) == 0
    assert (cfg.heads, cfg.head_dim, cfg.half_window, cfg.max_seqlen) == (12, 64, 64, 8192)
    assert (cfg.theta_global, cfg.theta_local) == (160000.0, 10000.0)
    assert lib.mbert_attn_default_config(None) == -1


def test_host_argument_checks_without_device(lib):
    """Host-side checks fail synchronously before touching a device."""
    assert lib.mbert_attn_forward(None, None, None, 1, 10, 0, 0, None, None) == -1
    assert lib.mbert_attn_key_counts(None, None, 1, 10, 0, 0, None, None) == -1
    assert lib.mbert_attn_get_error(None) == -1
    assert lib.mbert_attn_reserve(None, 1, 1) == -1
    lib.mbert_attn_destroy(None)
    h = ctypes.c_void_p()
    cfg = binding.Config()
    lib.mbert_attn_default_config(ctypes.byref(cfg))
    cfg.heads = 16
    assert lib.mbert_attn_create(ctypes.byref(h), ctypes.byref(cfg), 0) == -2
    lib.mbert_attn_default_config(ctypes.byref(cfg))
    cfg.half_window = -3
    assert lib.mbert_attn_create(ctypes.byref(h), ctypes.byref(cfg), 0) == -1
    assert lib.mbert_attn_create(None, None, 0) == -1


def test_binding_rejects_bad_kinds():
    with pytest.raises(ValueError):
        binding._kind("causal")
    assert binding._kind("global") == 0 and binding._kind("local") == 1


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(OSError):
        binding.load_library(str(tmp_path / "nope.so"))
