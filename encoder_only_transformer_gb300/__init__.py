"""ModernBERT-base bidirectional attention block, GB300-native (sm_103a).

The compute path is the C-ABI library ``libmbert_attn.so`` built from
``csrc/`` (hand-written tcgen05/TMA kernels); ``binding`` marshals arguments
to it.  Importing this package does not load the library: ``attention`` and
the other entry points load it on first use and raise if it is missing.
"""
_BINDING_NAMES = {
    "attention", "key_counts", "Attention", "MbertAttnError", "load_library",
    "GLOBAL", "LOCAL", "library_path",
}

__all__ = sorted(_BINDING_NAMES)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
