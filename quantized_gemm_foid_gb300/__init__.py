"""GB300 (sm_103a) AdaHOP MXFP4 linear layer.

The compute lives in libadahop.so (C ABI: include/adahop.h); this package is its thin Python
binding.  The library is loaded on first use of any binding name (so that
``quantized_gemm_foid_gb300.build`` can run before it exists); if it has not been built, that
first use raises ImportError.  There is no fallback implementation.
"""
_loaded = False


def _load() -> None:
    global _loaded
    from . import _lib, binding   # raises ImportError when libadahop.so is missing
    g = globals()
    for k in dir(binding):
        if not k.startswith("_"):
            g[k] = getattr(binding, k)
    g.update(LIB=_lib.LIB, PROTOTYPES=_lib.PROTOTYPES, AdahopPlan=_lib.AdahopPlan,
             AdahopOptions=_lib.AdahopOptions)
    _loaded = True


def __getattr__(name):
    if name.startswith("__") or name in ("build", "binding", "_lib"):
        raise AttributeError(name)
    if not _loaded:
        _load()
    try:
        return globals()[name]
    except KeyError:
        raise AttributeError(name) from None
