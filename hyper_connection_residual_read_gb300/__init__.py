"""GB300 hyper-connection residual read: a C-ABI CUDA library and its Python binding.

``synth`` (seeded inputs) imports without the library. The read itself
(``hc_read`` and friends) loads ``libhcread.so`` on first use and raises if it is
missing: there is no fallback implementation.
"""
from . import synth  # noqa: F401

_BINDING = ("hc_read_init", "hc_read", "hc_read_path", "hc_read_check", "hc_read_status",
            "hc_read_noalloc", "hc_read_upmix", "hc_read_lo_bf16", "hc_read_y",
            "hc_read_set_wait_limit", "hc_read_bounds_checked",
            "hc_read_shutdown", "hc_read_version", "strerror", "HcReadError", "load",
            "HC_PATH_AUTO", "HC_PATH_DECODE", "HC_PATH_PREFILL", "HC_PATH_PREFILL_UNFUSED",
            "HC_PATH_DECODE_ONE_KERNEL", "HC_PATH_PREFILL_BF16_LO",
            "HC_OK", "HC_ERR_ARG", "HC_ERR_NOT_INIT", "HC_ERR_ARCH", "HC_ERR_CUDA",
            "HC_ERR_TIMEOUT", "HC_ERR_CHECK", "HC_ERR_NOMEM", "HC_ERR_BOUNDS",
            "EXPORTS", "LIB_PATH")


def __getattr__(name):
    if name in _BINDING:
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
