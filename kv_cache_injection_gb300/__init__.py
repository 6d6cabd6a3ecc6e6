"""GB300-native retrieve + Chunked RoPE + paged KV injection (InferScale's
serving-time hot path), behind the C ABI of libinjectscale.so.

    from kv_cache_injection_gb300 import api
    store = api.is_store_create(api.make_config(...))

The binding loads the in-tree library on first use and raises if it is
missing; there is no CPU fallback.
"""
from . import api  # noqa: F401
from ._lib import LIB_PATH  # noqa: F401
