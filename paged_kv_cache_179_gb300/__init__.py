"""paged_kv_cache_179_gb300: the decode-step hot path of a paged KV cache on GB300.

The compute lives in libpa.so (CUDA for sm_103a, C ABI in include/pa.h);
``paged_kv_cache_179_gb300.ops`` binds it for torch tensors.  Importing this
package loads nothing; the library is loaded on first use.
"""
__all__ = ["ops", "workloads", "build"]


def __getattr__(name):
    if name == "ops":
        from . import _abi as ops
        return ops
    if name in ("workloads", "build"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
