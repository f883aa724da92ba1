"""GB300-native KPool DSA indexer (sm_103a CUDA kernels behind a C ABI).

The binding (``binding.py``) loads ``libkpool.so`` on first use of any
``kpool_*`` name and raises ImportError if the library has not been built;
there is no fallback path.  ``workloads`` (seeded synthetic inputs) imports
without the library.
"""
import importlib

__version__ = "1.0.0"


def __getattr__(name):
    if name.startswith("kpool_") or name in ("KPoolError", "new_workspace", "LIB_PATH",
                                             "STATUS_TIMEOUT", "STATUS_BAD_SEQLENS"):
        mod = importlib.import_module(".binding", __name__)
        return getattr(mod, name)
    raise AttributeError(name)
