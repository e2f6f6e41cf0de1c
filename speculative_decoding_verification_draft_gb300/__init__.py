"""GB300-native batched speculative-decoding verification and Saguaro pre-speculation.

The compute path is the CUDA library ``libssdv.so`` (hand-written sm_103a
kernels behind the C ABI declared in ``include/ssdv.h``).  ``ssdv`` is its thin
ctypes binding; ``workloads`` builds seeded synthetic inputs.  The binding is
imported lazily so that ``workloads`` can be used on machines without a GPU.
"""

__all__ = ["ssdv", "workloads"]


def __getattr__(name):
    if name in ("ssdv", "workloads"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
