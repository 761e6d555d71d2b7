"""B300-native (sm_103a) DeepSeek-V4 hybrid-attention forward: CSA + HCA + sliding window.

The compute path is the C-ABI CUDA library ``libhyb.so`` (include/hyb.h);
``ops`` is its thin torch binding and ``pipeline.HybridStep`` chains the five
calls into one forward step; ``session.DecodeSession`` runs token-by-token decode
over the heterogeneous KV cache.  ``workloads`` holds the benchmark shapes and the
seeded synthetic inputs.
"""
from . import workloads  # noqa: F401  (pure-python, no library needed)

__all__ = ["ops", "pipeline", "session", "workloads", "build"]


def __getattr__(name):
    if name in ("ops", "pipeline", "session", "build", "_abi"):
        import importlib

        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
