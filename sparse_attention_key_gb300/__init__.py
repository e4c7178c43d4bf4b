"""GB300-native Lightning Indexer (sm_103a).

The indexer scores every causal key of a query with the head-weighted sum of
relu(q_h . k) over 32 heads of 128 dims and keeps the best 2048 positions
exactly, under the tie/order rule of "Notes from an NVFP4 port of Kimi K3.1
Pro". The work runs in a C-ABI CUDA library (``csrc/``, header
``include/lightning_indexer.h``); ``binding`` marshals torch tensors into it.

``workloads`` holds the seeded synthetic inputs. Importing the package does not
load the CUDA library; the first call into ``binding`` does, and raises if the
library has not been built.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads", "binding"]


def __getattr__(name):
    if name == "binding":
        import importlib
        return importlib.import_module(__name__ + ".binding")
    raise AttributeError(name)
