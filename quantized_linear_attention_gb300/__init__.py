"""Per-window int8 recurrent-state decode for Gated DeltaNet / KDA on GB300 (sm_103a).

The hot path (append each token, fold each window) runs in hand-written CUDA
kernels inside the C-ABI library ``liblq.so`` (declared in ``include/lq.h``).
``lq`` is its thin ctypes binding; ``workload`` draws the seeded synthetic
inputs. Importing the package loads nothing: the CUDA library is loaded on the
first call into ``lq`` and a missing library raises.
"""
__all__ = ["lq", "workload"]
