"""Low-bit KV-cache decode attention for GB300 (sm_103a).

The compute path lives in the CUDA shared library ``libkvq.so`` built from
``csrc/``; ``binding`` is a thin ctypes layer over its C ABI (declared in
``include/kvq.h``).  ``workloads`` and ``synth`` describe and draw the
synthetic decode workloads.
"""
__all__ = ["binding", "workloads", "synth"]
