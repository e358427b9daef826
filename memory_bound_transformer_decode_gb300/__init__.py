"""GB300-native batch-B INT4 GQA transformer decode step.

The compute path is a C-ABI shared library of hand-written CUDA kernels for
sm_103a (``include/ddl.h``); this package holds its thin ctypes binding
(``ddl``), the workload shapes (``configs``), the seeded input generator
(``synth``) and the bytes/FLOPs model (``roofline``).
"""
from . import configs, roofline, synth  # noqa: F401

__all__ = ["configs", "roofline", "synth"]
