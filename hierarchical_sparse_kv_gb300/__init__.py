"""GB300-native ZoomR decode step: summary score -> top-k -> paged gather -> attention.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA kernels
(``csrc/``, declared in ``include/zoomr.h``). ``zoomr`` is its thin ctypes
binding; ``workloads`` draws seeded synthetic inputs; ``accounting`` counts
tokens and bytes. Importing this package does not load the library.
"""

__all__ = ["workloads", "accounting", "zoomr"]
