"""GB300-native Megatron tensor-parallel Transformer block.

The compute path is the C-ABI library ``libtp.so`` (CUDA kernels for
sm_103a), declared in ``include/tp.h``; ``binding`` is a thin ctypes layer
over it.  Importing this package does not load the library; ``binding.lib()``
does, and raises if it has not been built.
"""

__version__ = "0.1.0"
