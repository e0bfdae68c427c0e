"""GB300-native fused MoE-LoRA expert layer.

The compute lives in a C-ABI shared library (``libmoelora.so``, CUDA for
sm_103a) declared in ``include/moelora.h``; ``binding`` marshals arguments
to it.  Importing this package loads nothing: ``binding.load()`` does, and
raises if the library has not been built.
"""
__version__ = "0.1.0"
