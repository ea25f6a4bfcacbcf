"""GB300-native OasisKV lookahead sparse decode hot path.

The compute path is the CUDA library ``liboasis.so`` (built from ``csrc/``);
``binding`` marshals torch tensors into its C ABI.  ``synthetic`` draws the
seeded inputs.  Importing the package does not load the library.
"""
__all__ = ["binding", "synthetic"]
