"""libfattn: exact tiled scaled-dot-product attention (FlashAttention) for sm_103a.

The compute path is the C-ABI library ``libfattn.so`` built from ``csrc/``;
``fattn`` is its thin ctypes binding and ``inputs`` the seeded input generator.
Importing this package loads nothing: the binding loads the library on first
use and raises if it is missing.
"""
__all__ = ["fattn", "inputs"]
