"""GB300 (sm_103a) fused replicated KV-cache store.

``kvpub`` is the ctypes binding of the C-ABI library ``libkvpub.so``;
``inputs`` draws the seeded synthetic workloads.  Importing the package loads
nothing; the first call into ``kvpub`` loads the library and raises if it has
not been built.
"""

__all__ = ["kvpub", "inputs"]
