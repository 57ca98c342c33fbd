"""B300-native (sm_103a) Mamba selective-scan library.

The compute path is the C-ABI shared library ``libmamba_ssm.so`` built from
``csrc/``; ``ops`` is a thin ctypes binding over it (argument marshalling
only).  Importing this package loads nothing; the first call through ``ops``
loads the library and raises if it is missing.
"""
__all__ = ["inputs", "ops"]
