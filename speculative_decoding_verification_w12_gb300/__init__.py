"""GB300-native W12 speculative-decoding verify path.

The compute path is the C-ABI library ``libw12.so`` (hand-written sm_103a
kernels); ``w12`` is its thin ctypes binding. Importing the package does not
load the library; the first call into ``w12`` does, and raises if it is
missing or was not built for this GPU.
"""
__version__ = "0.1.0"
