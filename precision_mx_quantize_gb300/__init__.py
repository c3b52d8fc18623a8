"""GB300-native MX (microscaling) quantized-training kernels.

The compute lives in a C-ABI CUDA library (``libmxq.so``) built for sm_103a;
this package holds its thin ctypes binding and the seeded input generators.
"""
