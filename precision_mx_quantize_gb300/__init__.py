"""GB300-native MX (microscaling) quantized-training kernels.

The compute lives in a C-ABI CUDA library (``libmxq.so``) built for sm_103a
by ``build.py``.  This package holds its thin ctypes binding (``mxq``), the
MXFP8 all-gather of dim-0 weight shards over ``torch.distributed``
(``fsdp_gather``) and the seeded input generators (``synth``).
"""
