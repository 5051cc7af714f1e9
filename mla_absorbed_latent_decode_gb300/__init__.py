"""GB300-native absorbed-MLA latent decode.

The compute path is ``libmla.so`` (hand-written sm_103a CUDA kernels behind a C
ABI, declared in ``include/mla.h``); :mod:`.binding` is a thin ctypes layer over
it.  :mod:`.workloads` draws seeded synthetic inputs.
"""
