"""GB300-native MLA decode attention, weight-absorbed without materialisation.

The compute path is libmla_decode.so (hand-written sm_103a CUDA: tcgen05/TMEM
MMAs fed by TMA); this package is its ctypes binding plus the seeded input
generator.  See include/mla_decode.h for the C ABI.
"""
from .binding import Dims, MlaDecode, MlaDecodeError, decode, dims_for, lib  # noqa: F401
