"""Single-GPU mixture-of-experts layer for GB300 (sm_103a): a C-ABI CUDA
library (libmoe.so, include/moe.h) and a thin ctypes binding with the same
names.  Importing the package does not load the library; the first call does,
and fails loudly if it was not built."""

from .configs import CONFIGS, LayerConfig  # noqa: F401
