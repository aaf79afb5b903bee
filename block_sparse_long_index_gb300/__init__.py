"""GB300 (sm_103a) forward path of MiniMax Sparse Attention (MSA).

The product is ``libmsa.so`` (hand-written CUDA kernels behind the C ABI of
``include/msa.h``).  ``msa`` binds that ABI under the same names; ``api``
adds tensor-level helpers.  Importing the package loads the library and raises
if it is not built: there is no CPU or eager fallback.
"""
from . import msa  # noqa: F401  (loads libmsa.so, fails loudly if missing)
from .api import MsaDecode, MsaPrefill, decode, prefill  # noqa: F401
