"""GB300 (sm_103a) Mamba-1 selective scan: the C-ABI library's Python binding.

The compute runs in ``libssm_gb300.so`` (hand-written CUDA kernels); this
package only marshals arguments.  Importing it does not load the library; the
first call (or ``load()``) does, and raises if the library has not been built.
"""
from .binding import *  # noqa: F401,F403
from .binding import __all__ as _binding_all

__all__ = list(_binding_all)
