"""Exact scaled-dot-product attention forward for GB300 (sm_103a).

The compute path is the C-ABI library ``libattn.so`` built from ``csrc/``
(hand-written CUDA: TMA, tcgen05 MMAs accumulating in tensor memory, online
softmax). ``attn`` is its thin ctypes binding; ``synth`` draws the seeded
synthetic inputs. Importing the package loads nothing; the library is opened
on the first call and a missing library is an error, never a fallback.
"""
from .attn import fwd, library_path, load_library, AttnError  # noqa: F401
