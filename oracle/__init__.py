"""CPU oracle for the block-scaled fused dequantizing matmul -- TEST INFRASTRUCTURE.

A plain, slow, obviously correct numpy implementation of what the library
computes: format codecs (``codec``), the reference packer (``pack``), and the
exact float64 dequant / dequant-then-dot matmul with its error bound
(``reference``).  It shares no code with the CUDA/C++ library and the library
never imports it; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use it.

Every function is pinned by ``tests/test_oracle_*.py`` against facts fixed by
the pages and by mathematics (printed codebooks, closed forms, library
decoders, exact rational brute force).  No function here is "parity unpinned".
"""
from . import codec, pack, reference  # noqa: F401
from .pack import BLOCK, FORMATS, codes_nbytes, scales_nbytes  # noqa: F401
from .reference import dequant_exact, dequant_f32, qmm_ref, qmm_ref_sampled  # noqa: F401
