"""FP64 CPU oracle for the CODA GEMM-epilogue hot path.

TEST INFRASTRUCTURE ONLY. Nothing in the product (the C-ABI library and its
Python binding) imports, links or calls this package. Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) use it.

Every function is a plain, unfused NumPy float64 statement of what one step of
the method computes, written from the pages that describe CODA ("CODA:
Rewriting Transformer Blocks as GEMM-Epilogue Programs"):

* "CODA note" = the papernotes.org note on the paper; its method section has
  Key designs 1-4 (reparameterisation and delayed row scale; pairwise maps;
  backward duality and the row-statistic identity; the five epilogue
  primitives) and the kernel / block speedup tables.
* "pith page" = the pith.science page on arXiv 2605.19269 (figure captions,
  Appendix A.1 on the tile-wise backward epilogue).

Inputs are the exact bfloat16 values a kernel consumed, upcast to float64.
The oracle shares no code with the CUDA path; its only common dependency is
the seeded input generator ``coda_inputs``.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
identities stated on the pages, torch float64 library routines (autograd,
rms_norm, silu, cross_entropy, logsumexp), closed forms, finite differences
and brute-force scalar loops. Parity with values printed on the pages is
unpinned: the pages print no worked numeric example.
"""
from .ref import *  # noqa: F401,F403
from .ref import __all__  # noqa: F401
