"""Plain CPU oracle for the FLUX.3 Image Klein joint ``single_block`` forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` use it.  It shares no code with the
CUDA library (no kernels, headers, tables or helpers); the two meet only in the
seeded input generators of the ``synth`` package, which hold none of the
method's arithmetic.

Every function is written from the published description of the block and
cites the passage it follows:

* "FLUX.3 Image Klein support" (stable-diffusion.cpp issue #2142), comment
  "Structure (from dit.py)": block equation with eps, RoPE ids, tensor names
  and shapes ("Tensor names (distilled checkpoint)").
* "Welcome FLUX.3 Image Klein in Diffusers", sections "Inside one block"
  (block pseudocode), "Positions in four dimensions" (RoPE id table),
  "Two stages" (full joint attention).

Parity pins: see ``tests/test_oracle_pins.py``.  Functions whose result has no
pin beyond the invariants listed there are marked "parity unpinned" in their
docstring.
"""

from .flux3_oracle import *  # noqa: F401,F403
from . import nvfp4  # noqa: F401
from . import fp8r  # noqa: F401
from . import flux3_model  # noqa: F401
