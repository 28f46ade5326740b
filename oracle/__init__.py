"""Plain, slow, obviously-correct CPU oracle for the NVFP4 + LoRA + AQN-RMSNorm linear.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or run
anything in this package: only the test suite (``tests/``), the smoke check in
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of ``bench.py``
use it.  It shares no code, table, header or constant generator with the CUDA
library under ``precision_linear_gb300/``; the two meet only on the seeded
synthetic inputs that ``precision_linear_gb300.synthetic`` draws.

What it computes, and where the pages define it:

* ``oracle.nvfp4`` -- the NVFP4 storage format and the fixed-scale nearest-grid
  quantiser (QeRL: When Quantized Weights Help Reinforcement Learning, and Where
  the Evidence Stops -- section 3.1 "What the four bits represent": E2M1 grid,
  E4M3 block scale per 16 weights, FP32 tensor scale, reconstruction equation,
  argmin equation, 9P/16 storage equation).
* ``oracle.linear`` -- dequantisation, RMSNorm with the AQN noise folded into the
  norm scale (same page, section 5.1 "Deriving the RMSNorm identity") and the
  LoRA forward on the frozen quantised backbone (same page, section 2.1 "Weight
  storage and trainable state are different budgets", forward-map equation).

Floating point is FP64 except where the quantiser's code selection is defined
as a fixed sequence of IEEE FP32 operations (see ``oracle.nvfp4``); that is the
contract the GPU quantiser must reproduce bit for bit.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py`` against
values the pages print, closed forms, library routines and brute force.  No
function is "parity unpinned".
"""

from . import nvfp4, linear  # noqa: F401
