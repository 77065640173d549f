"""CPU oracle of the DFlash 2 block drafter — TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 numpy restatement of what the drafter computes, written
from the page "cortiq-engine 0.8.71 — src/dflash.rs" (the drafter and its
host block) with the number formats of ``oracle.quant``.  It exists to check
the CUDA library against: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product (``block_speculative_drafting_gb300``) never imports, links or
calls anything here, and nothing here imports the product: the two share only
the seeded input generators of ``workloads``.

Pins (``tests/test_oracle_*.py``): brute-force attention and softmax on tiny
inputs and a library attention routine; incremental append equal to a full
recomputation; the dequantised matvec equal to the integer group-sum
definition; RMSNorm's unit RMS and RoPE's norm preservation and relative
position property; the page's own ``top_k`` example; a closed form of the
head path; SiLU identities.  The end-to-end block has no printed values on
the pages: its composition is pinned only through those parts.
"""
from . import quant  # noqa: F401
from .drafter import (OracleModel, OracleSeq, Matrix, argmax_first, attention, block, inv_freq,  # noqa: F401
                      rms, rope, silu, softmax, top_k, row_conv, select)
