"""CPU oracle for context-parallel ring attention — TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct statement of what the
library computes, written in numpy float64 from the page
"G5 上下文并行建模设计规格" (G5 context-parallel modelling design spec, v1.1.1).
It exists to check the CUDA path, never to stand in for it:

* only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
  ``--impl reference`` legs of ``bench.py`` may import it;
* it shares no code with ``context_ring_attention_cp_gb300`` and imports
  nothing from it (inputs arrive as numpy arrays; bf16 inputs arrive as raw
  uint16 bit patterns and are decoded here exactly);
* every function cites the passage of the page it restates.

Modules
-------
``attention``  full causal softmax attention, row-sampled causal attention and
               pass-Q decode attention, by their plain definition.
``ring``       the balanced head/tail chunk plan, the ring schedule, the
               per-(rank, step) partial triple, the LSE merge and the
               ring restatement that merges all steps.
``comm``       the closed-form byte counts (pass-KV ring volume, pass-Q
               dispatch/reduce message sizes) as exact Python integers.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
something other than itself (arbitrary-precision brute force, closed forms,
algebraic invariants, integers printed on the page). No function is
"parity unpinned".
"""

from . import attention, comm, ring  # noqa: F401
from .attention import bf16_bits_to_f64  # noqa: F401
