"""CPU oracle for the sharded mixed-precision AdamW step over a flat, padded buffer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the CUDA library and its Python binding) never
imports, links or runs anything here, and this package imports nothing from
the product: the two share no code, tables or helpers.

What it computes is the plain definition of the method described in
"Infra: Data Parallel" (F. Pu), sections "Zero Redundancy Optimizer (ZeRO)"
and "Fully Sharded Data Parallel (FSDP)":

* ``layout``      - the FSDP1 FlatParameter: flatten, concatenate, pad, shard,
                    bucket (FSDP1 layout figure; ZeRO memory figure).
* ``numerics``    - bf16 round-to-nearest-even and fp32 widening, written
                    from the IEEE-754 definition on bit patterns.
* ``steps``       - micro-batch accumulation, Reduce-Scatter with averaging,
                    element-wise AdamW on a shard, All-Gather, the ZeRO-3
                    per-unit gather / reduce-scatter, and naive DP.
* ``accounting``  - model-state bytes held and bytes sent per rank, obtained
                    by counting the buffers each rank holds and the elements
                    that cross ranks in the simulated collectives.

Arithmetic is numpy float32, one IEEE-rounded operation per line, because the
pages fix the optimizer state to fp32 (k = 12 bytes per parameter: fp32 master
weights and both moments) and parameters/gradients to 16 bits.  bf16 values
are carried as ``numpy.uint16`` bit patterns.

Every function here is pinned by a ``-m "not gpu"`` test against something
other than itself (worked examples printed on the pages, closed forms,
brute force over tiny cases, exact rational arithmetic, library routines).
No function is "parity unpinned".
"""

from . import accounting, layout, numerics, steps  # noqa: F401
