"""CPU oracle for the GPUOS micro-op dispatcher -- TEST INFRASTRUCTURE ONLY.

``oracle.c`` holds the plain double-precision definitions of every micro-op;
``interp`` applies a descriptor stream to host copies of its buffers in
ticket order (sequential semantics), the meaning the dispatcher must
reproduce ("GPUOS: A GPU Operating System Primitive for Transparent
Operation Fusion", §2: "don't launch, call" changes how work is issued, not
what it computes).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product path never does, and the oracle
imports nothing from the product package.

Parity pins: every function is pinned in ``tests/test_oracle_pins.py`` by a
closed form, a special case, a brute-force evaluation or a printed constant
(see each test's docstring). No function is "parity unpinned".
"""
