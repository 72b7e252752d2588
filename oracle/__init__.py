"""CPU oracle for the 2:4 sparse FFN training path — TEST INFRASTRUCTURE ONLY.

This package is the slow, obviously-correct statement of what the GPU path
computes. It exists to check the CUDA kernels and nothing else: only the test
suite, the package's smoke check and the bench's CPU-baseline leg may import
it. The product path (the C-ABI library and its Python binding) never imports,
links or runs anything in here, and shares no code, tables or helpers with it.

Module map:
  prune24_oracle  bf16 rounding, the 2:4 magnitude pruner, compression into
                  values + 2-bit metadata, decompression, the double prune of
                  the transposed weight, fp32-accumulated GEMMs on the pruned
                  operands, masked weight gradient, bias gradients and the
                  full FFN training step composed from them.

Parity status: every function is pinned by tests/test_oracle_pins.py against
brute force, closed forms, hand-worked fixtures in tests/golden/ or an
independent library routine; none is "parity unpinned".
"""
