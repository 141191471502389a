"""fp64 CPU oracle of standard attention -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product library never imports,
links or falls back to it, and it shares no code with the CUDA path.
"""
