"""CPU oracle for the NVFP4 MoE expert computation (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product library never does.
"""
