"""CPU fp64 oracle for causal grouped-query attention.

Test infrastructure only: the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg use it. The GPU library never imports it.
"""
