"""Test infrastructure: the fp64 oracle.  Only tests/, the smoke check and the benchmark's
CPU-baseline leg import this package; the library never does."""
