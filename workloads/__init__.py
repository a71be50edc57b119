"""Seeded synthetic workloads (inputs only, no arithmetic of the method) shared by
the tests, the smoke check and the benchmark: the generators in ``inputs`` and
the copies of their arrays to the GPU in ``device``."""
