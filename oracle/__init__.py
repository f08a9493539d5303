"""fp64 CPU oracle for the MSA hot path.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package's smoke check
and by the benchmark's CPU-baseline leg, never by the product path.
"""
