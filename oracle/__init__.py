"""Float64 CPU oracle for masked second-order HLA (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU legs use this package.
"""
