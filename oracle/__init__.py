"""Float64 CPU oracle of the DFlash hot path.

Test infrastructure only: used by the test-suite, the smoke check and the
bench's CPU-baseline leg; never by the product path.
"""
