"""CPU oracle for order-independent floating-point summation.

Test infrastructure only: the test suite, the smoke check and the benchmark's
CPU-baseline leg are its only users.  The product library never imports it.
"""
from .oracle import *  # noqa: F401,F403
