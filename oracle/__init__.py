"""CPU oracle for INT8-KV decode attention.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the bench's
CPU-baseline leg may import this package; the product path never does.  The
arithmetic lives in ``kvq8_oracle.c`` (plain C, fp32 quantisation, fp64
attention); ``oracle.py`` loads it with ctypes and adds per-unit drivers.
"""
from .oracle import *  # noqa: F401,F403
