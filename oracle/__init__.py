"""Plain CPU oracle for the all-to-all permutations and the one-sided primitives.

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only tests, the smoke check and the
benchmark's CPU-baseline leg may import it.  See ``a2a_oracle.c``.
"""
from .oracle import Oracle, build, load, load_openmp  # noqa: F401
