"""CPU oracle for the AWQ scale search.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the ``smoke()`` check and
by the benchmark's CPU-baseline leg, never by the product path.
"""
from .awq_oracle import *  # noqa: F401,F403
from .awq_oracle import __all__  # noqa: F401
