"""CPU oracle for the ZeRO sharded-optimizer step (test infrastructure only).

Imported by the test suite, the package smoke check and the benchmark's CPU
baseline leg; never by the product path.
"""
from .zero_oracle import *  # noqa: F401,F403
from .zero_oracle import __all__  # noqa: F401
