"""CPU oracle for the convrot linear — test infrastructure only.

Imported by the tests, the smoke check and the benchmark's CPU-baseline leg;
never by the library.
"""
from .convrot_oracle import *  # noqa: F401,F403
from .convrot_oracle import __all__  # noqa: F401
