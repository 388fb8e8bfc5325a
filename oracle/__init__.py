"""Float64 CPU oracle of the EntropyCache denoising step (test infrastructure only).

Importable by the tests, the smoke check and the benchmark's CPU-baseline leg; never by the
product path.
"""
from .entropycache_oracle import *  # noqa: F401,F403
from .entropycache_oracle import __all__  # noqa: F401
