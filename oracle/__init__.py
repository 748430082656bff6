"""CPU oracle of the GPT training step (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  It shares no code with the CUDA path.
"""
from .gpt_oracle import *  # noqa: F401,F403
