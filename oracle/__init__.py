"""CPU oracle of the SpecFold folded verification pass.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg; never by the library or its binding.  Plain
numpy in float64; shares no code with the CUDA path.

Parity status: every function is pinned by the CPU tests (closed forms, hand
fixtures under tests/golden, library special cases and cross-form identities),
except the fold *fraction* a random-init model yields, which the pages only
report for trained checkpoints ("parity unpinned" for that statistic).
"""
from .specfold import *  # noqa: F401,F403
