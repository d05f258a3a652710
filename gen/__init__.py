"""Seeded synthetic-input generators (shared by tests, bench and oracle checks)."""
from .synth import *  # noqa: F401,F403
from .synth import WORKLOADS, workload, sample_rows  # noqa: F401
