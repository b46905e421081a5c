"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench."""
from .workloads import *  # noqa: F401,F403
