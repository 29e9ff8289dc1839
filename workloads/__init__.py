"""Seeded synthetic inputs for tree verification.

Shared by the CPU oracle tests, the GPU parity tests and the bench. It draws
random numbers and builds tree shapes; it computes nothing that the
verification path computes (no attention, no softmax, no acceptance rule).
"""
from .gen import *  # noqa: F401,F403
