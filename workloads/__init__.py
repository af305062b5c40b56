"""Seeded synthetic workloads shared by the tests, the bench and the smoke run."""
from . import configs, gen  # noqa: F401
