"""Seeded synthetic inputs (host generator in ``gen``, device fill in ``fill.cu``, workloads)."""
from . import gen, workloads  # noqa: F401
