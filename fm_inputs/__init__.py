"""Seeded synthetic inputs (bound vectors, Q/K/V/dO, chunk maps) shared by the
CPU oracle's tests, the CUDA library's tests and the benchmark.  This package
holds no attention arithmetic."""
from . import masks, tensors, configs  # noqa: F401
