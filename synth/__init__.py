"""Seeded synthetic inputs for the paged decode path (shared by the tests,
the benchmark and the oracle checks). Holds shapes, lengths, block placement
and random values only: none of the attention or cache arithmetic."""
from .configs import PRESETS, DecodeConfig, get  # noqa: F401
from .structure import PAD_BLOCK, Structure, build, build_grouped  # noqa: F401
