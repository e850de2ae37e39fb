"""Speculative pipeline decoding on one GB300: the pipeline step, the Pipeline Draft
Module and device-side streaming verification, as hand-written sm_103a CUDA behind the C
ABI in include/spd.h.  ``binding`` mirrors the ABI; ``engine.Engine`` is a thin wrapper
that lets PyTorch own device memory and streams."""
from . import binding  # noqa: F401

__all__ = ["binding", "engine", "build"]
