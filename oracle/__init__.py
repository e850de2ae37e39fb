"""CPU oracle for speculative pipeline decoding — TEST INFRASTRUCTURE.

A plain, slow, fp64 restatement of what the method computes, written from the
source pages (speculative pipeline decoding, arXiv 2605.30852: the abstract, the
machine review's reading / core claim / referee report, and the blog summary).
It shares no code with the CUDA path and is imported only by ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``.  The product
path never routes through it.

Modules:
  model     fp64 decoder layer, target logits, draft-module feature/projection/layers
  spd       stage bounds, autoregressive decode, the pipeline-step simulator with
            streaming verification / rollback / reseed, trace replay, closed-form alpha
  sampling  softmax sampling and speculative rejection sampling
  philox    Philox4x32-10 uniforms

Every function is pinned by a ``-m "not gpu"`` test against something other than
itself (closed forms, library routines, brute force, published known-answer values)
except the draft-aware speedup model (the paper's Eqs. 10-12), whose formulas are not
on the pages: parity unpinned, and not implemented.
"""
from .model import Model, KVCache, rmsnorm, rope, silu, layer_block, argmax_fp32, attend  # noqa: F401
from .spd import (SPDOracle, Replay, ar_decode, stage_bounds, closed_form_alpha,  # noqa: F401
                  replay_decisions, TrackedCache)
from . import philox, sampling  # noqa: F401
