"""Seeded synthetic inputs shared by the CUDA path's tests/bench and by the oracle.

This module holds no arithmetic of the method: it only defines the workload shapes
and draws random-init weights and prompt ids.  Both sides receive the same values
(the CUDA path as device tensors, the oracle as fp64 numpy arrays).

Recipe (the pages give no weights or datasets; random init stands in for the
trained Qwen3.5 target and draft module, uniform-random prompt ids stand in for
the MT-Bench / GSM8K / HumanEval prompts the paper evaluates on):
  * every matrix ~ N(0, 0.02^2), drawn per tensor from a torch CPU generator whose
    seed is derived from (weight_seed, tensor name), then rounded to the storage
    dtype (bf16 round-to-nearest-even, or kept fp32);
  * RMSNorm gains are 1 (``norms="ones"``), or 1 + N(0, 0.1^2) when a test wants
    the gains to matter (``norms="perturbed"``);
  * prompt ids ~ uniform{0..V-1} from a generator seeded with ``prompt_seed``.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class ModelDims:
    L: int          # decoder layers
    d: int          # model width
    Hq: int         # query heads
    Hkv: int        # key/value heads
    hd: int         # head dim
    F: int          # SwiGLU hidden width
    V: int          # vocabulary
    rope_theta: float = 1.0e4
    rms_eps: float = 1.0e-6
    dtype: str = "bf16"   # weight storage: "bf16" or "fp32"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: ModelDims
    n: int                      # pipeline stages
    anchors: tuple              # anchor depths B (0 = embedding)
    Ls: int                     # draft-module layers
    prompt_len: int
    max_new: int
    temperature: float = 0.0
    forced_p: tuple = ()        # forced-draft acceptance probabilities exercised


# The five workloads.  Anchor set {0,9,18,27,36} of the 8B shape is the reading of
# "5 evenly spaced anchors" over 36 layers; the T=1 workload uses the 4B shape and
# n=8 (its text says "as config 2", which has neither).
TINY = Workload("tiny-fp32", ModelDims(L=4, d=256, Hq=4, Hkv=4, hd=64, F=1024, V=1024, dtype="fp32"),
                n=2, anchors=(0, 2, 4), Ls=1, prompt_len=16, max_new=64, forced_p=(0.6,))
SHAPE_06B = Workload("0.6b-shape", ModelDims(L=28, d=1024, Hq=16, Hkv=8, hd=128, F=3072, V=151936),
                     n=4, anchors=(0, 7, 14, 21, 28), Ls=1, prompt_len=128, max_new=256, forced_p=(0.5, 0.8))
SHAPE_4B = Workload("4b-shape", ModelDims(L=36, d=2560, Hq=32, Hkv=8, hd=128, F=9728, V=151936),
                    n=8, anchors=(0, 9, 18, 27, 35), Ls=4, prompt_len=512, max_new=512, forced_p=(0.3, 0.6, 0.9))
SHAPE_8B = Workload("8b-shape", ModelDims(L=36, d=4096, Hq=32, Hkv=8, hd=128, F=12288, V=151936),
                    n=8, anchors=(0, 9, 18, 27, 36), Ls=2, prompt_len=4096, max_new=512, forced_p=(0.7,))
SHAPE_4B_T1 = Workload("4b-shape-t1", SHAPE_4B.dims, n=8, anchors=SHAPE_4B.anchors, Ls=4,
                       prompt_len=256, max_new=1024, temperature=1.0)

WORKLOADS = [TINY, SHAPE_06B, SHAPE_4B, SHAPE_8B, SHAPE_4B_T1]


def _tensor_seed(base: int, name: str) -> int:
    h = hashlib.sha256(f"{base}:{name}".encode()).hexdigest()
    return int(h[:15], 16)


_DEVICE = "cpu"


def _normal(shape, base: int, name: str, std: float) -> torch.Tensor:
    g = torch.Generator(device=_DEVICE).manual_seed(_tensor_seed(base, name))
    return torch.randn(*shape, generator=g, dtype=torch.float32, device=_DEVICE) * std


def _store(t: torch.Tensor, dtype: str) -> torch.Tensor:
    return t.to(torch.bfloat16) if dtype == "bf16" else t.contiguous()


def _norm_gain(d: int, base: int, name: str, norms: str) -> torch.Tensor:
    if norms == "ones":
        return torch.ones(d, dtype=torch.float32, device=_DEVICE)
    return 1.0 + _normal((d,), base, name, 0.1)


LAYER_MATS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def layer_shapes(dm: ModelDims) -> Dict[str, tuple]:
    return {
        "wq": (dm.Hq * dm.hd, dm.d), "wk": (dm.Hkv * dm.hd, dm.d), "wv": (dm.Hkv * dm.hd, dm.d),
        "wo": (dm.d, dm.Hq * dm.hd), "w_gate": (dm.F, dm.d), "w_up": (dm.F, dm.d), "w_down": (dm.d, dm.F),
    }


def make_layer(dm: ModelDims, base: int, prefix: str, norms: str = "ones") -> Dict[str, torch.Tensor]:
    """One decoder layer's tensors (matrices in dm.dtype, norm gains fp32)."""
    out = {}
    for name, shape in layer_shapes(dm).items():
        out[name] = _store(_normal(shape, base, f"{prefix}.{name}", 0.02), dm.dtype)
    out["attn_norm"] = _norm_gain(dm.d, base, f"{prefix}.attn_norm", norms)
    out["ffn_norm"] = _norm_gain(dm.d, base, f"{prefix}.ffn_norm", norms)
    return out


def make_target(dm: ModelDims, seed: int = 0, norms: str = "ones",
                layers: Optional[Sequence[int]] = None) -> Dict[str, object]:
    """Target model: embed [V][d], layers, final_norm [d], lm_head [V][d].

    ``layers`` restricts generation to a subset (for sampled checks); each tensor's
    values depend only on (seed, its name), never on which others were drawn."""
    idx = range(dm.L) if layers is None else layers
    return {
        "embed": _store(_normal((dm.V, dm.d), seed, "embed", 0.02), dm.dtype),
        "layers": {l: make_layer(dm, seed, f"layer{l}", norms) for l in idx},
        "final_norm": _norm_gain(dm.d, seed, "final_norm", norms),
        "lm_head": _store(_normal((dm.V, dm.d), seed, "lm_head", 0.02), dm.dtype),
    }


def make_pdm(dm: ModelDims, Ls: int, n_anchors: int, seed: int = 0, norms: str = "ones") -> Dict[str, object]:
    """Draft module: proj [d][|B|*d], Ls target-shaped layers, its own final norm.
    Its LM head is tied to the target's (no tensor here)."""
    return {
        "proj": _store(_normal((dm.d, n_anchors * dm.d), seed, "pdm.proj", 0.02), dm.dtype),
        "layers": {l: make_layer(dm, seed, f"pdm.layer{l}", norms) for l in range(Ls)},
        "final_norm": _norm_gain(dm.d, seed, "pdm.final_norm", norms),
    }


class on_device:
    """Draw the tensors directly on a device with that device's generator (same seeds and
    distribution, different values from the CPU draw).  For throughput runs whose
    weights the oracle never needs."""

    def __init__(self, device: str):
        self.device = device

    def __enter__(self):
        global _DEVICE
        self.prev, _DEVICE = _DEVICE, self.device

    def __exit__(self, *a):
        global _DEVICE
        _DEVICE = self.prev


def make_prompt(V: int, length: int, seed: int = 1) -> np.ndarray:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, V, (length,), generator=g, dtype=torch.int64).numpy().astype(np.int32)


def to_f64(t) -> np.ndarray:
    """Exact widening of a stored tensor (bf16 or fp32) to fp64 numpy."""
    return t.to(torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, dtype=np.float64)


def shrink(dm: ModelDims, **kw) -> ModelDims:
    return dataclasses.replace(dm, **kw)


def workload(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


__all__ = ["ModelDims", "Workload", "WORKLOADS", "TINY", "SHAPE_06B", "SHAPE_4B", "SHAPE_8B",
           "SHAPE_4B_T1", "make_target", "make_pdm", "make_layer", "make_prompt", "to_f64",
           "layer_shapes", "LAYER_MATS", "shrink", "workload", "on_device"]
