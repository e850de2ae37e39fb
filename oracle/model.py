"""fp64 CPU model math of the oracle: the target decoder and the Pipeline Draft Module.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this package; the
tests, the smoke check and the bench's CPU-baseline leg are its only callers.

The pages leave the decoder architecture to the workload descriptions (dense
pre-norm decoder, RMSNorm, RoPE, GQA, SwiGLU).  The readings taken here:
  * pre-norm block:  h += W_o Attn(RoPE(W_q x), RoPE(W_k x), W_v x),  x = rms(h) * g1
                     h += W_d (silu(W_g y) * (W_u y)),                 y = rms(h) * g2
  * rms(v) = v / sqrt(mean(v^2) + eps), eps = 1e-6;
  * RoPE: rotate-half pairing (i, i + hd/2), angle pos * theta^(-2i/hd), positions from 0;
  * attention: softmax(q k^T / sqrt(hd)) v, query head h reads kv head h // (Hq/Hkv);
  * logits = W_lm (rms(h_L) * g_f); argmax ties go to the lowest token id, decided on
    the logits rounded to fp32 (the precision the CUDA path decides in).
Pipeline Draft Module (speculative pipeline decoding page 2, "What carries the
argument" and "Core claim"; page 2 referee report, comment on section 3.3, Eq. 3):
  * an anchor h^(a) is the residual stream after a target layers (h^(0) = embedding);
  * a row's feature concatenates h^(a) over the anchor set B, with anchors deeper than
    the row's current depth replaced by zeros (in-flight tokens only have the
    checkpoints they have already computed; the newest token only the embedding);
  * f = W_p feature (one bias-free projection), then Ls target-shaped decoder layers
    with their own weights and final norm, then the (tied) target LM head.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

from spd_inputs import ModelDims, to_f64


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE.  x: [M][H][hd], pos: [M] absolute positions."""
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]      # [M][half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


class KVCache:
    """Per-layer K and V rows indexed by absolute position, plus the valid length
    of each layer (the entries past it are stale and never read)."""

    def __init__(self, n_layers: int, max_seq: int, Hkv: int, hd: int):
        self.K = [np.zeros((max_seq, Hkv, hd)) for _ in range(n_layers)]
        self.V = [np.zeros((max_seq, Hkv, hd)) for _ in range(n_layers)]
        self.length = [0] * n_layers


class Layer:
    def __init__(self, w: Dict[str, object]):
        self.wq = to_f64(w["wq"]); self.wk = to_f64(w["wk"]); self.wv = to_f64(w["wv"])
        self.wo = to_f64(w["wo"]); self.wg = to_f64(w["w_gate"]); self.wu = to_f64(w["w_up"])
        self.wd = to_f64(w["w_down"])
        self.g1 = to_f64(w["attn_norm"]); self.g2 = to_f64(w["ffn_norm"])


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """Causal GQA attention: q [M][Hq][hd] at absolute positions pos[M], K/V [S][Hkv][hd]
    for positions 0..S-1; row m sees positions <= pos[m].  softmax(q k^T / sqrt(hd)) v,
    query head h reading kv head h // (Hq / Hkv)."""
    M, Hq, hd = q.shape
    S, Hkv = K.shape[0], K.shape[1]
    group = Hq // Hkv
    scale = 1.0 / np.sqrt(hd)
    mask = np.asarray(pos)[:, None] >= np.arange(S)[None, :]           # [M][S]
    out = np.empty((M, Hq, hd))
    for h in range(Hq):
        kh = K[:, h // group, :]
        vh = V[:, h // group, :]
        sc = (q[:, h, :] @ kh.T) * scale                             # [M][S]
        sc = np.where(mask, sc, -np.inf)
        sc = sc - sc.max(axis=1, keepdims=True)
        p = np.exp(sc)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vh
    return out


def layer_block(dm: ModelDims, W: Layer, H: np.ndarray, pos0: int, cache: KVCache, li: int,
                reads: Optional[list] = None) -> np.ndarray:
    """One decoder layer over M consecutive positions pos0..pos0+M-1.

    H: [M][d] residual stream in.  Writes the rows' K,V at their positions in layer
    ``li`` of ``cache`` and attends causally to cache positions 0..p for row p.
    Returns the residual stream out.  ``reads`` (optional) collects
    (layer, first, last) position ranges read, for schedule checks."""
    M = H.shape[0]
    pos = np.arange(pos0, pos0 + M)
    x = rmsnorm(H, W.g1, dm.rms_eps)
    q = (x @ W.wq.T).reshape(M, dm.Hq, dm.hd)
    k = (x @ W.wk.T).reshape(M, dm.Hkv, dm.hd)
    v = (x @ W.wv.T).reshape(M, dm.Hkv, dm.hd)
    q = rope(q, pos, dm.rope_theta)
    k = rope(k, pos, dm.rope_theta)
    cache.K[li][pos0:pos0 + M] = k
    cache.V[li][pos0:pos0 + M] = v
    cache.length[li] = pos0 + M
    S = pos0 + M
    if reads is not None:
        reads.append((li, 0, S - 1))
    out = attend(q, cache.K[li][:S], cache.V[li][:S], pos)
    H = H + out.reshape(M, dm.Hq * dm.hd) @ W.wo.T
    y = rmsnorm(H, W.g2, dm.rms_eps)
    u = silu(y @ W.wg.T) * (y @ W.wu.T)
    return H + u @ W.wd.T


def argmax_fp32(z: np.ndarray) -> int:
    """Greedy pick: argmax of the logits rounded to fp32, lowest id on ties."""
    return int(np.argmax(z.astype(np.float32)))


class Model:
    """Target decoder + draft module in fp64, built from the stored (bf16/fp32) weights."""

    def __init__(self, dm: ModelDims, target: Dict[str, object], pdm: Optional[Dict[str, object]] = None,
                 anchors: Sequence[int] = ()):
        self.dm = dm
        self.embed = to_f64(target["embed"])
        self.layers = [Layer(target["layers"][l]) for l in range(dm.L)]
        self.gf = to_f64(target["final_norm"])
        self.lm_head = to_f64(target["lm_head"])
        self.anchors = tuple(anchors)
        if pdm is not None:
            self.proj = to_f64(pdm["proj"])
            self.pdm_layers = [Layer(pdm["layers"][l]) for l in range(len(pdm["layers"]))]
            self.pdm_gf = to_f64(pdm["final_norm"])
        else:
            self.pdm_layers = []

    # -- target -------------------------------------------------------------------
    def new_cache(self, max_seq: int) -> KVCache:
        return KVCache(self.dm.L, max_seq, self.dm.Hkv, self.dm.hd)

    def new_pdm_cache(self, max_seq: int) -> KVCache:
        return KVCache(len(self.pdm_layers), max_seq, self.dm.Hkv, self.dm.hd)

    def target_layers(self, H: np.ndarray, pos0: int, cache: KVCache, first: int, last: int,
                      anchor_out: Optional[Dict[int, np.ndarray]] = None, reads: Optional[list] = None) -> np.ndarray:
        """Run target layers first..last-1 on rows at pos0..; record anchors reached."""
        for li in range(first, last):
            H = layer_block(self.dm, self.layers[li], H, pos0, cache, li, reads)
            if anchor_out is not None and (li + 1) in self.anchors:
                anchor_out[li + 1] = H.copy()
        return H

    def logits(self, h: np.ndarray) -> np.ndarray:
        return rmsnorm(h, self.gf, self.dm.rms_eps) @ self.lm_head.T

    # -- draft module -----------------------------------------------------------------
    def feature(self, anchor_vals: Dict[int, np.ndarray], depth: int) -> np.ndarray:
        """Masked concatenation over B: anchors a <= depth present, deeper ones zero."""
        parts = []
        for a in self.anchors:
            parts.append(np.reshape(anchor_vals[a], -1) if a <= depth else np.zeros(self.dm.d))
        return np.concatenate(parts)

    def pdm_block(self, feats: np.ndarray, pos0: int, cache: KVCache) -> np.ndarray:
        """Project the rows' features and run the draft layers over positions pos0...
        Returns the rows' final residual streams."""
        H = feats @ self.proj.T
        for li, W in enumerate(self.pdm_layers):
            H = layer_block(self.dm, W, H, pos0, cache, li)
        return H

    def pdm_logits(self, h: np.ndarray) -> np.ndarray:
        return rmsnorm(h, self.pdm_gf, self.dm.rms_eps) @ self.lm_head.T
