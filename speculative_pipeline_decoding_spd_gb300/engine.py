"""Convenience wrapper around the C ABI: PyTorch owns the device memory (weights,
workspace, prompt and output buffers) and the stream; every step of the computation
runs in libspd_gb300.so.  Marshalling only."""
from __future__ import annotations

import ctypes as C
from typing import Dict, Optional, Sequence

import numpy as np
import torch

from . import binding as B

_LAYER_KEYS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "attn_norm", "ffn_norm")


def to_device(tensors, device="cuda"):
    """Recursively move a weight dict (from spd_inputs) to the device, keeping dtypes."""
    if isinstance(tensors, dict):
        return {k: to_device(v, device) for k, v in tensors.items()}
    if isinstance(tensors, torch.Tensor):
        return tensors.to(device).contiguous()
    return tensors


def _layer_struct(w) -> B.spd_layer_weights:
    return B.spd_layer_weights(*[w[k].data_ptr() for k in _LAYER_KEYS])


class Engine:
    """One handle: a target, an optional draft module, n stages, anchors and a run config."""

    def __init__(self, dims, target: Dict, pdm: Optional[Dict], n: int, anchors: Sequence[int], *,
                 max_seq: int, max_new: int, temperature: float = 0.0, seed: int = 2, force_p: float = -1.0,
                 forced_ref: Optional[torch.Tensor] = None, graph: bool = True, timing: bool = False,
                 stream: Optional[torch.cuda.Stream] = None, workspace_fill: Optional[int] = None,
                 bounds: Optional[Sequence[int]] = None, speculate: str = "input"):
        self.dims = dims
        self.n = n
        self.max_new = max_new
        self.L = dims.L
        self.V = dims.V
        self._keep = [target, pdm, forced_ref]
        dt = B.SPD_BF16 if dims.dtype == "bf16" else B.SPD_F32
        self.cd = B.spd_dims(dims.L, dims.d, dims.Hq, dims.Hkv, dims.hd, dims.F, dims.V, dims.rope_theta,
                             dims.rms_eps, dt)
        self._tl = (B.spd_layer_weights * dims.L)(*[_layer_struct(target["layers"][l]) for l in range(dims.L)])
        self.tw = B.spd_target_weights(target["embed"].data_ptr(), self._tl, target["final_norm"].data_ptr(),
                                       target["lm_head"].data_ptr())
        if pdm is not None:
            Ls = len(pdm["layers"])
            self._pl = (B.spd_layer_weights * max(1, Ls))(*[_layer_struct(pdm["layers"][l]) for l in range(Ls)])
            lm = pdm.get("lm_head", target["lm_head"])
            self.pw = B.spd_pdm_weights(Ls, pdm["proj"].data_ptr(), self._pl, pdm["final_norm"].data_ptr(),
                                        lm.data_ptr())
        else:
            self.pw = B.spd_pdm_weights(0, None, None, None, None)
        a = (C.c_int32 * B.SPD_MAX_ANCHORS)(*list(anchors))
        self.cfg = B.spd_config(n, len(anchors), a, float(temperature), int(seed), int(max_seq), int(max_new),
                                float(force_p), forced_ref.data_ptr() if forced_ref is not None else None,
                                int(forced_ref.numel()) if forced_ref is not None else 0, int(graph), int(timing))
        if bounds is not None:
            for i, v in enumerate(bounds):
                self.cfg.stage_bounds[i] = int(v)
        self.cfg.speculate = {"input": B.SPD_SPEC_INPUT, "output": B.SPD_SPEC_OUTPUT}[speculate]
        self.ws_bytes = B.spd_workspace_bytes(self.cd, self.pw, self.cfg)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        if workspace_fill is not None:   # tests: the library must not rely on zeroed memory
            self.workspace.fill_(workspace_fill)
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.h = B.spd_create(self.cd, self.tw, self.pw, self.cfg, self.workspace.data_ptr(), self.ws_bytes,
                              self.stream.cuda_stream)

    # ----------------------------------------------------------------------------------
    def prefill(self, prompt: torch.Tensor):
        assert prompt.is_cuda and prompt.dtype == torch.int32
        self._prompt = prompt
        B.spd_prefill(self.h, prompt.data_ptr(), prompt.numel())

    def step(self, k: int = 1, sync: bool = True):
        return B.spd_step(self.h, k, want_count=sync)

    def generate(self, prompt, on_host: bool = False):
        """Prefill + decode until max_new tokens.  ``prompt``: cuda int32 tensor (device
        buffers) or a numpy int32 array / pinned CPU tensor (host buffers)."""
        if on_host:
            p = torch.as_tensor(np.asarray(prompt, dtype=np.int32)).contiguous()
            out = torch.empty(self.max_new, dtype=torch.int32)
            n, st = B.spd_generate(self.h, p.data_ptr(), p.numel(), 1, out.data_ptr())
            return out[:n].numpy().tolist(), st
        out = torch.empty(self.max_new, dtype=torch.int32, device="cuda")
        self._prompt = prompt
        n, st = B.spd_generate(self.h, prompt.data_ptr(), prompt.numel(), 0, out.data_ptr())
        return out, n, st

    def tokens(self):
        buf = np.zeros(self.max_new, dtype=np.int32)
        cnt = B.spd_get_tokens(self.h, buf.ctypes.data, self.max_new)
        return buf[:min(cnt, self.max_new)].tolist()

    def trace(self):
        cap = self.n * self.max_new + 2 * self.n + 8
        lens = np.zeros((cap, self.L), dtype=np.int32)
        recs, cnt = B.spd_get_trace(self.h, cap, lens.ctypes.data)
        out = []
        for i in range(min(cnt, cap)):
            r = recs[i]
            out.append(dict(t=r.t, exit_pos=r.exit_pos, draft=r.draft, target=r.target, accept=r.accept,
                            commit=r.commit, pdm_top=r.pdm_top, new_draft=r.new_draft, N=r.n_committed,
                            n_active=r.n_active, target_logit=r.target_logit, pdm_logit=r.pdm_logit,
                            len=lens[i].tolist()))
        return out

    def stats(self) -> dict:
        s = B.spd_get_stats(self.h)
        return {k: getattr(s, k) for k, _ in B.spd_stats._fields_}

    def read(self, which: int, shape, dtype=np.float32, index: int = 0, offset: int = 0) -> np.ndarray:
        out = np.zeros(shape, dtype=dtype)
        B.spd_read_buffer(self.h, which, index, offset, out.ctypes.data, out.nbytes)
        return out

    def kernel_timing(self):
        return B.spd_kernel_timing(self.h)

    def reset(self):
        B.spd_reset(self.h)

    def close(self):
        if getattr(self, "h", None) is not None:
            B.spd_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
