"""Shared helpers of the GPU parity tests: build a seeded case, run it through the C ABI
and replay the oracle on the GPU's trace."""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

import spd_inputs as si
from oracle import Model, Replay, SPDOracle, ar_decode


@dataclasses.dataclass
class Case:
    dm: si.ModelDims
    n: int
    anchors: tuple
    Ls: int
    prompt_len: int
    max_new: int
    norms: str = "ones"
    seed: int = 0
    prompt_seed: int = 1

    def build(self):
        tg = si.make_target(self.dm, self.seed, norms=self.norms)
        pd = si.make_pdm(self.dm, self.Ls, len(self.anchors), self.seed, norms=self.norms) if self.Ls else None
        prompt = si.make_prompt(self.dm.V, self.prompt_len, self.prompt_seed)
        return tg, pd, prompt

    @property
    def max_seq(self):
        return self.prompt_len + self.max_new + self.n + 8

    @property
    def tol(self):
        return 1e-4 if self.dm.dtype == "fp32" else 2e-2

    @property
    def tol_draft(self):
        """Draft-module logits: at bf16 its GEMMs take bf16 activations (tensor-core operands)
        on top of full-depth target states that already carry the target's rounding, so the
        bound is twice the target's; at fp32 the module computes in fp32 like the target."""
        return self.tol if self.dm.dtype == "fp32" else 2 * self.tol


_cache = {}


def materialise(case: Case):
    """(target, pdm, prompt, oracle model, device target, device pdm), cached per case."""
    key = repr(case)
    if key not in _cache:
        from speculative_pipeline_decoding_spd_gb300.engine import to_device
        tg, pd, prompt = case.build()
        m = Model(case.dm, tg, pd, case.anchors)
        _cache.clear()
        _cache[key] = (tg, pd, prompt, m, to_device(tg), to_device(pd) if pd is not None else None)
    return _cache[key]


def engine(case: Case, n: Optional[int] = None, **kw):
    from speculative_pipeline_decoding_spd_gb300.engine import Engine
    tg, pd, prompt, m, dtg, dpd = materialise(case)
    return Engine(case.dm, dtg, dpd, n or case.n, case.anchors, max_seq=case.max_seq, max_new=case.max_new, **kw)


def run_gpu(case: Case, n: Optional[int] = None, **kw):
    tg, pd, prompt, m, dtg, dpd = materialise(case)
    e = engine(case, n=n, **kw)
    out, cnt, st = e.generate(torch.from_numpy(prompt).cuda())
    toks = out[:cnt].cpu().tolist()
    tr = e.trace()
    pf = e.read(9, (case.dm.V,))
    stats = e.stats()
    e.close()
    return toks, tr, stats, pf


def replay_oracle(case: Case, gpu_trace, gpu_tokens, n: Optional[int] = None, tol: Optional[float] = None,
                  forced_p=None, forced_ref=None, temperature=0.0, seed=2, max_steps=None):
    tg, pd, prompt, m, _, _ = materialise(case)
    rep = Replay(steps={}, prefill_y0=gpu_tokens[0], tol=tol if tol is not None else case.tol)
    for r in gpu_trace:
        d = {"pdm_top": r["pdm_top"]}
        if r["exit_pos"] >= 0:
            d["target"] = r["target"]
            d["accept"] = r["accept"]
            d["commit"] = r["commit"]
        if temperature > 0:
            d["new_draft_sample"] = r["new_draft"]
        rep.steps[r["t"]] = d
    o = SPDOracle(m, n or case.n, case.max_seq, temperature=temperature, seed=seed, forced_p=forced_p,
                  forced_ref=forced_ref, replay=rep)
    o.prefill(prompt)
    steps = len(gpu_trace) if max_steps is None else min(max_steps, len(gpu_trace))
    for _ in range(steps):
        o.step()
    return o, rep


def compare(case: Case, gpu_trace, o: SPDOracle, rep: Replay, check_logits=True):
    """Exact agreement of the integer trace; logits within the case tolerance."""
    assert rep.mismatches == [], rep.mismatches[:5]
    worst, where, worst_d, where_d = 0.0, None, 0.0, None
    for g, r in zip(gpu_trace, o.trace):
        for k in ("exit_pos", "accept", "commit", "draft", "new_draft", "len", "N"):
            assert g[k] == r[k], (k, g["t"], g[k], r[k])
        if check_logits and r["target_logit"] is not None:
            err = abs(g["target_logit"] - r["target_logit"]) / max(1.0, abs(r["target_logit"]))
            if err > worst:
                worst, where = err, (g["t"], g["target_logit"], r["target_logit"])
        if check_logits and r["pdm_logit"] is not None and r["pdm_top"] == g["pdm_top"]:
            err = abs(g["pdm_logit"] - r["pdm_logit"]) / max(1.0, abs(r["pdm_logit"]))
            if err > worst_d:
                worst_d, where_d = err, (g["t"], g["pdm_logit"], r["pdm_logit"])
    assert worst <= case.tol, ("target logit", worst, where)
    assert worst_d <= case.tol_draft, ("draft logit", worst_d, where_d)
    return max(worst, worst_d)


def ar_reference(case: Case):
    tg, pd, prompt, m, _, _ = materialise(case)
    return ar_decode(m, prompt, case.max_new, case.max_seq)
