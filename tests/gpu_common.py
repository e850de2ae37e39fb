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
        """One bound for hidden states and logits, target and draft module alike: rel 1e-4 for
        fp32 weights, rel 2e-2 for bf16 weights."""
        return 1e-4 if self.dm.dtype == "fp32" else 2e-2

    @property
    def kv_dtype(self):
        return np.float32   # the library's K/V caches hold fp32 rows for every weight type


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


def replay_record(gpu_trace, y0, tol, temperature=0.0):
    rep = Replay(steps={}, prefill_y0=y0, tol=tol)
    for r in gpu_trace:
        d = {"pdm_top": r["pdm_top"]}
        if r["exit_pos"] >= 0:
            d["target"] = r["target"]
            d["accept"] = r["accept"]
            d["commit"] = r["commit"]
        if temperature > 0:
            d["new_draft_sample"] = r["new_draft"]
        rep.steps[r["t"]] = d
    return rep


def replay_oracle(case: Case, gpu_trace, gpu_tokens, n: Optional[int] = None, tol: Optional[float] = None,
                  forced_p=None, forced_ref=None, temperature=0.0, seed=2, max_steps=None, bounds=None,
                  speculate="input"):
    tg, pd, prompt, m, _, _ = materialise(case)
    rep = replay_record(gpu_trace, gpu_tokens[0], tol if tol is not None else case.tol, temperature)
    o = SPDOracle(m, n or case.n, case.max_seq, temperature=temperature, seed=seed, forced_p=forced_p,
                  forced_ref=forced_ref, replay=rep, bounds=bounds, speculate=speculate)
    o.prefill(prompt)
    steps = len(gpu_trace) if max_steps is None else min(max_steps, len(gpu_trace))
    for _ in range(steps):
        o.step()
    return o, rep


# the replay rule may adopt the GPU's choice at near-ties.  Argmax and keep decisions are near a
# tie rarely: at most 5% of them (2 absolute); the full-size workloads adopt 0-1 of 158-1275.
# A draw from a flat distribution over the whole vocabulary (T = 1, random weights: typical
# p ~ 1 / V) moves across an index boundary whenever the two sides' cumulative sums differ by
# more than u's distance to it, so sampled picks may differ by a neighbouring index more often;
# each is still checked against tol_u: at most 10% (the T = 1 workload adopts 7 of 284).
ADOPT_SHARE = {"argmax": 0.05, "keep": 0.05, "sample": 0.10}


def compare(case: Case, gpu_trace, o: SPDOracle, rep: Replay, check_logits=True):
    """Exact agreement of the integer trace; the chosen tokens' logits within the case
    tolerance; the replay rule used only at a few near-ties."""
    assert rep.mismatches == [], rep.mismatches[:5]
    print(f"replay: {rep.adopted} of {rep.decisions} decisions adopted from the GPU at near-ties "
          f"(by kind {rep.adopted_by} of {rep.decisions_by})")
    for kind, share in ADOPT_SHARE.items():
        assert rep.adopted_by[kind] <= max(2, share * rep.decisions_by[kind]), (kind, rep.adopted_by, rep.decisions_by)
    worst, where = 0.0, None
    for g, r in zip(gpu_trace, o.trace):
        for k in ("exit_pos", "accept", "commit", "draft", "new_draft", "len", "N"):
            assert g[k] == r[k], (k, g["t"], g[k], r[k])
        if not check_logits:
            continue
        pairs = []
        if r["target_logit"] is not None:
            pairs.append(("target", g["target_logit"], r["target_logit"]))
        if r["pdm_logit"] is not None and r["pdm_top"] == g["pdm_top"]:
            pairs.append(("draft", g["pdm_logit"], r["pdm_logit"]))
        for what, gv, rv in pairs:
            err = abs(gv - rv) / max(1.0, abs(rv))
            if err > worst:
                worst, where = err, (what, g["t"], gv, rv)
    assert worst <= case.tol, ("chosen logit", worst, where)
    return worst


def vec_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / max(1, max |ref|): error against the vector's scale (hidden states,
    anchors, K/V rows)."""
    return float(np.max(np.abs(got - ref)) / max(1.0, float(np.max(np.abs(ref)))))


def elem_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max_i |got_i - ref_i| / max(1, |ref_i|): every entry on its own scale (logits)."""
    return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref))))


def step_and_compare_vectors(case: Case, e, o: SPDOracle, steps: int, tol: Optional[float] = None):
    """Run the engine and the oracle (already prefilled, replaying nothing) one step at a
    time and compare, after every step:
      * the target logits of the exiting token and the draft module's newest-row logits,
        entry by entry (SPD_BUF_LOGITS against the oracle's verification and draft logits);
      * the draft block's final residual rows (SPD_BUF_PDM_RESIDUAL);
      * every in-flight token's residual stream and the anchor states it has reached
        (SPD_BUF_RESIDUAL / SPD_BUF_ANCHORS, slots found by position);
      * the K and V rows that the step wrote: every layer each stage ran, at its token's
        position, and the draft layers' rows of the whole draft block.
    The oracle follows the GPU's choices only at near-ties (replay rule).  Returns the
    worst error of each kind."""
    from speculative_pipeline_decoding_spd_gb300 import binding as B
    tol = case.tol if tol is None else tol
    dm, n = case.dm, o.n
    kvw = dm.Hkv * dm.hd
    ksz = np.dtype(case.kv_dtype).itemsize
    worst = dict(logits_t=0.0, logits_d=0.0, pdm_rows=0.0, residual=0.0, anchors=0.0, kv=0.0, pdm_kv=0.0)
    for k in range(steps):
        # stages and positions before the step: the K,V rows it writes
        runs = [(s, tk.pos) for s, tk in enumerate(o.slots) if tk is not None]
        e.step(1)
        tr = e.trace()
        g = tr[-1]
        o.replay.steps[g["t"]] = {"pdm_top": g["pdm_top"], **({"target": g["target"], "accept": g["accept"],
                                                               "commit": g["commit"]} if g["exit_pos"] >= 0 else {}),
                                  **({"new_draft_sample": g["new_draft"]} if o.T > 0 else {})}
        r = o.step()
        for key in ("exit_pos", "accept", "commit", "new_draft", "len"):
            assert g[key] == r[key], (key, k, g[key], r[key])
        lg = e.read(B.SPD_BUF_LOGITS, (2, dm.V))
        if r["exit_pos"] >= 0:
            worst["logits_t"] = max(worst["logits_t"], elem_err(lg[0], o.last_zT))
        if o.last_zD is not None:
            worst["logits_d"] = max(worst["logits_d"], elem_err(lg[1], o.last_zD))
            R = o.last_Hp.shape[0]
            xp = e.read(B.SPD_BUF_PDM_RESIDUAL, (n + 1, dm.d))[:R]
            worst["pdm_rows"] = max(worst["pdm_rows"], vec_err(xp, o.last_Hp))
            pos0 = r["pdm_rows"][0][0]
            for li in range(len(o.m.pdm_layers)):
                for which, ref in ((B.SPD_BUF_PDM_KCACHE, o.pkv.K[li]), (B.SPD_BUF_PDM_VCACHE, o.pkv.V[li])):
                    got = e.read(which, (R, kvw), dtype=case.kv_dtype, index=li, offset=pos0 * kvw * ksz)
                    worst["pdm_kv"] = max(worst["pdm_kv"], vec_err(got.astype(np.float64),
                                                                   ref[pos0:pos0 + R].reshape(R, kvw)))
        for s, pos in runs:
            for li in range(o.b[s], o.b[s + 1]):
                for which, ref in ((B.SPD_BUF_KCACHE, o.kv.K[li]), (B.SPD_BUF_VCACHE, o.kv.V[li])):
                    got = e.read(which, (kvw,), dtype=case.kv_dtype, index=li, offset=pos * kvw * ksz)
                    worst["kv"] = max(worst["kv"], vec_err(got.astype(np.float64), ref[pos].reshape(kvw)))
        X = e.read(B.SPD_BUF_RESIDUAL, (n + 1, dm.d))
        A = e.read(B.SPD_BUF_ANCHORS, (n + 1, len(case.anchors), dm.d))
        slots = e.read(B.SPD_BUF_SLOTS, (3, n + 1), dtype=np.int32)
        for s, tk in enumerate(o.slots):
            if tk is None:
                continue
            idx = [i for i in range(n + 1) if slots[0][i] and slots[1][i] == tk.pos]
            assert idx, (k, tk.pos)
            worst["residual"] = max(worst["residual"], vec_err(X[idx[0]], tk.H[0]))
            for ai, a in enumerate(case.anchors):
                if a in tk.anchors:
                    worst["anchors"] = max(worst["anchors"], vec_err(A[idx[0], ai], tk.anchors[a]))
    print("worst errors:", {k: f"{v:.2e}" for k, v in worst.items()})
    for key, v in worst.items():
        assert v <= tol, (key, v, worst)
    assert o.replay.mismatches == [], o.replay.mismatches[:5]
    return worst


def ar_reference(case: Case):
    tg, pd, prompt, m, _, _ = materialise(case)
    return ar_decode(m, prompt, case.max_new, case.max_seq)
