"""Autoregressive decode and the speculative-pipeline-decoding simulator (oracle side).

TEST INFRASTRUCTURE ONLY: the product path never imports this module.

Method (speculative pipeline decoding; page 1 abstract; page 2 "The reading",
"What carries the argument", "Core claim", referee comments on sections 3.3, 3.4 and
4.2 Eq. 9, and section 3.5 on rejection sampling):
  * the L target layers are cut into n stages; stage s holds layers [b_s, b_{s+1}),
    b_s = floor(s L / n) (uniform split), or an explicit non-uniform partition;
  * n in-flight tokens of ONE sequence occupy the stages, the token in stage s sitting
    one position behind the token in stage s-1; one step runs every occupied stage on
    its own token, then shifts all tokens one stage deeper;
  * concurrently, the draft module reads the step's INPUT states (early-start
    schedule) and proposes the token after the newest one; it enters stage 0 (the
    ablated alternative, also simulated: the module runs after the step on its OUTPUT
    states);
  * when a token leaves the last stage its target prediction verifies the draft one
    position later (streaming verification, one check per step); on a mismatch the KV
    cache is truncated after the exiting token, every in-flight token is dropped and
    stage 0 is reseeded with the target's token.
Readings where the pages are silent or garbled:
  * the draft module's rows in a step are: the token that exited in the previous step
    (now complete, with all anchors; its draft-module K,V stay cached from then on)
    followed by the in-flight tokens oldest first; rows are consecutive positions, so
    block-causal attention over "cached prefix + block" is plain causal attention;
  * the verified draft is never counted twice: y0 from the prefill is committed, each
    verification commits exactly one token (the kept draft or the correction), and no
    bonus token exists, so alpha = N / K <= 1 and the draft-free speedup S0 = alpha * n;
  * after a rejection the emptied stages do no work (bubbles exist, contrary to the
    blog page's claim that no stage idles);
  * generation stops as soon as 1 + N reaches max_new (y0 counts), in-flight tokens are
    discarded; no EOS (random weights).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

from . import philox
from .model import KVCache, Model, argmax_fp32
from .sampling import inverse_cdf, keep, probs, residual


def stage_bounds(L: int, n: int, bounds: Optional[Sequence[int]] = None) -> List[int]:
    """Stage s holds layers [b_s, b_{s+1}), s = 0..n-1.

    Uniform split (the pages speak of L/n layers per stage): b_s = floor(s L / n).
    ``bounds`` gives a non-uniform partition instead (page 2, referee report, minor
    comment on Appendix C.1: concrete non-uniform layer assignments, not yet tried in the
    paper): n + 1 integers 0 = b_0 < b_1 < ... < b_n = L, every stage non-empty."""
    if not (1 <= n <= L):
        raise ValueError("need 1 <= n <= L")
    if bounds is None:
        return [(s * L) // n for s in range(n + 1)]
    b = [int(x) for x in bounds]
    if len(b) != n + 1 or b[0] != 0 or b[-1] != L or any(b[i + 1] <= b[i] for i in range(n)):
        raise ValueError("stage bounds must be 0 = b_0 < b_1 < ... < b_n = L")
    return b


def closed_form_alpha(n: int, p: float) -> float:
    """Expected commits per step under forced drafts kept with probability p.

    Renewal argument (derived here, not printed on the pages): after each rejection
    the reseeded token needs n-1 steps before it reaches the last stage; from then on
    every step commits one token until the next rejection, a Geometric(1-p) run, so a
    cycle commits 1/(1-p) tokens in n-1 + 1/(1-p) steps."""
    if p >= 1.0:
        return 1.0
    return 1.0 / (1.0 + (n - 1) * (1.0 - p))


@dataclasses.dataclass
class Replay:
    """Teacher forcing on another implementation's trace.

    For each step t the other side's choices are given; where this oracle's own
    decision is within tolerance of a tie (top-2 logit margin <= tol * |top-1|, or a
    uniform within ``tol_u`` of a CDF boundary / keep-ratio), the other side's choice is
    adopted; elsewhere the two must agree and any disagreement is recorded."""
    steps: Dict[int, dict]
    prefill_y0: Optional[int] = None
    tol: float = 2e-2
    tol_u: float = 1e-4
    mismatches: list = dataclasses.field(default_factory=list)
    adopted: int = 0
    decisions: int = 0
    # the same two counts per kind of decision: "argmax", "sample", "keep"
    adopted_by: dict = dataclasses.field(default_factory=lambda: {"argmax": 0, "sample": 0, "keep": 0})
    decisions_by: dict = dataclasses.field(default_factory=lambda: {"argmax": 0, "sample": 0, "keep": 0})

    def _count(self, kind: str, adopted: bool):
        self.decisions += 1
        self.decisions_by[kind] += 1
        if adopted:
            self.adopted += 1
            self.adopted_by[kind] += 1

    def pick_argmax(self, z: np.ndarray, other: Optional[int], what: str, t: int) -> int:
        mine = argmax_fp32(z)
        if other is None:
            return mine
        if other == mine:
            self._count("argmax", False)
            return mine
        z32 = z.astype(np.float64)
        top = z32[mine]
        if z32[other] >= top - self.tol * abs(top):
            self._count("argmax", True)
            return int(other)
        self._count("argmax", False)
        self.mismatches.append((t, what, mine, int(other), float(top - z32[other])))
        return mine

    def pick_sample(self, w: np.ndarray, u: float, other: Optional[int], what: str, t: int) -> int:
        mine = inverse_cdf(w, u)
        if other is None:
            return mine
        if other == mine:
            self._count("sample", False)
            return mine
        c = np.cumsum(w) / np.sum(w)
        # the other pick owns the interval [c[other-1], c[other]) of the unit line; it is
        # adopted only when u lies within tol_u of that interval (a draw that moved across
        # one boundary because the two sides' cumulative sums differ by rounding)
        if 0 <= other < len(w) and w[other] > 0.0:
            lo = c[other - 1] if other > 0 else 0.0
            if lo - self.tol_u <= u < c[other] + self.tol_u:
                self._count("sample", True)
                return int(other)
        self._count("sample", False)
        self.mismatches.append((t, what, mine, int(other), float(u)))
        return mine

    def pick_keep(self, ratio: float, u1: float, other: Optional[int], t: int) -> bool:
        mine = bool(u1 < ratio)
        if other is None:
            return mine
        if bool(other) == mine:
            self._count("keep", False)
            return mine
        if abs(u1 - ratio) <= self.tol * max(ratio, 1e-30) or abs(u1 - ratio) <= self.tol_u:
            self._count("keep", True)
            return bool(other)
        self._count("keep", False)
        self.mismatches.append((t, "keep", int(mine), int(other), float(u1 - ratio)))
        return mine


class _Tok:
    __slots__ = ("pos", "tok", "H", "anchors", "pD")

    def __init__(self, pos, tok, H, anchors, pD=None):
        self.pos, self.tok, self.H, self.anchors, self.pD = pos, tok, H, anchors, pD


class TrackedCache(KVCache):
    """KVCache that also records which entries hold live data, so the schedule checks
    can assert that every attention read hits a written, not-yet-truncated entry."""

    def __init__(self, *a):
        super().__init__(*a)
        self.live = [np.zeros(self.K[0].shape[0], dtype=bool) for _ in self.K]
        self.bad_reads: list = []


def _check_reads(cache: KVCache, reads: list, t: int):
    if not isinstance(cache, TrackedCache):
        return
    for (li, first, last) in reads:
        if not cache.live[li][first:last + 1].all():
            cache.bad_reads.append((t, li, first, last))


class SPDOracle:
    """Step-by-step simulator of the pipeline step, draft module and verification."""

    def __init__(self, model: Model, n: int, max_seq: int, temperature: float = 0.0, seed: int = 2,
                 forced_p: Optional[float] = None, forced_ref: Optional[Sequence[int]] = None,
                 replay: Optional[Replay] = None, track: bool = False,
                 accept_script: Optional[Sequence[int]] = None, bounds: Optional[Sequence[int]] = None,
                 speculate: str = "input"):
        dm = model.dm
        # schedule checks only: a list of keep decisions consumed one per verification,
        # overriding the token comparison (the committed token is then the draft or the
        # target's token as the decision says)
        self.script = None if accept_script is None else list(accept_script)
        self.m, self.n, self.T, self.seed = model, n, float(temperature), int(seed)
        self.b = stage_bounds(dm.L, n, bounds)
        if speculate not in ("input", "output"):
            raise ValueError("speculate must be 'input' or 'output'")
        # "input": the draft module reads the step's input states, concurrently with the
        # step (the paper's early-start schedule); "output": it runs after the step on its
        # output states (the ablation the referee report lists)
        self.speculate = speculate
        if forced_p is not None and forced_ref is None:
            raise ValueError("forced drafts need the reference stream")
        self.forced_p, self.ref = forced_p, (None if forced_ref is None else np.asarray(forced_ref))
        self.replay = replay
        Cache = TrackedCache if track else KVCache
        self.kv = Cache(dm.L, max_seq, dm.Hkv, dm.hd)
        self.pkv = KVCache(len(model.pdm_layers), max_seq, dm.Hkv, dm.hd)
        self.tokens: List[int] = []
        self.slots: List[Optional[_Tok]] = [None] * n
        self.pending: Optional[_Tok] = None
        self.t = 0
        self.N = 0
        self.K = 0
        self.trace: List[dict] = []
        self.max_inflight_partial = 0

    # ----------------------------------------------------------------------------------
    def _embed_tok(self, pos: int, tok: int, pD=None) -> _Tok:
        e = self.m.embed[tok].copy()
        return _Tok(pos, tok, e[None, :], {0: e.copy()}, pD)

    def _pick_target(self, z: np.ndarray, u_purpose_t: int, what: str, other: Optional[int]) -> int:
        if self.T == 0.0:
            if self.replay is not None:
                return self.replay.pick_argmax(z, other, what, u_purpose_t)
            return argmax_fp32(z)
        w = probs(z, self.T)
        u = philox.uniform(self.seed, u_purpose_t, philox.PURPOSE_TARGET)
        if self.replay is not None:
            return self.replay.pick_sample(w, u, other, what, u_purpose_t)
        return inverse_cdf(w, u)

    def prefill(self, prompt: Sequence[int]) -> int:
        """Whole-prompt pass (all layers), the draft module's cached prefix, then y0."""
        m = self.m
        prompt = [int(x) for x in prompt]
        Sp = len(prompt)
        self.tokens = list(prompt)
        H = m.embed[prompt]
        anchors: Dict[int, np.ndarray] = {0: H.copy()}
        H = m.target_layers(H, 0, self.kv, 0, m.dm.L, anchors)
        if isinstance(self.kv, TrackedCache):
            for lv in self.kv.live:
                lv[:Sp] = True
        if m.pdm_layers:
            feats = np.stack([m.feature({a: anchors[a][i] for a in m.anchors}, m.dm.L) for i in range(Sp)])
            m.pdm_block(feats, 0, self.pkv)
        z = m.logits(H[-1])
        other = None if self.replay is None else self.replay.prefill_y0
        y0 = self._pick_target(z, 0, "y0", other)
        self.tokens.append(y0)
        self.slots = [self._embed_tok(Sp, y0)] + [None] * (self.n - 1)
        self.pending = None
        self.prefill_logits = z
        return y0

    def _draft(self, P: int, zD: np.ndarray, pdm_top: int, rep: Optional[dict]):
        """The token proposed for position P+1 (and its draft distribution at T>0)."""
        dm = self.m.dm
        if self.forced_p is not None:
            c = philox.u24(self.seed, self.t, philox.PURPOSE_COIN)
            r = int(self.ref[P + 1])
            if c < self.forced_p * 16777216.0:
                return r, None
            a = philox.u24(self.seed, self.t, philox.PURPOSE_ALT)
            return (r + 1 + ((a * (dm.V - 1)) >> 24)) % dm.V, None
        if self.T == 0.0:
            return pdm_top, None
        pD = probs(zD, self.T)
        u0 = philox.uniform(self.seed, self.t, philox.PURPOSE_DRAFT)
        other = None if rep is None else rep.get("new_draft_sample")
        if self.replay is not None:
            return self.replay.pick_sample(pD, u0, other, "draft", self.t), pD
        return inverse_cdf(pD, u0), pD

    def _draft_rows(self) -> List[tuple]:
        """(token, depth) rows of the draft module in this step, oldest position first.

        Input-state schedule (before the step's target work): the token that left the
        pipeline in the previous step, at full depth L (its K,V join the module's cache
        for good), then the in-flight tokens from the deepest stage to stage 0 at their
        stages' input depths b_s.  Output-state schedule (after the target work): the
        in-flight tokens at their output depths b_{s+1}; the one leaving the last stage
        is then at depth L and joins the cache."""
        n, b, L = self.n, self.b, self.m.dm.L
        rows = []
        if self.speculate == "input":
            if self.pending is not None:
                rows.append((self.pending, L))
            for s in range(n - 1, -1, -1):
                if self.slots[s] is not None:
                    rows.append((self.slots[s], b[s]))
        else:
            for s in range(n - 1, -1, -1):
                if self.slots[s] is not None:
                    rows.append((self.slots[s], b[s + 1]))
        for i in range(1, len(rows)):
            assert rows[i][0].pos == rows[i - 1][0].pos + 1, "draft-module rows must be consecutive"
        return rows

    def _run_draft_module(self, rows, rep, t):
        """Project the rows' masked anchor features, run the draft layers over their
        positions (causal over the cached prefix and the block), final norm, LM head.
        Returns (logits of the newest row, its argmax under the replay rule)."""
        m = self.m
        feats = np.stack([m.feature(tk.anchors, dep) for (tk, dep) in rows])
        Hp = m.pdm_block(feats, rows[0][0].pos, self.pkv)
        self.last_Hp = Hp
        zD = m.pdm_logits(Hp[-1])
        if self.replay is not None and self.forced_p is None and self.T == 0.0:
            top = self.replay.pick_argmax(zD, None if rep is None else rep.get("pdm_top"), "pdm", t)
        else:
            top = argmax_fp32(zD)
        return zD, top

    def step(self) -> dict:
        m, n, b = self.m, self.n, self.b
        self.t += 1
        t = self.t
        rep = None if self.replay is None else self.replay.steps.get(t)
        newest = self.slots[0]
        P = newest.pos
        pdm_top = -1
        zD = None
        rows: List[tuple] = []
        # ---- input-state schedule: the draft module on the step's input states ------------
        if self.speculate == "input":
            rows = self._draft_rows()
            if m.pdm_layers:
                zD, pdm_top = self._run_draft_module(rows, rep, t)
        # ---- target: each occupied stage runs its own layers on its own token ---------
        for s in range(n):
            tk = self.slots[s]
            if tk is None:
                continue
            reads: list = []
            tk.H = m.target_layers(tk.H, tk.pos, self.kv, b[s], b[s + 1], tk.anchors, reads)
            if isinstance(self.kv, TrackedCache):
                for li in range(b[s], b[s + 1]):
                    self.kv.live[li][tk.pos] = True
                _check_reads(self.kv, reads, t)
        # ---- output-state schedule: the draft module after the step, on its outputs ---------
        if self.speculate == "output":
            rows = self._draft_rows()
            if m.pdm_layers:
                zD, pdm_top = self._run_draft_module(rows, rep, t)
        partial = sum(1 for (tk, dep) in rows if dep < m.dm.L)
        self.max_inflight_partial = max(self.max_inflight_partial, partial)
        self.last_zD = zD
        self.pkv_len = rows[0][0].pos + sum(1 for (tk, dep) in rows if dep == m.dm.L)
        draft_tok, draft_pD = self._draft(P, zD, pdm_top, rep)
        # ---- streaming verification of the draft one position behind the exiting token
        ex = self.slots[n - 1]
        rec = dict(t=t, exit_pos=-1, draft=-1, target=-1, accept=-1, commit=-1,
                   pdm_top=pdm_top, new_draft=int(draft_tok), pdm_logit=(None if zD is None else float(zD[pdm_top])),
                   target_logit=None, pdm_rows=[(tk.pos, dep) for (tk, dep) in rows])
        flushed = False
        if ex is not None:
            q = ex.pos
            zT = m.logits(ex.H[0])
            self.last_zT = zT
            if n >= 2:
                nxt = self.slots[n - 2]
                x, pD = nxt.tok, nxt.pD
            else:
                x, pD = draft_tok, draft_pD
            if self.T == 0.0:
                y = self._pick_target(zT, t, "target", None if rep is None else rep.get("target"))
                ok = (x == y)
                if self.script is not None and self.script:
                    ok = bool(self.script.pop(0))
                rec["target_logit"] = float(zT[y])
            else:
                pT = probs(zT, self.T)
                u1 = philox.uniform(self.seed, t, philox.PURPOSE_ACCEPT)
                ratio = pT[x] / pD[x]
                if self.replay is not None:
                    ok = self.replay.pick_keep(ratio, u1, None if rep is None else rep.get("accept"), t)
                else:
                    ok = bool(u1 < ratio)
                if ok:
                    y = x
                else:
                    u2 = philox.uniform(self.seed, t, philox.PURPOSE_TARGET)
                    w = residual(pT, pD)
                    other = None if rep is None else rep.get("commit")
                    y = (self.replay.pick_sample(w, u2, other, "residual", t) if self.replay is not None
                         else inverse_cdf(w, u2))
            commit = x if ok else y
            self.tokens.append(int(commit))
            self.N += 1
            rec.update(exit_pos=q, draft=int(x), target=int(y), accept=int(ok), commit=int(commit))
            # input-state schedule: the exited token is the draft module's full-depth row of
            # the next step (the output-state schedule took it in this step)
            self.pending = ex if self.speculate == "input" else None
            if not ok:
                flushed = True
                for li in range(m.dm.L):
                    self.kv.length[li] = q + 1
                    if isinstance(self.kv, TrackedCache):
                        self.kv.live[li][q + 1:] = False
                self.slots = [self._embed_tok(q + 1, int(y))] + [None] * (n - 1)
        else:
            self.pending = None
        if not flushed:
            self.slots = [self._embed_tok(P + 1, int(draft_tok), draft_pD)] + self.slots[:n - 1]
        self.K += 1
        rec["len"] = list(self.kv.length)
        rec["N"] = self.N
        self.trace.append(rec)
        return rec

    def fork(self, n: Optional[int] = None, forced_p: Optional[float] = None,
             forced_ref: Optional[Sequence[int]] = None, replay: Optional[Replay] = None,
             bounds: Optional[Sequence[int]] = None, speculate: Optional[str] = None) -> "SPDOracle":
        """A copy of this simulator right after its prefill, before the first step, with its
        own stage count, draft rule and replay record: several runs from one prompt pass.
        The model's weights are shared; caches, token list and stage slots are copied."""
        if self.t != 0 or self.K != 0 or not self.tokens:
            raise ValueError("fork only between prefill and the first step")
        if isinstance(self.kv, TrackedCache):
            raise ValueError("fork does not carry schedule tracking")
        if forced_p is not None and forced_ref is None:
            raise ValueError("forced drafts need the reference stream")
        o = SPDOracle.__new__(SPDOracle)
        o.__dict__.update(self.__dict__)
        o.n = self.n if n is None else n
        o.b = stage_bounds(self.m.dm.L, o.n, bounds)
        if speculate is not None:
            o.speculate = speculate
        o.forced_p, o.ref = forced_p, (None if forced_ref is None else np.asarray(forced_ref))
        o.replay = replay
        for name in ("kv", "pkv"):
            src = getattr(self, name)
            c = KVCache.__new__(KVCache)
            c.K = [k.copy() for k in src.K]
            c.V = [v.copy() for v in src.V]
            c.length = list(src.length)
            setattr(o, name, c)
        o.tokens = list(self.tokens)
        y0 = self.slots[0]
        o.slots = [_Tok(y0.pos, y0.tok, y0.H.copy(), {a: h.copy() for a, h in y0.anchors.items()}, y0.pD)]
        o.slots += [None] * (o.n - 1)
        o.pending = None
        o.trace = []
        return o

    def run(self, prompt: Sequence[int], max_new: int, max_steps: Optional[int] = None) -> List[int]:
        self.prefill(prompt)
        Sp = len(prompt)
        while 1 + self.N < max_new and (max_steps is None or self.K < max_steps):
            self.step()
        return self.tokens[Sp:]

    def stats(self) -> dict:
        alpha = self.N / self.K if self.K else 0.0
        runs, cur = [], 0
        for r in self.trace:
            if r["accept"] == 1:
                cur += 1
            elif r["accept"] == 0:
                runs.append(cur)
                cur = 0
        return dict(N=self.N, K=self.K, alpha=alpha, S0=alpha * self.n,
                    rejects=sum(1 for r in self.trace if r["accept"] == 0),
                    accepts=sum(1 for r in self.trace if r["accept"] == 1),
                    mean_kept_run=(float(np.mean(runs)) if runs else float(cur)))


def ar_decode(model: Model, prompt: Sequence[int], max_new: int, max_seq: int,
              temperature: float = 0.0, seed: int = 2) -> List[int]:
    """Plain autoregressive decode: prefill, then one full pass per token.
    At T > 0 token k (k = 0 for the prefill's) is drawn with uniform (k, purpose 2)."""
    dm = model.dm
    kv = model.new_cache(max_seq)
    prompt = [int(x) for x in prompt]
    H = model.target_layers(model.embed[prompt], 0, kv, 0, dm.L)
    out: List[int] = []
    h = H[-1]
    pos = len(prompt)
    for k in range(max_new):
        z = model.logits(h)
        if temperature == 0.0:
            y = argmax_fp32(z)
        else:
            y = inverse_cdf(probs(z, temperature), philox.uniform(seed, k, philox.PURPOSE_TARGET))
        out.append(y)
        if k + 1 == max_new:
            break
        h = model.target_layers(model.embed[[y]], pos, kv, 0, dm.L)[0]
        pos += 1
    return out


def replay_decisions(n: int, L: int, prompt_len: int, steps: Sequence[dict],
                     bounds: Optional[Sequence[int]] = None) -> List[dict]:
    """Pure state machine of the staircase (no arithmetic): given, per step, the token the
    draft module proposed (``new_draft``) and, when a token exits, the target's choice
    (``target``) and the keep decision (``accept``; derived as draft == target when
    absent), recompute exit positions, commits and the per-layer KV lengths.  Used to
    check another implementation's trace at any size."""
    b = stage_bounds(L, n, bounds)
    slots: List[Optional[list]] = [[prompt_len, None]] + [None] * (n - 1)   # [pos, tok]
    length = [prompt_len] * L
    out = []
    for st in steps:
        for s in range(n):
            if slots[s] is not None:
                for li in range(b[s], b[s + 1]):
                    length[li] = slots[s][0] + 1
        ex = slots[n - 1]
        rec = dict(exit_pos=-1, accept=-1, commit=-1)
        P = slots[0][0]
        flushed = False
        if ex is not None:
            q = ex[0]
            x = slots[n - 2][1] if n >= 2 else st["new_draft"]
            y = st["target"]
            ok = st["accept"] if st.get("accept", -1) in (0, 1) else int(x == y)
            commit = x if ok else y
            rec.update(exit_pos=q, accept=int(ok), commit=int(commit), draft=int(x))
            if not ok:
                flushed = True
                length = [q + 1] * L
                slots = [[q + 1, commit]] + [None] * (n - 1)
        if not flushed:
            slots = [[P + 1, st["new_draft"]]] + slots[:n - 1]
        rec["len"] = list(length)
        out.append(rec)
    return out
