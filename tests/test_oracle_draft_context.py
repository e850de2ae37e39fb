"""Pins of the oracle's draft-module context and of its replay checker.

The draft module (page 2, "What carries the argument" and "Core claim"; referee comment
on section 3.3, Eq. 3) reads, per token, the target's hidden states at the anchor depths
that token has already reached: verified tokens at full depth, in-flight tokens at their
stage's depth (a depth staircase), the newest one at its embedding only.  The oracle
computes this incrementally: each token's draft-module K,V are cached once, when it has
left the pipeline, and the in-flight rows are recomputed every step.  Losslessness holds
for ANY draft, so the pins of the token stream cannot see a mistake here; these can:

* caching invariance: after every step, the newest row's draft logits equal a from-scratch
  recomputation that runs the whole token sequence through a fresh target pass (anchors
  of every position), builds every position's masked feature at the depth the schedule
  gives it, and runs the draft layers over all positions as one causal block with a fresh
  cache, then the module's own final norm and the head, written out here;
* the row set of every step, brute-forced over keep/reject patterns against a closed-form
  event model of the staircase;
* the replay checker adopts the other side's choice only at near-ties and records every
  other disagreement.

Both schedules are covered: input states (the draft module runs beside the step) and
output states (it runs after the step), and non-uniform stage partitions."""
import itertools

import numpy as np
import pytest

import spd_inputs as si
from oracle import Model, Replay, SPDOracle, ar_decode, layer_block, rmsnorm, stage_bounds

MICRO = si.ModelDims(L=5, d=16, Hq=2, Hkv=1, hd=8, F=32, V=40, dtype="fp32")


def micro(L, anchors, Ls=2, seed=0, V=40):
    dm = si.shrink(MICRO, L=L, V=V)
    tg = si.make_target(dm, seed, norms="perturbed")
    pd = si.make_pdm(dm, Ls, len(anchors), seed, norms="perturbed")
    m = Model(dm, tg, pd, anchors)
    # the module's final norm must differ from the target's for the pin to see a swap
    assert not np.allclose(m.pdm_gf, m.gf)
    return m


def sequence(o: SPDOracle) -> tuple:
    """(token ids of positions 0..P, {position: stage} of the in-flight tokens) before a step."""
    inflight = {tk.pos: s for s, tk in enumerate(o.slots) if tk is not None}
    P = max(inflight)
    seq = list(o.tokens[: P + 1]) + [None] * (P + 1 - min(len(o.tokens), P + 1))
    for s, tk in enumerate(o.slots):
        if tk is None:
            continue
        if tk.pos < len(o.tokens):
            assert o.tokens[tk.pos] == tk.tok          # committed and still in flight
        seq[tk.pos] = tk.tok
    assert all(x is not None for x in seq)
    return seq, inflight


def from_scratch_draft_logits(m: Model, seq, depth_of) -> np.ndarray:
    """Draft logits of the last position, recomputed with no cache reuse at all."""
    dm = m.dm
    P = len(seq) - 1
    kv = m.new_cache(P + 1)
    anchors = {0: m.embed[seq].copy()}
    m.target_layers(m.embed[seq], 0, kv, 0, dm.L, anchors)
    feats = []
    for p in range(P + 1):
        dep = depth_of(p)
        feats.append(np.concatenate([anchors[a][p] if a <= dep else np.zeros(dm.d) for a in m.anchors]))
    H = np.stack(feats) @ m.proj.T
    pkv = m.new_pdm_cache(P + 1)
    for li, W in enumerate(m.pdm_layers):
        H = layer_block(dm, W, H, 0, pkv, li)
    return rmsnorm(H[-1], m.pdm_gf, dm.rms_eps) @ m.lm_head.T


def expected_depths(o: SPDOracle, inflight, mode):
    """Depth of every position in this step's draft block, per the schedule."""
    b, L = o.b, o.m.dm.L
    if mode == "input":
        return lambda p: b[inflight[p]] if p in inflight else L
    return lambda p: b[inflight[p] + 1] if p in inflight else L


CASES = [
    # (L, anchors, n, bounds, mode kwargs)
    (4, (0, 1, 2, 3, 4), 2, None, {}),                       # an anchor at every depth
    (5, (0, 1, 2, 3, 4, 5), 3, None, dict(forced_p=0.5)),
    (5, (0, 2, 5), 3, (0, 1, 4, 5), {}),                     # non-uniform stages
    (6, (0, 1, 2, 3, 4, 5, 6), 4, (0, 3, 4, 5, 6), dict(forced_p=0.6)),
    (4, (0, 1, 2, 3, 4), 1, None, {}),
    (5, (0, 1, 3, 4, 5), 2, None, dict(temperature=1.0)),
]


@pytest.mark.parametrize("mode", ["input", "output"])
@pytest.mark.parametrize("L,anchors,n,bounds,kw", CASES)
def test_incremental_draft_module_equals_from_scratch(mode, L, anchors, n, bounds, kw):
    m = micro(L, anchors, seed=L + n)
    if kw.get("temperature"):
        m.lm_head = m.lm_head * 20.0        # sharper laws: rejections happen
    prompt = si.make_prompt(m.dm.V, 4, seed=n)
    steps = 26
    extra = {}
    if "forced_p" in kw:
        ar = ar_decode(m, prompt, steps + 2, 64)
        extra = dict(forced_p=kw["forced_p"], forced_ref=list(prompt) + ar + [0] * (n + 4))
    o = SPDOracle(m, n, 64, seed=7, bounds=bounds, speculate=mode, temperature=kw.get("temperature", 0.0), **extra)
    o.prefill(prompt)
    worst = 0.0
    rejects = 0
    for _ in range(steps):
        seq, inflight = sequence(o)
        dep = expected_depths(o, inflight, mode)
        rec = o.step()
        ref = from_scratch_draft_logits(m, seq, dep)
        err = np.max(np.abs(o.last_zD - ref)) / max(1.0, np.max(np.abs(ref)))
        worst = max(worst, err)
        rejects += rec["accept"] == 0
    assert worst < 1e-10, worst
    if n > 1:
        assert rejects > 0                     # rollbacks were exercised


def event_rows(n, L, b, prompt_len, bits, steps, mode):
    """Closed-form draft rows per step: an epoch's k-th token (position p0 + k) enters
    stage 0 at step t0 + k, so at step t it sits in stage t - t0 - k; the token at stage
    n - 1 leaves at the end of the step.  A rejected check at step t starts the next epoch
    at the exiting position + 1, entering at t + 1.  Input schedule: rows are the previous
    step's exit (depth L) then the in-flight tokens at b_stage; output schedule: the
    in-flight tokens at b_{stage+1}."""
    p0, t0 = prompt_len, 1
    bits = list(bits)
    prev_exit = None
    out = []
    for t in range(1, steps + 1):
        inflight = [(p0 + k, t - t0 - k) for k in range(max(0, t - t0 - (n - 1)), t - t0 + 1)]
        if mode == "input":
            rows = ([(prev_exit, L)] if prev_exit is not None else []) + [(p, b[s]) for p, s in inflight]
        else:
            rows = [(p, b[s + 1]) for p, s in inflight]
        out.append(rows)
        k_exit = t - (n - 1) - t0
        prev_exit = None
        if k_exit >= 0:
            q = p0 + k_exit
            prev_exit = q
            ok = bits.pop(0) if bits else 1
            if not ok:
                p0, t0 = q + 1, t + 1
    return out


@pytest.mark.parametrize("mode", ["input", "output"])
@pytest.mark.parametrize("n,L,bounds", [(1, 3, None), (2, 3, None), (3, 5, None), (3, 5, (0, 3, 4, 5)), (2, 4, (0, 1, 4))])
def test_draft_rows_match_event_model_bruteforce(mode, n, L, bounds):
    """Every keep/reject pattern of length <= 7: the rows of every step are exactly the
    previous exit at full depth (input schedule) and the in-flight tokens at the depth
    the schedule gives their stage, at consecutive positions; at most n rows have
    partial-depth features (Eq. 3 as the referee restates it)."""
    m = micro(L, tuple(range(L + 1)), Ls=1, seed=3)
    b = stage_bounds(L, n, bounds)
    prompt = [1, 2, 3]
    for length in range(0, 8):
        for bits in itertools.product([0, 1], repeat=length):
            steps = 2 * n + length + 3
            o = SPDOracle(m, n, 64, accept_script=bits + (1,) * 64, bounds=bounds, speculate=mode)
            o.prefill(prompt)
            for _ in range(steps):
                o.step()
            ev = event_rows(n, L, b, len(prompt), bits, steps, mode)
            for r, e in zip(o.trace, ev):
                assert r["pdm_rows"] == e, (bits, r["t"], r["pdm_rows"], e)
            assert o.max_inflight_partial <= n


def test_output_schedule_is_lossless_and_differs_from_input():
    """Both schedules commit exactly the greedy stream (any draft is lossless); their draft
    modules see different features, so their draft logits differ."""
    m = micro(5, (0, 2, 5), seed=11)
    prompt = si.make_prompt(m.dm.V, 4, seed=2)
    ar = ar_decode(m, prompt, 24, 64)
    tops = {}
    for mode in ("input", "output"):
        o = SPDOracle(m, 3, 64, speculate=mode, track=True)
        assert o.run(prompt, 24) == ar
        assert o.kv.bad_reads == []
        tops[mode] = np.array([r["pdm_logit"] for r in o.trace])
    assert np.max(np.abs(tops["input"] - tops["output"])) > 1e-3


def test_non_uniform_stages_lossless_and_validated():
    m = micro(6, (0, 3, 6), seed=12)
    prompt = si.make_prompt(m.dm.V, 4, seed=5)
    ar = ar_decode(m, prompt, 20, 64)
    for bounds in [(0, 1, 6), (0, 4, 5, 6), (0, 1, 2, 3, 4, 5, 6)]:
        o = SPDOracle(m, len(bounds) - 1, 64, bounds=bounds, track=True)
        assert o.run(prompt, 20) == ar
        assert o.kv.bad_reads == []
    for bad in [(0, 3, 3, 6), (1, 3, 6), (0, 3, 5), (0, 7)]:
        with pytest.raises(ValueError):
            stage_bounds(6, len(bad) - 1, bad)


# ---- the replay checker ------------------------------------------------------------------

def test_replay_argmax_adopts_only_near_ties():
    z = np.zeros(10)
    z[3], z[7], z[5] = 5.0, 4.95, 2.0          # 3 wins; 7 within 2e-2 * 5 = 0.1 of it; 5 far
    rep = Replay(steps={}, tol=2e-2)
    assert rep.pick_argmax(z, 3, "t", 1) == 3 and rep.adopted == 0 and rep.mismatches == []
    assert rep.pick_argmax(z, 7, "t", 2) == 7 and rep.adopted == 1 and rep.mismatches == []
    assert rep.pick_argmax(z, 5, "t", 3) == 3 and rep.adopted == 1
    assert rep.mismatches == [(3, "t", 3, 5, 3.0)]
    z[7] = 4.85                                 # now 0.15 below the top: outside the tolerance
    assert rep.pick_argmax(z, 7, "t", 4) == 3 and len(rep.mismatches) == 2
    assert rep.decisions == 4
    assert rep.decisions_by == {"argmax": 4, "sample": 0, "keep": 0}
    assert rep.adopted_by == {"argmax": 1, "sample": 0, "keep": 0}
    # no other side: the oracle's own pick, not counted as a decision
    assert rep.pick_argmax(z, None, "t", 5) == 3 and rep.decisions == 4


def test_replay_sample_adopts_only_the_neighbour_across_a_boundary():
    w = np.array([0.1, 0.2, 0.3, 0.4])          # cumulative 0.1, 0.3, 0.6, 1.0
    rep = Replay(steps={}, tol_u=1e-4)
    assert rep.pick_sample(w, 0.45, 2, "s", 1) == 2 and rep.adopted == 0
    # u in the middle of 2's interval: any other pick is a mismatch
    assert rep.pick_sample(w, 0.45, 3, "s", 2) == 2
    assert rep.pick_sample(w, 0.45, 0, "s", 3) == 2
    assert len(rep.mismatches) == 2 and rep.adopted == 0
    # u just below the 2|3 boundary: 3 (the neighbour across it) is adopted ...
    assert rep.pick_sample(w, 0.6 - 5e-5, 3, "s", 4) == 3 and rep.adopted == 1
    # ... and just above it, 2 is
    assert rep.pick_sample(w, 0.6 + 5e-5, 2, "s", 5) == 2 and rep.adopted == 2
    # but not a far pick, and not the neighbour on the other side
    assert rep.pick_sample(w, 0.6 - 5e-5, 0, "s", 6) == 2
    assert rep.pick_sample(w, 0.6 - 5e-5, 1, "s", 7) == 2
    # an index with zero weight is never adopted, nor one outside the vocabulary
    w0 = np.array([0.3, 0.0, 0.7])
    assert rep.pick_sample(w0, 0.3 - 5e-5, 1, "s", 8) == 0
    assert rep.pick_sample(w0, 0.3 - 5e-5, 9, "s", 9) == 0
    assert len(rep.mismatches) == 6 and rep.adopted == 2
    assert rep.adopted_by["sample"] == 2 and rep.decisions_by["sample"] == 9


def test_replay_keep_adopts_only_near_the_ratio():
    rep = Replay(steps={}, tol=2e-2, tol_u=1e-4)
    assert rep.pick_keep(0.5, 0.2, 1, 1) is True
    assert rep.pick_keep(0.5, 0.2, 0, 2) is True and len(rep.mismatches) == 1
    assert rep.pick_keep(0.5, 0.8, 1, 3) is False and len(rep.mismatches) == 2
    assert rep.pick_keep(0.5, 0.5 - 5e-3, 0, 4) is False and rep.adopted == 1    # |u1 - r| <= tol r
    assert rep.pick_keep(0.5, 0.5 + 5e-3, 1, 5) is True and rep.adopted == 2
    assert rep.pick_keep(1e-6, 1e-6 + 5e-5, 1, 6) is True and rep.adopted == 3   # |u1 - r| <= tol_u
    assert rep.pick_keep(0.5, 0.5 + 2e-2, 1, 7) is False and len(rep.mismatches) == 3


def test_replayed_simulation_records_a_planted_wrong_choice():
    """End to end: replaying a run's own trace adopts nothing; the same trace with one
    target choice changed to a token far below the top is recorded as a mismatch."""
    m = micro(4, (0, 2, 4), seed=4, V=40)
    m.lm_head = m.lm_head * 30.0                # clear margins
    prompt = si.make_prompt(m.dm.V, 4, seed=9)
    o = SPDOracle(m, 2, 64)
    o.run(prompt, 14)
    steps = {r["t"]: {"pdm_top": r["pdm_top"], **({"target": r["target"]} if r["exit_pos"] >= 0 else {})}
             for r in o.trace}
    rep = Replay(steps=steps, prefill_y0=o.tokens[4])
    o2 = SPDOracle(m, 2, 64, replay=rep)
    o2.prefill(prompt)
    for _ in range(len(o.trace)):
        o2.step()
    assert rep.mismatches == [] and rep.adopted == 0 and rep.decisions > 10
    t = next(r["t"] for r in o.trace if r["exit_pos"] >= 0)
    bad = dict(steps)
    bad[t] = dict(bad[t], target=(bad[t]["target"] + 1) % m.dm.V)   # logits x 30: far below the top
    rep2 = Replay(steps=bad, prefill_y0=o.tokens[4])
    o3 = SPDOracle(m, 2, 64, replay=rep2)
    o3.prefill(prompt)
    for _ in range(len(o.trace)):
        o3.step()
    assert len(rep2.mismatches) >= 1 and rep2.mismatches[0][0] == t and rep2.mismatches[0][1] == "target"
