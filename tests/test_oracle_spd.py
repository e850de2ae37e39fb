"""Pins of the oracle's pipeline-step simulator against what the method fixes:
losslessness (SPD greedy == AR greedy), exact commit counts at p in {0, 1}, the
closed-form commit rate, the draft-free speedup identity S0 = alpha * n, and a
brute-force comparison of the staircase / rollback schedule with an independent
closed-form event model."""
import itertools

import numpy as np
import pytest

import spd_inputs as si
from oracle import (Model, SPDOracle, ar_decode, closed_form_alpha, replay_decisions,
                    stage_bounds)

MICRO = si.ModelDims(L=6, d=16, Hq=2, Hkv=1, hd=8, F=32, V=24, dtype="fp32")


def micro_model(L=6, anchors=None, seed=0, V=24):
    dm = si.shrink(MICRO, L=L, V=V)
    anchors = anchors or tuple(sorted({0, L // 2, L}))
    tg = si.make_target(dm, seed, norms="perturbed")
    pd = si.make_pdm(dm, 1, len(anchors), seed, norms="perturbed")
    return Model(dm, tg, pd, anchors)


def test_stage_bounds_values():
    # the 4B workload's stages have 4-5 layers and its anchors 9, 18, 27 sit on stage edges
    assert stage_bounds(36, 8) == [0, 4, 9, 13, 18, 22, 27, 31, 36]
    assert stage_bounds(28, 4) == [0, 7, 14, 21, 28]
    assert stage_bounds(4, 2) == [0, 2, 4]
    for L in range(1, 40):
        for n in range(1, L + 1):
            b = stage_bounds(L, n)
            sizes = np.diff(b)
            assert b[0] == 0 and b[-1] == L and sizes.min() >= 1 and sizes.max() - sizes.min() <= 1


@pytest.mark.parametrize("n", [1, 2, 3, 4, 6])
def test_lossless_greedy_with_draft_module(n):
    m = micro_model()
    prompt = si.make_prompt(m.dm.V, 5, seed=7)
    ar = ar_decode(m, prompt, 20, 64)
    o = SPDOracle(m, n, 64, track=True)
    assert o.run(prompt, 20) == ar
    assert o.kv.bad_reads == []
    assert o.max_inflight_partial <= n          # at most n rows with partial-depth features


@pytest.mark.parametrize("n,p", [(2, 0.0), (3, 0.3), (4, 0.7), (5, 1.0), (1, 0.5)])
def test_lossless_forced_drafts(n, p):
    m = micro_model(seed=1)
    prompt = si.make_prompt(m.dm.V, 4, seed=3)
    ar = ar_decode(m, prompt, 24, 80)
    ref = list(prompt) + ar + [0] * (n + 2)
    o = SPDOracle(m, n, 80, forced_p=p, forced_ref=ref, seed=11, track=True)
    assert o.run(prompt, 24) == ar
    assert o.kv.bad_reads == []


@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_exact_counts_at_p0_and_p1(n):
    m = micro_model(seed=2)
    prompt = si.make_prompt(m.dm.V, 3, seed=4)
    ar = ar_decode(m, prompt, 16, 80)
    ref = list(prompt) + ar + [0] * (n + 2)
    for p, count in ((1.0, lambda K: max(0, K - n + 1)), (0.0, lambda K: K // n)):
        o = SPDOracle(m, n, 80, forced_p=p, forced_ref=ref)
        o.run(prompt, 16)
        for rec, K in zip(o.trace, itertools.count(1)):
            assert rec["N"] == count(K), (p, K)


def test_speedup_identity_from_trace():
    """S0 = alpha * n with alpha = commits / steps counted from the per-step trace."""
    m = micro_model(seed=3)
    prompt = si.make_prompt(m.dm.V, 4, seed=5)
    ar = ar_decode(m, prompt, 30, 90)
    o = SPDOracle(m, 3, 90, forced_p=0.6, forced_ref=list(prompt) + ar + [0] * 5, seed=5)
    o.run(prompt, 30)
    commits = sum(1 for r in o.trace if r["commit"] >= 0)
    st = o.stats()
    assert commits == st["N"] == 29 and len(o.trace) == st["K"]
    assert st["S0"] == pytest.approx(3 * commits / len(o.trace))
    assert 1.0 / 3 - 1e-12 <= st["alpha"] <= 1.0


@pytest.mark.parametrize("n,p", [(2, 0.6), (4, 0.5), (4, 0.8), (6, 0.3)])
def test_alpha_matches_closed_form_statistically(n, p):
    m = micro_model(seed=4)
    prompt = si.make_prompt(m.dm.V, 2, seed=6)
    total = 1200
    ar = ar_decode(m, prompt, total, total + 16)
    o = SPDOracle(m, n, total + 16, forced_p=p, forced_ref=list(prompt) + ar + [0] * (n + 2), seed=99)
    assert o.run(prompt, total) == ar
    a = closed_form_alpha(n, p)
    # renewal-reward standard error (delta method), 4 sigma
    G = 1.0 / (1.0 - p)
    cycles = o.N * (1.0 - p)
    sd = (n - 1) / ((n - 1) + G) ** 2 * np.sqrt(p / (1 - p) ** 2 / cycles)
    assert abs(o.stats()["alpha"] - a) < 4 * sd + 2.0 * n / o.K, (o.stats()["alpha"], a)


def test_closed_form_alpha_values():
    expect = {(2, .6): 0.714, (4, .5): 0.400, (4, .8): 0.625, (8, .3): 0.169, (8, .6): 0.263,
              (8, .9): 0.588, (8, .7): 0.323, (16, .7): 0.182}
    for (n, p), v in expect.items():
        assert closed_form_alpha(n, p) == pytest.approx(v, abs=6e-4)


# ---- schedule brute force against an independent event model ---------------------------

def event_model(n, L, prompt_len, bits, steps):
    """Closed-form staircase: an epoch starts with a committed seed at position p0 that
    enters stage 0 at step t0; its k-th successor enters at t0 + k and leaves the last
    stage at t0 + k + n - 1, where it verifies position p0 + k + 1.  A failed check at step
    t starts a new epoch (seed at that position, entering at t + 1).  The KV length of a
    layer in stage s after step t is p0 + max(0, t - t0 - s + 1)."""
    b = stage_bounds(L, n)
    stage_of = [s for s in range(n) for _ in range(b[s], b[s + 1])]
    p0, t0 = prompt_len, 1
    bits = list(bits)
    out = []
    for t in range(1, steps + 1):
        rec = {}
        k_exit = t - (n - 1) - t0
        new_epoch = None
        if k_exit >= 0:
            q = p0 + k_exit
            ok = bits.pop(0) if bits else 1
            rec.update(exit_pos=q, accept=ok)
            if not ok:
                new_epoch = (q + 1, t + 1)
        else:
            rec.update(exit_pos=-1, accept=-1)
        rec["len"] = [p0 + max(0, t - t0 - stage_of[li] + 1) for li in range(L)]
        if new_epoch:
            p0, t0 = new_epoch
            rec["len"] = [p0] * L
        out.append(rec)
    return out


def scripted_steps(n, L, Sp, bits, steps):
    """Feed ``replay_decisions`` drafts/targets that realise the keep pattern ``bits``."""
    recs = []
    it = iter(bits)
    ev = event_model(n, L, Sp, bits, steps)
    for e in ev:
        st = {"new_draft": 1, "target": 1}
        if e["exit_pos"] >= 0:
            st["accept"] = e["accept"]
            st["target"] = 1 if e["accept"] else 2
        recs.append(st)
    return recs, ev


@pytest.mark.parametrize("n,L", [(1, 3), (2, 3), (2, 5), (3, 3), (3, 6)])
def test_state_machine_matches_event_model_bruteforce(n, L):
    Sp = 4
    for length in range(0, 9):
        for bits in itertools.product([0, 1], repeat=length):
            steps = 3 * n + 2 * length
            st, ev = scripted_steps(n, L, Sp, bits, steps)
            got = replay_decisions(n, L, Sp, st)
            for g, e in zip(got, ev):
                assert g["exit_pos"] == e["exit_pos"] and g["len"] == e["len"], (bits, g, e)
                if e["exit_pos"] >= 0:
                    assert g["accept"] == e["accept"]


@pytest.mark.parametrize("n,L", [(2, 3), (3, 5), (3, 6)])
def test_simulator_schedule_bruteforce(n, L):
    """The full simulator, driven by a keep pattern, follows the event model: exit
    positions and per-layer KV lengths after every step; no attention read touches an
    unwritten or truncated KV entry; at most n partial-depth rows."""
    m = micro_model(L=L, seed=5)
    prompt = [1, 2, 3, 4]
    for bits in itertools.product([0, 1], repeat=6):
        steps = 3 * n + 12
        o = SPDOracle(m, n, 64, track=True, accept_script=bits + (1,) * 64)
        o.prefill(prompt)
        for _ in range(steps):
            o.step()
        ev = event_model(n, L, len(prompt), bits, steps)
        for r, e in zip(o.trace, ev):
            assert r["exit_pos"] == e["exit_pos"] and r["len"] == e["len"], (bits, r["t"])
        assert o.kv.bad_reads == []
        assert o.max_inflight_partial <= n


def test_replay_decisions_reproduces_simulator_trace():
    m = micro_model(seed=6)
    prompt = si.make_prompt(m.dm.V, 5, seed=8)
    ar = ar_decode(m, prompt, 30, 90)
    o = SPDOracle(m, 3, 90, forced_p=0.5, forced_ref=list(prompt) + ar + [0] * 5, seed=3)
    o.run(prompt, 30)
    got = replay_decisions(3, m.dm.L, len(prompt), o.trace)
    for g, r in zip(got, o.trace):
        assert (g["exit_pos"], g["accept"], g["commit"], g["len"]) == (r["exit_pos"], r["accept"], r["commit"], r["len"])


def test_fork_after_prefill_equals_fresh_runs():
    """A fork taken right after one prefill runs exactly like a fresh simulator that did its
    own prefill: for other stage counts and draft rules, and without disturbing the parent."""
    m = micro_model(seed=2)
    prompt = si.make_prompt(m.dm.V, 6, seed=4)
    ar = ar_decode(m, prompt, 18, 72)
    ref = list(prompt) + ar + [0] * 8
    base = SPDOracle(m, 3, 72, seed=9)
    base.prefill(prompt)
    for n, p in [(3, None), (2, 0.5), (4, 0.8), (1, 0.3)]:
        kw = dict(forced_p=p, forced_ref=ref) if p is not None else {}
        f = base.fork(n=n, **kw)
        fresh = SPDOracle(m, n, 72, seed=9, **kw)
        fresh.prefill(prompt)
        for _ in range(14):
            assert f.step() == fresh.step()
        assert f.tokens == fresh.tokens
    # the parent is untouched and still runs like a fresh one
    fresh = SPDOracle(m, 3, 72, seed=9)
    fresh.prefill(prompt)
    for _ in range(10):
        assert base.step() == fresh.step()
    with pytest.raises(ValueError):
        base.fork()
