"""Parity at the five workloads' full model sizes (0.6B, 4B and 8B shapes, bf16).

The fp64 oracle runs on the host cores and replays the GPU's trace (the replay rule follows
the GPU only at near-ties).  Every workload starts from its own full prompt:
  * config 2 (0.6B): whole 256-token generations, draft-module greedy and forced p = 0.5, 0.8;
  * config 3 (4B): 600 steps at forced p = 0.6 and prefixes of the other modes (greedy
    drafting, p = 0.3 and 0.9);
  * config 5 (4B, T = 1): 256 steps of rejection sampling, dozens of residual resamples;
  * config 4 (8B): the 4096-token prompt through the oracle's prefill, then 16 steps at
    n = 8 and at n = 16; and the whole 512-token generation on the GPU at both n against
    the library's one-stage decode (a property that holds at any size).
On top of the traces, the first steps of configs 2 to 5 compare vectors: logits entry by
entry, the draft block's rows, residual streams, anchors and the K/V rows written.

With SPD_LONG_PARITY=1 config 3's forced p = 0.6 and greedy runs go to their 512th token
(about 2000 and 4100 steps), and config 5 to its 1024th.  The oracle needs about 0.35 s a step
at the 4B shape on 16 host cores, so those are opt-in.

Forced drafts follow the oracle's own greedy stream, so no oracle input comes from the GPU.
Each workload is built once: weights drawn on the host from the seeded generators and
copied to the GPU, one oracle prefill forked for every run of that workload."""
import gc
import os

import numpy as np
import pytest
import torch

import spd_inputs as si
from gpu_common import Case, compare, materialise, replay_record, run_gpu, step_and_compare_vectors
from oracle import Replay, SPDOracle, ar_decode

pytestmark = pytest.mark.gpu

LONG = os.environ.get("SPD_LONG_PARITY", "0") == "1"


def case_of(wl: si.Workload, **over) -> Case:
    kw = dict(n=wl.n, anchors=wl.anchors, Ls=wl.Ls, prompt_len=wl.prompt_len, max_new=wl.max_new)
    kw.update(over)
    return Case(wl.dims, **kw)


def gpu_steps(case: Case, steps, n=None, **kw):
    """Prefill + `steps` pipeline steps (None: until max_new tokens) on the GPU;
    (trace, committed tokens)."""
    from speculative_pipeline_decoding_spd_gb300.engine import Engine
    tg, pd, prompt, m, dtg, dpd = materialise(case)
    e = Engine(case.dm, dtg, dpd, n or case.n, case.anchors, max_seq=case.max_seq, max_new=case.max_new, **kw)
    if steps is None:
        out, cnt, _ = e.generate(torch.from_numpy(prompt).cuda())
    else:
        e.prefill(torch.from_numpy(prompt).cuda())
        e.step(steps)
    tr = e.trace()
    toks = e.tokens()
    e.close()
    return tr, toks


def replay(base: SPDOracle, case: Case, tr, y0: int, n=None, forced_p=None, forced_ref=None, temperature=0.0):
    """Fork the prefilled oracle and replay the GPU trace step by step."""
    rep = replay_record(tr, y0, case.tol, temperature)
    o = base.fork(n=n, forced_p=forced_p, forced_ref=forced_ref, replay=rep)
    for _ in range(len(tr)):
        o.step()
    return o, rep


def oracle_base(case: Case, temperature=0.0, seed=2, y0=None):
    tg, pd, prompt, m, _, _ = materialise(case)
    rep = None if y0 is None else Replay(steps={}, prefill_y0=y0, tol=case.tol)
    o = SPDOracle(m, case.n, case.max_seq, temperature=temperature, seed=seed, replay=rep)
    o.prefill(prompt)
    return o


def forced_ref(case: Case, new_tokens: int):
    """prompt + the oracle's greedy continuation (new_tokens of it), zero-padded to the
    furthest position a run of this case can read."""
    tg, pd, prompt, m, _, _ = materialise(case)
    ar = ar_decode(m, prompt, new_tokens, case.max_seq)
    ref = np.zeros(case.prompt_len + case.max_new + max(case.n, 16) + 8, dtype=np.int32)
    ref[: case.prompt_len] = prompt
    ref[case.prompt_len: case.prompt_len + len(ar)] = ar
    return ref, ar


def forced_ref_from(base: SPDOracle, case: Case, new_tokens: int):
    """The same as forced_ref, from an already prefilled oracle: one stage (n = 1) commits
    the greedy stream one token per step (losslessness), with no second prefill."""
    f = base.fork(n=1)
    for _ in range(new_tokens - 1):
        f.step()
    ar = f.tokens[case.prompt_len:]
    ref = np.zeros(case.prompt_len + case.max_new + max(case.n, 16) + 8, dtype=np.int32)
    ref[: case.prompt_len] = f.tokens[: case.prompt_len]
    ref[case.prompt_len: case.prompt_len + len(ar)] = ar
    return ref


def vectors(case: Case, base: SPDOracle, steps: int, n=None, p=None, ref=None, temperature=0.0):
    """Step-by-step vector comparison of the first `steps` steps from the workload's prompt."""
    from speculative_pipeline_decoding_spd_gb300.engine import Engine
    tg, pd, prompt, m, dtg, dpd = materialise(case)
    kw = {} if p is None else dict(force_p=p, forced_ref=torch.from_numpy(ref).cuda())
    e = Engine(case.dm, dtg, dpd, n or case.n, case.anchors, max_seq=case.max_seq, max_new=case.max_new, seed=2,
               graph=False, temperature=temperature, **kw)
    e.prefill(torch.from_numpy(prompt).cuda())
    rep = Replay(steps={}, prefill_y0=e.tokens()[0], tol=case.tol)
    o = base.fork(n=n, forced_p=p, forced_ref=ref, replay=rep)
    worst = step_and_compare_vectors(case, e, o, steps)
    e.close()
    return worst


def release():
    materialise.__globals__["_cache"].clear()
    gc.collect()
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------------
def test_config2_06b_whole_generation():
    """0.6B shape, n = 4, Ls = 1, prompt 128, 256 new tokens: the draft module's greedy drafts
    and forced drafts at p = 0.5 and 0.8, each run to the end and replayed in full; vectors
    over the first 8 steps."""
    wl = si.SHAPE_06B
    case = case_of(wl)
    ref, _ = forced_ref(case, case.max_new)
    base = None
    for p in (None,) + wl.forced_p:
        kw = {} if p is None else dict(force_p=p, forced_ref=torch.from_numpy(ref).cuda(), seed=2)
        toks, tr, st, pf = run_gpu(case, **kw)
        if base is None:
            base = oracle_base(case, y0=toks[0])
            z = base.prefill_logits
            assert np.max(np.abs(pf - z) / np.maximum(1.0, np.abs(z))) <= case.tol
        o, rep = replay(base, case, tr, toks[0], forced_p=p, forced_ref=None if p is None else ref)
        compare(case, tr, o, rep)
        assert o.tokens[case.prompt_len:] == toks
    vectors(case, base, 8, p=0.5, ref=ref)
    release()


def test_config3_4b_all_modes():
    """4B shape, n = 8, Ls = 4, prompt 512: forced p = 0.6, greedy drafting and p = 0.3 / 0.9
    replayed over prefixes (p = 0.6 and greedy to the 512th token with SPD_LONG_PARITY=1);
    vectors over the first 8 steps."""
    wl = si.SHAPE_4B
    case = case_of(wl)
    ref, _ = forced_ref(case, case.max_new)
    base = None
    runs = [(0.6, None if LONG else 600), (None, None if LONG else 300), (0.3, 200), (0.9, 200)]
    for p, steps in runs:
        kw = {} if p is None else dict(force_p=p, forced_ref=torch.from_numpy(ref).cuda(), seed=2)
        tr, toks = gpu_steps(case, steps, **kw)
        if base is None:
            base = oracle_base(case, y0=toks[0])
        o, rep = replay(base, case, tr, toks[0], forced_p=p, forced_ref=None if p is None else ref)
        compare(case, tr, o, rep)
        assert o.tokens[case.prompt_len: case.prompt_len + len(toks)] == toks
        if steps is None:
            assert len(toks) == case.max_new
        print(f"config 3 p={p}: {len(tr)} steps, {len(toks)} tokens, alpha {o.stats()['alpha']:.3f}")
    vectors(case, base, 8, p=0.6, ref=ref)
    release()


def test_config5_4b_sampling():
    """4B shape at T = 1, n = 8, prompt 256: 256 steps (the whole 1024 tokens with
    SPD_LONG_PARITY=1) of sampled drafts verified by rejection sampling with a residual
    resample, replayed against the oracle on the same Philox uniforms; vectors over the
    first 8 steps."""
    wl = si.SHAPE_4B_T1
    case = case_of(wl)
    tr, toks = gpu_steps(case, None if LONG else 256, temperature=1.0, seed=2)
    base = oracle_base(case, temperature=1.0, seed=2, y0=toks[0])
    o, rep = replay(base, case, tr, toks[0], temperature=1.0)
    compare(case, tr, o, rep)
    assert o.tokens[case.prompt_len: case.prompt_len + len(toks)] == toks
    rejects = sum(1 for r in tr if r["accept"] == 0)
    print(f"config 5: {len(tr)} steps, {len(toks)} tokens, {rejects} residual resamples")
    assert rejects >= 24                                  # the residual path ran many times
    vectors(case, base, 8, temperature=1.0)
    release()


def test_config4_8b_full_prompt_replay_and_whole_generation():
    """8B shape, Ls = 2, forced p = 0.7, 4096-token prompt.  The oracle prefills the whole
    prompt; 16 steps at n = 8 and at n = 16 (17 draft rows: two 16-row mma tiles) are
    replayed against it, and vectors are compared over the first 6 steps at n = 8.  Then
    the whole 512-token generation at both n commits exactly the tokens of the library's
    one-stage decode."""
    from speculative_pipeline_decoding_spd_gb300.engine import Engine
    wl = si.SHAPE_8B
    full = case_of(wl)
    steps = 16
    tg, pd, prompt, m, dtg, dpd = materialise(full)
    e = Engine(full.dm, dtg, dpd, full.n, full.anchors, max_seq=full.max_seq, max_new=full.max_new)
    e.prefill(torch.from_numpy(prompt).cuda())
    y0 = e.tokens()[0]
    e.close()
    base = oracle_base(full, y0=y0)            # the 4096-token prefill, once
    ref = forced_ref_from(base, full, steps + 16 + 4)
    for n in (8, 16):
        tr, toks = gpu_steps(full, steps, n=n, force_p=0.7, forced_ref=torch.from_numpy(ref).cuda(), seed=2)
        assert toks[0] == y0
        o, rep = replay(base, full, tr, toks[0], n=n, forced_p=0.7, forced_ref=ref)
        compare(full, tr, o, rep)
        assert o.tokens[full.prompt_len: full.prompt_len + len(toks)] == toks
    vectors(full, base, 6, p=0.7, ref=ref)
    del base
    gc.collect()
    # the whole generation on the GPU against its own one-stage decode
    p_full = torch.from_numpy(prompt).cuda()
    ar = Engine(full.dm, dtg, dpd, 1, full.anchors, max_seq=full.max_seq + 40, max_new=full.max_new + 24)
    out, cnt, _ = ar.generate(p_full)
    ar_toks = out[:cnt].cpu().tolist()
    ar.close()
    ref_gpu = torch.cat([p_full, out[:cnt], torch.zeros(full.n * 2 + 8, dtype=torch.int32, device="cuda")]).contiguous()
    for n in (8, 16):
        e = Engine(full.dm, dtg, dpd, n, full.anchors, max_seq=full.max_seq + 16, max_new=full.max_new,
                   force_p=0.7, forced_ref=ref_gpu, seed=2)
        o2, c2, st = e.generate(p_full)
        toks = o2[:c2].cpu().tolist()
        e.close()
        assert toks == ar_toks[: full.max_new], n
        assert st.accepts > 0 and st.rejects > 0
    release()
