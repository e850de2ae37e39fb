"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Integer results (token ids, keep decisions, commits, exit positions, per-layer KV valid
lengths) must agree exactly; where the oracle's own decision is within the tolerance of
a tie (top-2 logit margin <= tol * |top-1|) it follows the GPU's choice (replay rule).
Logits agree within rel 1e-4 (fp32 weights) or 2e-2 (bf16 weights), relative to
max(1, |logit|).
"""
import numpy as np
import pytest
import torch

import spd_inputs as si
from gpu_common import (Case, ar_reference, compare, engine, materialise, replay_oracle, run_gpu,
                        step_and_compare_vectors)
from oracle import Replay, SPDOracle

pytestmark = pytest.mark.gpu

TINY = Case(si.TINY.dims, n=2, anchors=(0, 2, 4), Ls=1, prompt_len=16, max_new=64)
# bf16, hd 64, GQA 2, prompt long enough for several 128-position attention chunks + tail
SMALL = Case(si.ModelDims(L=6, d=256, Hq=4, Hkv=2, hd=64, F=512, V=2000), n=3, anchors=(0, 3, 6), Ls=2,
             prompt_len=300, max_new=48, norms="perturbed")
# bf16, hd 128, GQA 4 (the 4B shape's head layout), 5 layers over 4 stages (ragged stages)
HD128 = Case(si.ModelDims(L=5, d=512, Hq=8, Hkv=2, hd=128, F=1024, V=3000), n=4, anchors=(0, 2, 5), Ls=1,
             prompt_len=140, max_new=40, norms="perturbed")
# bf16, rows longer than one 4 KB tile chunk (d 2560, F 2304: two K chunks per row)
MULTI = Case(si.ModelDims(L=4, d=2560, Hq=8, Hkv=2, hd=128, F=2304, V=1000), n=3, anchors=(0, 2, 4), Ls=1,
             prompt_len=200, max_new=40, norms="perturbed")
# bf16, 16 stages of 2 layers: 17 draft rows take two 16-row mma tiles
WIDE = Case(si.ModelDims(L=32, d=256, Hq=4, Hkv=2, hd=64, F=512, V=1500), n=16, anchors=(0, 16, 32), Ls=1,
            prompt_len=40, max_new=40, norms="perturbed")
# bf16, d 2560 with 17 draft rows: the draft QKV and gate/up need two K slabs (RoPE and KV append
# happen in the slab-finishing pass), down three
WIDEK = Case(si.ModelDims(L=32, d=2560, Hq=8, Hkv=2, hd=128, F=2560, V=1000), n=16, anchors=(0, 16, 32), Ls=1,
             prompt_len=40, max_new=40, norms="perturbed")
# bf16, 2 stages of 3 layers with 2 draft layers (more draft layers relative to the stages)
INROUNDS = Case(si.ModelDims(L=6, d=512, Hq=8, Hkv=2, hd=64, F=1024, V=1600), n=2, anchors=(0, 3, 6), Ls=2,
                prompt_len=200, max_new=48, norms="perturbed")
# bf16, the 8B shape's width and heads (d 4096, 32q/8kv x 128) over 5 one-layer stages: 6 draft
# rows (12 with their lo parts) split the draft QKV, O and gate/up into two K slabs, and the LM
# head's 8 KB rows take two pieces per tile
D4096 = Case(si.ModelDims(L=5, d=4096, Hq=32, Hkv=8, hd=128, F=2048, V=2048), n=5, anchors=(0, 2, 5), Ls=1,
             prompt_len=64, max_new=32, norms="perturbed")
# MULTI's draft projection (K = 5 x 2560) is split into K slabs across CTAs; its QKV, O, gate/up
# and down keep x in registers (one 16-row tile, K <= 2560); WIDE's 17 rows keep x in shared memory.


def _prefill_logits_close(case, pf):
    tg, pd, prompt, m, _, _ = materialise(case)
    from oracle import SPDOracle
    o = SPDOracle(m, case.n, case.max_seq)
    o.prefill(prompt)
    z = o.prefill_logits
    err = np.max(np.abs(pf - z)) / max(1.0, np.max(np.abs(z)))
    assert err <= case.tol, err
    return err


@pytest.mark.parametrize("case", [TINY, SMALL, HD128, MULTI], ids=["tiny", "small", "hd128", "multi"])
def test_prefill_logits(case):
    toks, tr, st, pf = run_gpu(case, force_p=1.0, forced_ref=torch.zeros(case.max_seq, dtype=torch.int32).cuda())
    _prefill_logits_close(case, pf)


@pytest.mark.parametrize("case", [TINY, SMALL, HD128, MULTI, WIDEK],
                         ids=["tiny", "small", "hd128", "multi", "widek"])
def test_prefill_kv_caches_match_oracle(case):
    """Every layer's K and V rows of the prompt, target and draft module, and the prompt's
    last-position logits entry by entry, against the oracle's prefill (the tensor-core
    GEMMs and attention of a bf16 prefill, the CUDA-core ones of an fp32 model)."""
    from gpu_common import elem_err, vec_err
    from speculative_pipeline_decoding_spd_gb300 import binding as B
    tg, pd, prompt, m, _, _ = materialise(case)
    e = engine(case, graph=False)
    e.prefill(torch.from_numpy(prompt).cuda())
    o = SPDOracle(m, case.n, case.max_seq)
    o.prefill(prompt)
    Sp, kvw = case.prompt_len, case.dm.Hkv * case.dm.hd
    worst = 0.0
    for li in range(case.dm.L):
        for which, ref in ((B.SPD_BUF_KCACHE, o.kv.K[li]), (B.SPD_BUF_VCACHE, o.kv.V[li])):
            got = e.read(which, (Sp, kvw), dtype=case.kv_dtype, index=li).astype(np.float64)
            worst = max(worst, vec_err(got, ref[:Sp].reshape(Sp, kvw)))
    for li in range(case.Ls):
        for which, ref in ((B.SPD_BUF_PDM_KCACHE, o.pkv.K[li]), (B.SPD_BUF_PDM_VCACHE, o.pkv.V[li])):
            got = e.read(which, (Sp, kvw), dtype=case.kv_dtype, index=li).astype(np.float64)
            worst = max(worst, vec_err(got, ref[:Sp].reshape(Sp, kvw)))
    pf = e.read(B.SPD_BUF_PREFILL_LOGITS, (case.dm.V,))
    e.close()
    lerr = elem_err(pf, o.prefill_logits)
    print(f"prefill: K/V {worst:.2e}, logits {lerr:.2e}")
    assert worst <= case.tol and lerr <= case.tol, (worst, lerr)


@pytest.mark.parametrize("case", [TINY, SMALL, HD128, MULTI, WIDE, WIDEK, INROUNDS],
                         ids=["tiny", "small", "hd128", "multi", "wide", "widek", "inrounds"])
def test_greedy_draft_module_replay(case):
    toks, tr, st, pf = run_gpu(case)
    o, rep = replay_oracle(case, tr, toks)
    compare(case, tr, o, rep)
    assert o.tokens[case.prompt_len:] == toks
    assert st["N"] == case.max_new - 1 and st["K"] == len(tr)


@pytest.mark.parametrize("case,p", [(TINY, 0.6), (SMALL, 0.5), (SMALL, 0.9), (HD128, 0.7), (MULTI, 0.6), (WIDE, 0.8),
                                    (INROUNDS, 0.7)],
                         ids=["tiny-0.6", "small-0.5", "small-0.9", "hd128-0.7", "multi-0.6", "wide-0.8", "inrounds-0.7"])
def test_forced_draft_replay(case, p):
    ar = ar_reference(case)
    tg, pd, prompt, m, _, _ = materialise(case)
    ref = np.array(list(prompt) + ar + [0] * (case.n + 8), dtype=np.int32)
    toks, tr, st, pf = run_gpu(case, force_p=p, forced_ref=torch.from_numpy(ref).cuda(), seed=5)
    o, rep = replay_oracle(case, tr, toks, forced_p=p, forced_ref=ref, seed=5)
    compare(case, tr, o, rep)
    assert o.tokens[case.prompt_len:] == toks
    assert st["accepts"] > 0 and st["rejects"] > 0


@pytest.mark.parametrize("case", [TINY, SMALL, HD128, MULTI], ids=["tiny", "small", "hd128", "multi"])
def test_pipeline_equals_single_stage_bitwise(case):
    """Losslessness on the device: for every n the pipelined decode commits the same
    tokens as n = 1 (one token through all layers per step), and the per-step target
    logits are bit-identical, because no kernel's arithmetic depends on which stages
    share a launch."""
    ar_toks, ar_tr, _, _ = run_gpu(case, n=1)
    ar_logit = {r["exit_pos"]: r["target_logit"] for r in ar_tr if r["exit_pos"] >= 0}
    for n in sorted({2, case.n, min(case.dm.L, 5)}):
        toks, tr, st, _ = run_gpu(case, n=n)
        assert toks == ar_toks, n
        for r in tr:
            if r["exit_pos"] >= 0:
                assert r["target_logit"] == ar_logit[r["exit_pos"]], (n, r["exit_pos"])


@pytest.mark.parametrize("case,n", [(MULTI, 1), (MULTI, 3), (SMALL, 3)], ids=["multi-1", "multi-3", "small-3"])
def test_workspace_contents_do_not_matter(case, n):
    """The workspace the caller hands over holds garbage (here all bytes 0xFF): every counter
    and state word the library uses must be initialised by spd_create / spd_prefill."""
    a = run_gpu(case, n=n)[:2]
    b = run_gpu(case, n=n, workspace_fill=0xFF)[:2]
    assert a[0] == b[0]
    assert [r["len"] for r in a[1]] == [r["len"] for r in b[1]]


def test_graph_and_eager_agree():
    a = run_gpu(SMALL, graph=False)[:2]
    b = run_gpu(SMALL, graph=True)[:2]
    assert a[0] == b[0] and [r["len"] for r in a[1]] == [r["len"] for r in b[1]]


def test_host_buffers_generate():
    tg, pd, prompt, m, _, _ = materialise(SMALL)
    e = engine(SMALL)
    host_toks, st = e.generate(prompt, on_host=True)
    e.close()
    dev_toks = run_gpu(SMALL)[0]
    assert host_toks == dev_toks


def test_step_by_step_state_matches_oracle_hidden_states():
    """Residual stream of every in-flight slot after each of the first steps, against
    the oracle's in-flight hidden states (same tolerance)."""
    case = SMALL
    tg, pd, prompt, m, _, _ = materialise(case)
    e = engine(case, graph=False)
    e.prefill(torch.from_numpy(prompt).cuda())
    from oracle import Replay, SPDOracle
    gtr = []
    o = None
    for k in range(1, 9):
        e.step(1)
        tr = e.trace()
        o, rep = replay_oracle(case, tr, e.tokens(), max_steps=k)
        X = e.read(0, (case.n + 1, case.dm.d))
        slots = e.read(7, (3, case.n + 1), dtype=np.int32)
        for s, tk in enumerate(o.slots):
            if tk is None or s == 0:
                continue      # stage 0 holds a just-embedded token
            # find the slot holding this position
            idx = [i for i in range(case.n + 1) if slots[0][i] and slots[1][i] == tk.pos]
            assert idx, (k, tk.pos)
            ref = tk.H[0]
            err = np.max(np.abs(X[idx[0]] - ref)) / max(1.0, np.max(np.abs(ref)))
            assert err <= case.tol, (k, s, err)
    e.close()


# bf16 with a vocabulary that is not a multiple of 8: the LM head runs as the grouped GEMV
# (ragged last tile group) instead of the tensor-core GEMM
RAGGEDV = Case(si.ModelDims(L=6, d=256, Hq=4, Hkv=2, hd=64, F=512, V=2001), n=3, anchors=(0, 3, 6), Ls=2,
               prompt_len=120, max_new=40, norms="perturbed")


def test_ragged_vocab_replay():
    toks, tr, st, pf = run_gpu(RAGGEDV)
    o, rep = replay_oracle(RAGGEDV, tr, toks)
    compare(RAGGEDV, tr, o, rep)
    assert o.tokens[RAGGEDV.prompt_len:] == toks


def test_untied_head_copy_replay():
    """The draft module's LM head given as a separate copy of the target's: the library takes
    the untied path (the grouped GEMV with one head per row), and the results still follow the
    oracle, whose head is the target's."""
    from speculative_pipeline_decoding_spd_gb300.engine import Engine
    case = SMALL
    tg, pd, prompt, m, dtg, dpd = materialise(case)
    dpd2 = dict(dpd)
    dpd2["lm_head"] = dtg["lm_head"].clone()
    e = Engine(case.dm, dtg, dpd2, case.n, case.anchors, max_seq=case.max_seq, max_new=case.max_new)
    out, cnt, _ = e.generate(torch.from_numpy(prompt).cuda())
    toks = out[:cnt].cpu().tolist()
    tr = e.trace()
    e.close()
    o, rep = replay_oracle(case, tr, toks)
    compare(case, tr, o, rep)
    assert o.tokens[case.prompt_len:] == toks


# ---- vectors, step by step --------------------------------------------------------------

VEC_CASES = [
    ("tiny", TINY, {}),
    ("small", SMALL, {}),
    ("small-forced", SMALL, dict(p=0.6)),
    ("hd128-forced", HD128, dict(p=0.6)),
    ("multi", MULTI, {}),
    ("wide-forced", WIDE, dict(p=0.7)),
    ("widek", WIDEK, {}),
    ("d4096-forced", D4096, dict(p=0.6)),
    ("inrounds-forced", INROUNDS, dict(p=0.6)),
    ("small-output", SMALL, dict(speculate="output", p=0.6)),
    ("hd128-bounds", HD128, dict(bounds=(0, 1, 2, 4, 5), p=0.6)),
]


def vector_run(case, steps, p=None, speculate="input", bounds=None, n=None):
    """Prefill both sides, then compare the vectors after each of `steps` steps."""
    tg, pd, prompt, m, _, _ = materialise(case)
    n = n or case.n
    kw = dict(speculate=speculate, bounds=bounds)
    okw = dict(speculate=speculate, bounds=bounds)
    if p is not None:
        ref = np.array(list(prompt) + ar_reference(case) + [0] * (case.n + 8), dtype=np.int32)
        kw.update(force_p=p, forced_ref=torch.from_numpy(ref).cuda(), seed=5)
        okw.update(forced_p=p, forced_ref=ref, seed=5)
    e = engine(case, n=n, graph=False, **kw)
    e.prefill(torch.from_numpy(prompt).cuda())
    y0 = e.tokens()[0]
    o = SPDOracle(m, n, case.max_seq, replay=Replay(steps={}, prefill_y0=y0, tol=case.tol), **okw)
    o.prefill(prompt)
    worst = step_and_compare_vectors(case, e, o, steps)
    e.close()
    return worst, o


@pytest.mark.parametrize("name,case,kw", VEC_CASES, ids=[c[0] for c in VEC_CASES])
def test_vectors_match_oracle_step_by_step(name, case, kw):
    """Logits entry by entry, the draft block's residual rows, every in-flight residual
    stream and anchor state, and the K/V rows each step writes, against the oracle after
    each of the first steps (12, or 2n when the pipeline is deeper), all within the case's one
    tolerance."""
    worst, o = vector_run(case, max(12, 2 * case.n), **kw)   # past the first exits and a rollback
    if kw.get("p") is not None:
        assert any(r["accept"] == 0 for r in o.trace)     # a rollback happened inside the window


# ---- the output-state schedule and non-uniform stages -----------------------------------

@pytest.mark.parametrize("case,p", [(SMALL, None), (SMALL, 0.6), (HD128, 0.7), (WIDE, 0.8), (TINY, 0.6)],
                         ids=["small", "small-0.6", "hd128-0.7", "wide-0.8", "tiny-0.6"])
def test_output_state_schedule_replay(case, p):
    """The draft module after the step, on its output states (stage s at depth b_{s+1}):
    the whole run replayed against the oracle's output-state simulator; the committed
    tokens are the same as under the input-state schedule."""
    kw, okw = {}, {}
    if p is not None:
        tg, pd, prompt, m, _, _ = materialise(case)
        ref = np.array(list(prompt) + ar_reference(case) + [0] * (case.n + 8), dtype=np.int32)
        kw = dict(force_p=p, forced_ref=torch.from_numpy(ref).cuda(), seed=5)
        okw = dict(forced_p=p, forced_ref=ref, seed=5)
    toks, tr, st, pf = run_gpu(case, speculate="output", **kw)
    o, rep = replay_oracle(case, tr, toks, speculate="output", **okw)
    compare(case, tr, o, rep)
    assert o.tokens[case.prompt_len:] == toks
    if p is None:
        # the schedules' draft modules see different features
        toks_in, tr_in, _, _ = run_gpu(case)
        assert toks_in == toks
        assert [r["pdm_logit"] for r in tr_in] != [r["pdm_logit"] for r in tr]


@pytest.mark.parametrize("case,bounds,p", [(SMALL, (0, 1, 5, 6), None), (SMALL, (0, 4, 5, 6), 0.6),
                                           (HD128, (0, 3, 4, 5), 0.7), (WIDE, tuple(range(0, 33, 2)), 0.8),
                                           (MULTI, (0, 1, 4), 0.6)],
                         ids=["small-1-4-1", "small-4-1-1", "hd128-3-1-1", "wide-uniform", "multi-1-3"])
def test_non_uniform_stages_replay(case, bounds, p):
    """Explicit stage partitions (the referee report's Appendix C.1 comment): the whole run
    replayed against the oracle with the same bounds; per-layer KV lengths follow them."""
    n = len(bounds) - 1
    kw, okw = {}, {}
    if p is not None:
        tg, pd, prompt, m, _, _ = materialise(case)
        ref = np.array(list(prompt) + ar_reference(case) + [0] * (n + 8), dtype=np.int32)
        kw = dict(force_p=p, forced_ref=torch.from_numpy(ref).cuda(), seed=5)
        okw = dict(forced_p=p, forced_ref=ref, seed=5)
    toks, tr, st, pf = run_gpu(case, n=n, bounds=bounds, **kw)
    o, rep = replay_oracle(case, tr, toks, n=n, bounds=bounds, **okw)
    compare(case, tr, o, rep)
    assert o.tokens[case.prompt_len:] == toks


def test_bad_stage_bounds_are_refused():
    from speculative_pipeline_decoding_spd_gb300 import binding as B
    for bounds in [(0, 3, 3, 6), (1, 3, 6), (0, 2, 5)]:
        with pytest.raises(B.SPDError) as e:
            engine(SMALL, n=len(bounds) - 1, bounds=bounds)
        assert e.value.code == B.SPD_EINVAL


def test_trace_view_is_the_device_copy_of_the_trace():
    """spd_get_trace_view hands out the device records and KV lengths that spd_get_trace copies."""
    import ctypes as C
    from speculative_pipeline_decoding_spd_gb300 import binding as B
    tg, pd, prompt, m, _, _ = materialise(SMALL)
    e = engine(SMALL)
    e.generate(torch.from_numpy(prompt).cuda())
    tr = e.trace()
    v = B.spd_get_trace_view(e.h)
    assert v.count == len(tr) and v.L == SMALL.dm.L
    lib = B.load()   # the CUDA runtime the library links resolves through its handle
    lib.cudaMemcpy.argtypes = [C.c_void_p, C.c_void_p, C.c_size_t, C.c_int]
    recs = (B.spd_trace_rec * v.count)()
    lens = np.zeros((v.count, v.L), dtype=np.int32)
    assert lib.cudaMemcpy(C.addressof(recs), v.recs, C.sizeof(recs), 2) == 0
    assert lib.cudaMemcpy(lens.ctypes.data, v.kv_len, lens.nbytes, 2) == 0
    e.close()
    for r, g, ln in zip(tr, recs, lens):
        assert (r["t"], r["exit_pos"], r["commit"], r["new_draft"]) == (g.t, g.exit_pos, g.commit, g.new_draft)
        assert r["len"] == ln.tolist()


@pytest.mark.parametrize("case", [SMALL, HD128, TINY], ids=["small", "hd128", "tiny"])
def test_sampling_replay(case):
    """T = 1: drafts sampled from the draft module's softmax, speculative rejection sampling with
    residual resamples, on the same Philox uniforms as the oracle.  bf16 cases draw the draft
    inside the tensor-core LM head (its softmax statistics merged across CTAs); the fp32 case
    in the verification kernel."""
    toks, tr, st, pf = run_gpu(case, temperature=1.0, seed=3)
    o, rep = replay_oracle(case, tr, toks, temperature=1.0, seed=3)
    compare(case, tr, o, rep)
    assert o.tokens[case.prompt_len:] == toks
    assert sum(1 for r in tr if r["accept"] == 0) > 0 and sum(1 for r in tr if r["accept"] == 1) > 0
